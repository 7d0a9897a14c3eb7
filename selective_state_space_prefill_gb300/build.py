"""Build libssm.so (the CUDA kernels and their C ABI) in-tree for sm_103a.

Each translation unit in ``csrc/`` is compiled by its own nvcc process (in
parallel), then linked into ``_build/libssm.so``.  ptxas resource usage
(registers, spills, shared memory) is kept in ``_build/ptxas.log``.

A build is reused only when ``_build/libssm.sha256`` holds the digest of exactly
the sources, headers, flags and compiler it was made from (file times are not
trusted: a copied tree keeps a library newer than edited sources).
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
INCLUDE = PKG.parent / "include"
LIB = BUILD / "libssm.so"
STAMP = BUILD / "libssm.sha256"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                     "--expt-relaxed-constexpr", "-I", str(INCLUDE)]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found; libssm needs the CUDA toolkit to build")


def _sources():
    return sorted(CSRC.glob("*.cu"))


def _deps():
    return sorted(CSRC.glob("*.cu")) + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + \
        sorted(INCLUDE.glob("*.h"))


def source_digest(cc: str | None = None) -> str:
    """SHA-256 over every source and header (name and bytes), the flags and the compiler path."""
    h = hashlib.sha256()
    for p in _deps():
        h.update(p.name.encode() + b"\0" + p.read_bytes() + b"\0")
    h.update(" ".join(NVCC_FLAGS).encode())
    h.update((cc or nvcc()).encode())
    return h.hexdigest()


def up_to_date() -> bool:
    if not (LIB.exists() and STAMP.exists()):
        return False
    try:
        return STAMP.read_text().strip() == source_digest()
    except (OSError, RuntimeError):
        return False


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile and link libssm.so; returns its path.  Raises on any compiler error."""
    if not force and up_to_date():
        return LIB
    BUILD.mkdir(parents=True, exist_ok=True)
    cc = nvcc()
    digest = source_digest(cc)
    objdir = BUILD / f"obj.{os.getpid()}"          # concurrent builders never share an object file
    objdir.mkdir(exist_ok=True)

    def compile_one(src: Path):
        obj = objdir / (src.stem + ".o")
        cmd = [cc, *NVCC_FLAGS, "-c", str(src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(len(_sources()), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    (BUILD / "ptxas.log").write_text("".join(log for _, log in results))
    tmp = BUILD / f"libssm.so.{os.getpid()}.tmp"       # concurrent builders never share a file
    cmd = [cc, *ARCH, "-shared", "-o", str(tmp), *[str(o) for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    shutil.rmtree(objdir, ignore_errors=True)
    stamp_tmp = BUILD / f"libssm.sha256.{os.getpid()}.tmp"
    stamp_tmp.write_text(digest + "\n")
    os.replace(stamp_tmp, STAMP)
    if verbose:
        print((BUILD / "ptxas.log").read_text())
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
