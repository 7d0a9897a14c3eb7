"""The build reuses a library only when it was made from exactly the current sources.

No GPU and no compiler run is needed: the checks work on a copy of the sources in a
temporary tree, with a stand-in library file whose time stamp is newer than every source.
"""
import os
import shutil

from selective_state_space_prefill_gb300 import build
import oracle.oracle as orc


def _tree(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    inc = tmp_path / "include"
    shutil.copytree(build.CSRC, csrc)
    shutil.copytree(build.INCLUDE, inc)
    out = tmp_path / "_build"
    out.mkdir()
    monkeypatch.setattr(build, "CSRC", csrc)
    monkeypatch.setattr(build, "INCLUDE", inc)
    monkeypatch.setattr(build, "LIB", out / "libssm.so")
    monkeypatch.setattr(build, "STAMP", out / "libssm.sha256")
    monkeypatch.setattr(build, "nvcc", lambda: "/usr/local/cuda/bin/nvcc")
    build.LIB.write_bytes(b"stand-in")
    return csrc, inc


def test_a_library_without_a_stamp_is_rebuilt(tmp_path, monkeypatch):
    _tree(tmp_path, monkeypatch)
    assert not build.up_to_date()


def test_touched_source_forces_a_rebuild_whatever_the_file_times(tmp_path, monkeypatch):
    csrc, inc = _tree(tmp_path, monkeypatch)
    build.STAMP.write_text(build.source_digest() + "\n")
    assert build.up_to_date()
    # edit one kernel source, then make the library look newer than every source
    src = csrc / "prefill.cu"
    src.write_text(src.read_text() + "\n// edited\n")
    future = max(p.stat().st_mtime for p in build._deps()) + 3600
    os.utime(build.LIB, (future, future))
    assert not build.up_to_date()
    # a header edit counts too
    build.STAMP.write_text(build.source_digest() + "\n")
    assert build.up_to_date()
    h = inc / "ssm.h"
    h.write_text(h.read_text() + "\n")
    assert not build.up_to_date()


def test_flags_are_part_of_the_digest(tmp_path, monkeypatch):
    _tree(tmp_path, monkeypatch)
    before = build.source_digest()
    monkeypatch.setattr(build, "NVCC_FLAGS", build.NVCC_FLAGS + ["-DSOMETHING"])
    assert build.source_digest() != before


def test_oracle_rebuilds_when_its_source_changes(tmp_path):
    src = tmp_path / "o.c"
    src.write_text("int f(void) { return 1; }\n")
    out = tmp_path / "libo.so"
    orc.build(src, out)
    first = out.stat().st_mtime_ns
    assert orc.build(src, out).stat().st_mtime_ns == first        # reused: same bytes
    src.write_text("int f(void) { return 2; }\n")
    os.utime(src, (0, 0))                                         # older than the library
    orc.build(src, out)
    import ctypes
    assert ctypes.CDLL(str(out)).f() == 2                         # rebuilt from the new bytes
