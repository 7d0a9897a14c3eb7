"""ctypes marshalling for ssm_oracle.c (test infrastructure only).

Arrays are widened nowhere here: the C code reads the same float32 / bfloat16
bytes the CUDA path reads and widens them to double itself.  Outputs are
float64 numpy arrays (q8: int32 sums, float32 scales/out, bfloat16 bits).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "ssm_oracle.c"
_BUILD = _HERE / "_build"

F32, BF16 = 0, 1

_lib = None


def lib_path() -> Path:
    return _BUILD / "libssm_oracle.so"


def build(src: Path | None = None, out: Path | None = None, force: bool = False) -> Path:
    """Compile the oracle with the host C compiler (gcc/cc), OpenMP if available.

    A build is reused only when the digest beside it matches the source bytes and compiler,
    never on file times (a copied tree may carry a library newer than an edited source).
    """
    src = Path(src) if src else _SRC
    out = Path(out) if out else lib_path()
    cc = os.environ.get("CC", "gcc")
    stamp = Path(str(out) + ".sha256")
    digest = hashlib.sha256(src.read_bytes() + b"\0" + cc.encode()).hexdigest()
    if (out.exists() and stamp.exists() and not force and
            stamp.read_text().strip() == digest):
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"        # concurrent builders (spawned ranks) never share a file
    base = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", str(src),
            "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    Path(tmp + ".sha256").write_text(digest + "\n")
    os.replace(tmp + ".sha256", stamp)
    return out


def _bind(lib):
    P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_prefill.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I]
    lib.oracle_prefill.restype = I
    lib.oracle_decode_step.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_decode_step.restype = I
    lib.oracle_scan_sequential.argtypes = [L, P, P, D, P]
    lib.oracle_scan_sequential.restype = None
    lib.oracle_scan_chunked.argtypes = [L, P, P, D, L, P]
    lib.oracle_scan_chunked.restype = None
    lib.oracle_q8_reduce.argtypes = [I, P, I, L, I, P, P, P, P]
    lib.oracle_q8_reduce.restype = I
    lib.oracle_q8_block_absmax.argtypes = [P, I, L, I, P]
    lib.oracle_q8_block_absmax.restype = I
    lib.oracle_q8_quantize_shared.argtypes = [P, I, L, I, P, P, P]
    lib.oracle_q8_quantize_shared.restype = I
    lib.oracle_q8_sum_dequant.argtypes = [I, P, P, L, I, P, P, P]
    lib.oracle_q8_sum_dequant.restype = I
    lib.oracle_out_proj.argtypes = [L, L, L, I, P, P, P, P, P, I]
    lib.oracle_out_proj.restype = I
    lib.oracle_ssd_prefill.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, I,
                                       P, P, P, I]
    lib.oracle_ssd_prefill.restype = I
    return lib


def load(path: Path | None = None):
    """Load (building first if needed) the oracle library; a custom path loads a fresh copy."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(str(build())))
    return _lib


def _threads(n):
    if n:
        return int(n)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _raw(t):
    """(contiguous numpy array of the raw element bytes, dtype code) for a torch tensor or ndarray."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), BF16
            if t.dtype == torch.float32:
                return t.numpy(), F32
            raise TypeError(f"unsupported dtype {t.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"unsupported dtype {a.dtype}")


def _f32(t):
    a, code = _raw(t)
    if code != F32:
        raise TypeError("parameters must be float32")
    return np.ascontiguousarray(a)


def _f64(t):
    if t is None:
        return None
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(t, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def prefill(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state_in=None, ssm_state_in=None,
            channels=None, n_threads=None, lib=None):
    """Oracle prefill.  Token tensors are [batch, L, d_inner] / [batch, L, N].

    ``channels`` (optional index list) evaluates only those channels; every
    channel is independent, so this is the same computation restricted to them.
    Returns dict(out [b, L, c], conv_state [b, W-1, c], ssm_state [b, c, N]) in float64.
    """
    lib = lib or load()
    xr, code = _raw(x)
    zr, code_z = _raw(z)
    dtr, code_dt = _raw(dt)
    Br, code_b = _raw(B)
    Cr, code_c = _raw(C)
    if len({code, code_z, code_dt, code_b, code_c}) != 1:
        raise TypeError("x, z, dt, B, C must share one dtype")
    A, D, dt_bias, conv_w, conv_b = map(_f32, (A, D, dt_bias, conv_w, conv_b))
    csi, ssi = _f64(conv_state_in), _f64(ssm_state_in)
    if channels is not None:
        idx = np.asarray(channels, dtype=np.int64)
        xr, zr, dtr = (np.ascontiguousarray(a[..., idx]) for a in (xr, zr, dtr))
        A, D, dt_bias, conv_w, conv_b = (np.ascontiguousarray(a[idx]) for a in (A, D, dt_bias, conv_w, conv_b))
        if csi is not None:
            csi = np.ascontiguousarray(csi[..., idx])
        if ssi is not None:
            ssi = np.ascontiguousarray(ssi[:, idx])
    batch, L, Dn = xr.shape
    N = Br.shape[-1]
    W = conv_w.shape[-1]
    out = np.empty((batch, L, Dn), np.float64)
    cso = np.empty((batch, W - 1, Dn), np.float64)
    sso = np.empty((batch, Dn, N), np.float64)
    rc = lib.oracle_prefill(batch, L, Dn, N, W, code, _p(xr), _p(zr), _p(dtr), _p(Br), _p(Cr),
                            _p(A), _p(D), _p(dt_bias), _p(conv_w), _p(conv_b), _p(csi), _p(ssi),
                            _p(out), _p(cso), _p(sso), _threads(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_prefill rejected the sizes (rc={rc})")
    return dict(out=out, conv_state=cso, ssm_state=sso)


def decode_step(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state, ssm_state, lib=None):
    """Oracle decode step for [batch, d_inner] tokens.  States are copied, not modified.

    Returns dict(out [b, d], conv_state, ssm_state) in float64 (the updated states).
    """
    lib = lib or load()
    xr, code = _raw(x)
    zr, _ = _raw(z)
    dtr, _ = _raw(dt)
    Br, _ = _raw(B)
    Cr, _ = _raw(C)
    A, D, dt_bias, conv_w, conv_b = map(_f32, (A, D, dt_bias, conv_w, conv_b))
    cs = _f64(conv_state).copy()
    ss = _f64(ssm_state).copy()
    batch, Dn = xr.shape
    N = Br.shape[-1]
    W = conv_w.shape[-1]
    out = np.empty((batch, Dn), np.float64)
    rc = lib.oracle_decode_step(batch, Dn, N, W, code, _p(xr), _p(zr), _p(dtr), _p(Br), _p(Cr),
                                _p(A), _p(D), _p(dt_bias), _p(conv_w), _p(conv_b), _p(cs), _p(ss),
                                _p(out))
    if rc != 0:
        raise ValueError(f"oracle_decode_step rejected the sizes (rc={rc})")
    return dict(out=out, conv_state=cs, ssm_state=ss)


def scan_sequential(a, b, h0=0.0, lib=None):
    lib = lib or load()
    a = np.ascontiguousarray(a, np.float64)
    b = np.ascontiguousarray(b, np.float64)
    h = np.empty_like(a)
    lib.oracle_scan_sequential(a.size, _p(a), _p(b), float(h0), _p(h))
    return h


def scan_chunked(a, b, h0=0.0, chunk=64, lib=None):
    lib = lib or load()
    a = np.ascontiguousarray(a, np.float64)
    b = np.ascontiguousarray(b, np.float64)
    h = np.empty_like(a)
    lib.oracle_scan_chunked(a.size, _p(a), _p(b), float(h0), int(chunk), _p(h))
    return h


def q8_reduce(partials, block=128, lib=None):
    """Returns dict(sums int32 [n], scales float32 [nblk], out_f32 [n], out_bf16 uint16 bits [n])."""
    lib = lib or load()
    raws = [_raw(p) for p in partials]
    codes = {c for _, c in raws}
    if len(codes) != 1:
        raise TypeError("partials must share one dtype")
    arrs = [np.ascontiguousarray(r.reshape(-1)) for r, _ in raws]
    n = arrs[0].size
    P = len(arrs)
    ptrs = (ctypes.c_void_p * P)(*[a.ctypes.data for a in arrs])
    nblk = (n + block - 1) // block
    sums = np.empty(n, np.int32)
    scales = np.empty(nblk, np.float32)
    out_f32 = np.empty(n, np.float32)
    out_bf16 = np.empty(n, np.uint16)
    rc = lib.oracle_q8_reduce(P, ctypes.cast(ptrs, ctypes.c_void_p), codes.pop(), n, block,
                              _p(sums), _p(scales), _p(out_f32), _p(out_bf16))
    if rc != 0:
        raise ValueError(f"oracle_q8_reduce rejected the sizes (rc={rc})")
    return dict(sums=sums, scales=scales, out_f32=out_f32, out_bf16=out_bf16)


def q8_block_absmax(x, block=128, lib=None):
    """float32 [nblk] block maxima of |x| (x flattened)."""
    lib = lib or load()
    r, code = _raw(x)
    a = np.ascontiguousarray(r.reshape(-1))
    n = a.size
    amax = np.empty((n + block - 1) // block, np.float32)
    if lib.oracle_q8_block_absmax(a.ctypes.data, code, n, block, _p(amax)) != 0:
        raise ValueError("oracle_q8_block_absmax rejected the sizes")
    return amax


def q8_quantize_shared(x, amax, block=128, lib=None):
    """Returns dict(codes int8 [n], scales float32 [nblk]) for the shared maxima `amax`."""
    lib = lib or load()
    r, code = _raw(x)
    a = np.ascontiguousarray(r.reshape(-1))
    n = a.size
    am = np.ascontiguousarray(np.asarray(amax, np.float32).reshape(-1))
    codes = np.empty(n, np.int8)
    scales = np.empty((n + block - 1) // block, np.float32)
    if lib.oracle_q8_quantize_shared(a.ctypes.data, code, n, block, _p(am), _p(codes), _p(scales)) != 0:
        raise ValueError("oracle_q8_quantize_shared rejected the sizes")
    return dict(codes=codes, scales=scales)


def q8_sum_dequant(codes, scales, block=128, lib=None):
    """codes: P int8 arrays [n]; returns dict(sums int32, out_f32 float32, out_bf16 uint16 bits)."""
    lib = lib or load()
    cs = [np.ascontiguousarray(np.asarray(c, np.int8).reshape(-1)) for c in codes]
    n = cs[0].size
    P = len(cs)
    ptrs = (ctypes.c_void_p * P)(*[c.ctypes.data for c in cs])
    sc = np.ascontiguousarray(np.asarray(scales, np.float32).reshape(-1))
    sums = np.empty(n, np.int32)
    out_f32 = np.empty(n, np.float32)
    out_bf16 = np.empty(n, np.uint16)
    if lib.oracle_q8_sum_dequant(P, ctypes.cast(ptrs, ctypes.c_void_p), _p(sc), n, block, _p(sums), _p(out_f32),
                                 _p(out_bf16)) != 0:
        raise ValueError("oracle_q8_sum_dequant rejected the sizes")
    return dict(sums=sums, out_f32=out_f32, out_bf16=out_bf16)


def out_proj(y, W, n_threads=None, lib=None):
    """One rank's out_proj partial: y [M, K] and W [N, K] (same dtype).

    Returns dict(out [M, N] float64, amax [ceil(M*N/128)] float64, absdot [M, N] float64),
    absdot = |y| @ |W|^T (the scale of the rounding error of any fp32 evaluation).
    """
    lib = lib or load()
    yr, cy = _raw(y)
    wr, cw = _raw(W)
    if cy != cw:
        raise TypeError("y and W must share one dtype")
    yr = np.ascontiguousarray(yr.reshape(yr.shape[0], -1) if yr.ndim > 2 else yr)
    wr = np.ascontiguousarray(wr)
    M, K = yr.shape
    N, K2 = wr.shape
    if K != K2:
        raise ValueError("y and W disagree on K")
    out = np.empty((M, N), np.float64)
    absdot = np.empty((M, N), np.float64)
    amax = np.empty(((M * N) + 127) // 128, np.float64)
    rc = lib.oracle_out_proj(M, N, K, cy, _p(yr), _p(wr), _p(out), _p(amax), _p(absdot), _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_out_proj rejected its arguments")
    return dict(out=out, amax=amax, absdot=absdot)


def ssd_prefill(xBC, z, dt, conv_w, conv_b, A, D, dt_bias, n_heads, head_dim, n_groups, d_state,
                conv_state_in=None, ssm_state_in=None, heads=None, n_threads=None, lib=None):
    """Oracle prefill of the SSD (Mamba-2-style) mixer.

    xBC [batch, L, H*P + 2*G*N] (channels x | B | C), z [batch, L, H*P], dt [batch, L, H];
    conv_w [Cx, W], conv_b [Cx], A / D / dt_bias [H] (float32); optional float64 states
    conv_state_in [batch, W-1, Cx] and ssm_state_in [batch, H, P, N].  ``heads`` (optional
    index list) evaluates only those heads; the other heads' outputs, states and x conv
    channels are left NaN.
    Returns dict(out [b, L, H*P], conv_state [b, W-1, Cx], ssm_state [b, H, P, N]) in float64.
    """
    lib = lib or load()
    xr, code = _raw(xBC)
    zr, code_z = _raw(z)
    dtr, code_dt = _raw(dt)
    if len({code, code_z, code_dt}) != 1:
        raise TypeError("xBC, z, dt must share one dtype")
    conv_w, conv_b, A, D, dt_bias = map(_f32, (conv_w, conv_b, A, D, dt_bias))
    csi, ssi = _f64(conv_state_in), _f64(ssm_state_in)
    H, P, G, N = int(n_heads), int(head_dim), int(n_groups), int(d_state)
    batch, L, Cx = xr.shape
    if Cx != H * P + 2 * G * N or zr.shape != (batch, L, H * P) or dtr.shape != (batch, L, H):
        raise ValueError("inconsistent SSD shapes")
    W = conv_w.shape[-1]
    hl = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    out = np.full((batch, L, H * P), np.nan)
    cso = np.full((batch, W - 1, Cx), np.nan)
    sso = np.full((batch, H, P, N), np.nan)
    rc = lib.oracle_ssd_prefill(batch, L, H, P, G, N, W, code, _p(xr), _p(zr), _p(dtr), _p(conv_w),
                                _p(conv_b), _p(A), _p(D), _p(dt_bias), _p(csi), _p(ssi), _p(hl),
                                0 if hl is None else int(hl.size), _p(out), _p(cso), _p(sso),
                                _threads(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_ssd_prefill rejected its arguments (rc={rc})")
    return dict(out=out, conv_state=cso, ssm_state=sso)
