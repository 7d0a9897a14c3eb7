"""Thin ctypes binding over libssm (include/ssm.h): argument marshalling only.

Every function takes CUDA torch tensors, checks their layouts, passes raw device
pointers, element strides and the current torch stream to the C ABI, and raises
``SSMError`` on a negative status.  All compute happens in libssm's kernels;
there is no CPU or PyTorch fallback, and a missing library or device is an error.
Output tensors are allocated with torch when the caller does not pass them.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from .build import LIB

SSM_F32, SSM_BF16 = 0, 1
_STATUS = {0: "SSM_OK", -1: "SSM_ERR_INVALID_ARG", -2: "SSM_ERR_UNSUPPORTED", -3: "SSM_ERR_MISALIGNED",
           -4: "SSM_ERR_CUDA", -5: "SSM_ERR_DEVICE_TIMEOUT"}
DEV_WAIT_TIMEOUT, DEV_BAD_SLOT = 1, 2

EXPORTS = ("ssm_abi_version", "ssm_prefill", "ssm_prefill_workspace_bytes", "ssm_prefill_segmented",
           "ssm_prefill_segmented_noalloc", "ssm_decode_step", "ssm_decode_tokens", "ssm_out_proj_partial",
           "q8_reduce_partials", "q8_block_absmax", "q8_quantize_shared", "q8_sum_dequant",
           "ssd_prefill_workspace_bytes", "ssd_prefill", "ssd_decode_step",
           "ssm_selftest_expire_wait", "ssm_device_status", "ssm_last_error")
NOALLOC_SCRATCH_BYTES = 4 << 20     # SSM_NOALLOC_SCRATCH_BYTES


class SSMError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} -> {_STATUS.get(code, code)}: {msg}")
        self.code = code


_lib = None


def load(path: Path | str | None = None):
    """Load libssm.so (built by ``selective_state_space_prefill_gb300.build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else LIB
    if not p.exists():
        raise ImportError(f"libssm is not built ({p} missing): run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(str(p))
    P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.ssm_abi_version.argtypes = []
    lib.ssm_abi_version.restype = I
    lib.ssm_last_error.argtypes = []
    lib.ssm_last_error.restype = ctypes.c_char_p
    lib.ssm_prefill.argtypes = [I, I, I, I, I, I, I, P, P, P, L, L, P, P, P, P, P, P, P, P, P, L, L,
                                P, L, L, P, P, P]
    lib.ssm_prefill.restype = I
    lib.ssm_prefill_workspace_bytes.argtypes = [I, I, I, I]
    lib.ssm_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.ssm_prefill_segmented.argtypes = lib.ssm_prefill.argtypes[:-1] + [I, P, ctypes.c_size_t, P]
    lib.ssm_prefill_segmented.restype = I
    lib.ssm_prefill_segmented_noalloc.argtypes = lib.ssm_prefill.argtypes[:-1] + [I, P]
    lib.ssm_prefill_segmented_noalloc.restype = I
    lib.ssm_decode_step.argtypes = [I, I, I, I, I, I, P, P, P, L, P, P, P, P, P, P, P, P, P, L, L, I, P,
                                    P, L, P]
    lib.ssm_decode_step.restype = I
    lib.ssm_decode_tokens.argtypes = [I, I, I, I, I, I, I, P, P, P, L, L, P, P, P, P, P, P, P, P, P, L, L, I,
                                      P, P, L, L, P]
    lib.ssm_decode_tokens.restype = I
    lib.ssm_out_proj_partial.argtypes = [L, L, L, P, L, P, L, I, P, L, P, P]
    lib.ssm_out_proj_partial.restype = I
    lib.q8_reduce_partials.argtypes = [I, P, I, L, I, P, I, P, P, P]
    lib.q8_reduce_partials.restype = I
    lib.q8_block_absmax.argtypes = [P, I, L, I, P, P]
    lib.q8_block_absmax.restype = I
    lib.q8_quantize_shared.argtypes = [P, I, L, I, P, P, P, P]
    lib.q8_quantize_shared.restype = I
    lib.q8_sum_dequant.argtypes = [I, P, P, L, I, P, I, P, P]
    lib.q8_sum_dequant.restype = I
    lib.ssd_prefill_workspace_bytes.argtypes = [I, I, I, I]
    lib.ssd_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.ssd_prefill.argtypes = [I, I, I, I, I, I, I, I, I, P, L, L, P, L, L, P, L, L, P, P, P, P, P, P, P,
                                P, L, L, P, P, P, ctypes.c_size_t, P]
    lib.ssd_prefill.restype = I
    lib.ssd_decode_step.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, I, P, P, P]
    lib.ssd_decode_step.restype = I
    lib.ssm_selftest_expire_wait.argtypes = [I, P]
    lib.ssm_selftest_expire_wait.restype = I
    lib.ssm_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), I]
    lib.ssm_device_status.restype = I
    if path is None:
        _lib = lib
    return lib


def _check(lib, fn: str, rc: int):
    if rc != 0:
        raise SSMError(fn, rc, lib.ssm_last_error().decode())


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SSM_F32
    if t == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported dtype {t} (float32 or bfloat16)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libssm takes CUDA tensors only (no CPU path)")


def _chan_contig(t, name):
    if t.stride(-1) != 1:
        raise ValueError(f"{name} must have channel stride 1")


def _param(t, shape, name):
    if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be contiguous float32 {tuple(shape)}")


def _conv_state_layout(t, batch, d_inner, name):
    if t.dtype != torch.float32 or tuple(t.shape) != (batch, 3, d_inner) or t.stride(2) != 1 \
            or t.stride(0) != 3 * t.stride(1):
        raise ValueError(f"{name} must be float32 [batch, 3, d_inner] with rows of one stride")
    return t.stride(1)


def _ssm_state_layout(t, batch, d_inner, name):
    if t.dtype != torch.float32 or tuple(t.shape) != (batch, d_inner, 16) or t.stride(2) != 1 \
            or t.stride(1) != 16:
        raise ValueError(f"{name} must be float32 [batch, d_inner, 16] with channel stride 16")
    return t.stride(0)


def prefill_workspace_bytes(batch: int, seqlen: int, d_inner: int, seg_len: int) -> int:
    """ssm_prefill_workspace_bytes: device bytes the segmented prefill needs."""
    return int(load().ssm_prefill_workspace_bytes(batch, seqlen, d_inner, seg_len))


def suggest_seg_len(batch: int, seqlen: int, d_inner: int, n_sm: int, ctas_per_sm: int = 3) -> int | None:
    """A segment length that brings batch x ceil(d_inner/16) x segments close to the GPU's
    resident CTA slots, or None when the rows already fill it.  The choice depends on
    d_inner, so channel-slice runs that must match bit for bit pass one seg_len explicitly."""
    rows = batch * ((d_inner + 15) // 16)
    slots = n_sm * ctas_per_sm
    n_seg = min(slots // rows if rows else 1, (seqlen + 63) // 64)
    if n_seg < 2:
        return None
    return ((seqlen + n_seg - 1) // n_seg + 63) // 64 * 64


def prefill(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state_in=None, ssm_state_in=None,
            out=None, out_dtype=torch.float32, conv_state_out=None, ssm_state_out=None, stream=None,
            seg_len=None, workspace=None, noalloc=False):
    """ssm_prefill over [batch, L, d_inner] x/z/dt (channel-stride-1 views allowed).

    With ``seg_len`` (a multiple of 64) the rows are cut into segments that run in parallel
    (ssm_prefill_segmented); ``workspace`` is then a CUDA uint8 tensor of at least
    prefill_workspace_bytes(...) bytes, allocated here with torch when not given.  With
    ``noalloc=True`` (and ``seg_len``) the call is ssm_prefill_segmented_noalloc: the scratch
    is the library's fixed array of NOALLOC_SCRATCH_BYTES and no workspace is allocated.
    Returns (out, conv_state_out, ssm_state_out).
    """
    lib = load()
    _need_cuda(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state_in, ssm_state_in)
    batch, L, d_inner = x.shape
    if z.shape != x.shape or dt.shape != x.shape or z.stride() != x.stride() or dt.stride() != x.stride():
        raise ValueError("x, z, dt must share shape and strides")
    if z.dtype != x.dtype or dt.dtype != x.dtype or B.dtype != x.dtype or C.dtype != x.dtype:
        raise ValueError("x, z, dt, B, C must share one dtype")
    for t, n in ((x, "x"),):
        _chan_contig(t, n)
    for t, n in ((B, "B"), (C, "C")):
        if tuple(t.shape) != (batch, L, 16) or not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous [batch, L, 16]")
    _param(A, (d_inner, 16), "A")
    for t, n in ((D, "D"), (dt_bias, "dt_bias"), (conv_b, "conv_b")):
        _param(t, (d_inner,), n)
    _param(conv_w, (d_inner, 4), "conv_w")
    dev = x.device
    if out is None:
        out = torch.empty(batch, L, d_inner, device=dev, dtype=out_dtype)
    _chan_contig(out, "out")
    if conv_state_out is None:
        conv_state_out = torch.empty(batch, 3, d_inner, device=dev, dtype=torch.float32)
    if ssm_state_out is None:
        ssm_state_out = torch.empty(batch, d_inner, 16, device=dev, dtype=torch.float32)
    ld = _conv_state_layout(conv_state_out, batch, d_inner, "conv_state_out")
    sb = _ssm_state_layout(ssm_state_out, batch, d_inner, "ssm_state_out")
    if conv_state_in is not None and _conv_state_layout(conv_state_in, batch, d_inner, "conv_state_in") != ld:
        raise ValueError("conv_state_in and conv_state_out must share the row stride")
    if ssm_state_in is not None and _ssm_state_layout(ssm_state_in, batch, d_inner, "ssm_state_in") != sb:
        raise ValueError("ssm_state_in and ssm_state_out must share the batch stride")
    args = (batch, L, d_inner, 16, 4, _dtype_code(x.dtype), _dtype_code(out.dtype),
            _ptr(x), _ptr(z), _ptr(dt), x.stride(0), x.stride(1), _ptr(B), _ptr(C),
            _ptr(A), _ptr(D), _ptr(dt_bias), _ptr(conv_w), _ptr(conv_b),
            _ptr(conv_state_in), _ptr(ssm_state_in), ld, sb,
            _ptr(out), out.stride(0), out.stride(1),
            _ptr(conv_state_out), _ptr(ssm_state_out))
    if seg_len is None:
        rc = lib.ssm_prefill(*args, _stream(stream))
        _check(lib, "ssm_prefill", rc)
        return out, conv_state_out, ssm_state_out
    if noalloc:
        if workspace is not None:
            raise ValueError("noalloc=True takes no workspace")
        rc = lib.ssm_prefill_segmented_noalloc(*args, int(seg_len), _stream(stream))
        _check(lib, "ssm_prefill_segmented_noalloc", rc)
        return out, conv_state_out, ssm_state_out
    need = int(lib.ssm_prefill_workspace_bytes(batch, L, d_inner, int(seg_len)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    if workspace is not None:
        _need_cuda(workspace)
        if not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.ssm_prefill_segmented(*args, int(seg_len), _ptr(workspace), ws_bytes, _stream(stream))
    _check(lib, "ssm_prefill_segmented", rc)
    return out, conv_state_out, ssm_state_out


def decode_step(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state, ssm_state, state_slot=None,
                out=None, out_dtype=torch.float32, stream=None):
    """ssm_decode_step: x/z/dt [batch, d_inner], B/C [batch, 16]; states updated in place.

    conv_state [n_slots, 3, d_inner], ssm_state [n_slots, d_inner, 16] (channel-slice views allowed).
    Returns out [batch, d_inner].
    """
    lib = load()
    _need_cuda(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state, ssm_state, state_slot)
    batch, d_inner = x.shape
    if z.shape != x.shape or dt.shape != x.shape or z.stride() != x.stride() or dt.stride() != x.stride():
        raise ValueError("x, z, dt must share shape and strides")
    _chan_contig(x, "x")
    for t, n in ((B, "B"), (C, "C")):
        if tuple(t.shape) != (batch, 16) or not t.is_contiguous() or t.dtype != x.dtype:
            raise ValueError(f"{n} must be contiguous [batch, 16] of the input dtype")
    _param(A, (d_inner, 16), "A")
    for t, n in ((D, "D"), (dt_bias, "dt_bias"), (conv_b, "conv_b")):
        _param(t, (d_inner,), n)
    _param(conv_w, (d_inner, 4), "conv_w")
    n_slots = conv_state.shape[0]
    if ssm_state.shape[0] != n_slots:
        raise ValueError("conv_state and ssm_state must have the same number of slots")
    ld = _conv_state_layout(conv_state, n_slots, d_inner, "conv_state")
    sb = _ssm_state_layout(ssm_state, n_slots, d_inner, "ssm_state")
    if state_slot is not None and (state_slot.dtype != torch.int32 or tuple(state_slot.shape) != (batch,)
                                   or not state_slot.is_contiguous()):
        raise ValueError("state_slot must be contiguous int32 [batch]")
    if out is None:
        out = torch.empty(batch, d_inner, device=x.device, dtype=out_dtype)
    _chan_contig(out, "out")
    rc = lib.ssm_decode_step(batch, d_inner, 16, 4, _dtype_code(x.dtype), _dtype_code(out.dtype),
                             _ptr(x), _ptr(z), _ptr(dt), x.stride(0), _ptr(B), _ptr(C),
                             _ptr(A), _ptr(D), _ptr(dt_bias), _ptr(conv_w), _ptr(conv_b),
                             _ptr(conv_state), _ptr(ssm_state), ld, sb, n_slots, _ptr(state_slot),
                             _ptr(out), out.stride(0), _stream(stream))
    _check(lib, "ssm_decode_step", rc)
    return out


def decode_tokens(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state, ssm_state, state_slot=None,
                  out=None, out_dtype=torch.float32, stream=None):
    """ssm_decode_tokens: x/z/dt [batch, T, d_inner] (channel-stride-1 views), B/C [batch, T, 16];
    the cached states (as for decode_step) advance T tokens in place.  Returns out [batch, T, d_inner]."""
    lib = load()
    _need_cuda(x, z, dt, B, C, A, D, dt_bias, conv_w, conv_b, conv_state, ssm_state, state_slot)
    batch, T, d_inner = x.shape
    if z.shape != x.shape or dt.shape != x.shape or z.stride() != x.stride() or dt.stride() != x.stride():
        raise ValueError("x, z, dt must share shape and strides")
    _chan_contig(x, "x")
    for t, n in ((B, "B"), (C, "C")):
        if tuple(t.shape) != (batch, T, 16) or not t.is_contiguous() or t.dtype != x.dtype:
            raise ValueError(f"{n} must be contiguous [batch, T, 16] of the input dtype")
    _param(A, (d_inner, 16), "A")
    for t, n in ((D, "D"), (dt_bias, "dt_bias"), (conv_b, "conv_b")):
        _param(t, (d_inner,), n)
    _param(conv_w, (d_inner, 4), "conv_w")
    n_slots = conv_state.shape[0]
    if ssm_state.shape[0] != n_slots:
        raise ValueError("conv_state and ssm_state must have the same number of slots")
    ld = _conv_state_layout(conv_state, n_slots, d_inner, "conv_state")
    sb = _ssm_state_layout(ssm_state, n_slots, d_inner, "ssm_state")
    if state_slot is not None and (state_slot.dtype != torch.int32 or tuple(state_slot.shape) != (batch,)
                                   or not state_slot.is_contiguous()):
        raise ValueError("state_slot must be contiguous int32 [batch]")
    if out is None:
        out = torch.empty(batch, T, d_inner, device=x.device, dtype=out_dtype)
    _chan_contig(out, "out")
    rc = lib.ssm_decode_tokens(batch, T, d_inner, 16, 4, _dtype_code(x.dtype), _dtype_code(out.dtype),
                               _ptr(x), _ptr(z), _ptr(dt), x.stride(0), x.stride(1), _ptr(B), _ptr(C),
                               _ptr(A), _ptr(D), _ptr(dt_bias), _ptr(conv_w), _ptr(conv_b),
                               _ptr(conv_state), _ptr(ssm_state), ld, sb, n_slots, _ptr(state_slot),
                               _ptr(out), out.stride(0), out.stride(1), _stream(stream))
    _check(lib, "ssm_decode_tokens", rc)
    return out


def q8_reduce(partials, block=128, out=None, out_dtype=None, sums=None, scales=None, stream=None):
    """q8_reduce_partials over P equal-shaped partial tensors (flattened).

    Returns (out, sums, scales); pass sums=False / scales=False to skip writing them.
    """
    lib = load()
    _need_cuda(*partials)
    P = len(partials)
    shape, dtype = partials[0].shape, partials[0].dtype
    for p in partials:
        if p.shape != shape or p.dtype != dtype or not p.is_contiguous():
            raise ValueError("partials must be contiguous tensors of one shape and dtype")
    n = partials[0].numel()
    dev = partials[0].device
    out_dtype = out_dtype or dtype
    if out is None:
        out = torch.empty(shape, device=dev, dtype=out_dtype)
    if sums is None:
        sums = torch.empty(n, device=dev, dtype=torch.int32)
    if scales is None:
        scales = torch.empty((n + block - 1) // block, device=dev, dtype=torch.float32)
    sums = sums if sums is not False else None
    scales = scales if scales is not False else None
    ptrs = (ctypes.c_void_p * P)(*[p.data_ptr() for p in partials])
    rc = lib.q8_reduce_partials(P, ctypes.cast(ptrs, ctypes.c_void_p), _dtype_code(dtype), n, block,
                                _ptr(out), _dtype_code(out.dtype), _ptr(sums), _ptr(scales), _stream(stream))
    _check(lib, "q8_reduce_partials", rc)
    return out, sums, scales


def q8_block_absmax(x, block=128, out=None, stream=None):
    """q8_block_absmax: per-128-block maxima of |x| (x flattened, contiguous) -> float32 [nblk]."""
    lib = load()
    _need_cuda(x, out)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    n = x.numel()
    if out is None:
        out = torch.empty((n + block - 1) // block, device=x.device, dtype=torch.float32)
    rc = lib.q8_block_absmax(_ptr(x), _dtype_code(x.dtype), n, block, _ptr(out), _stream(stream))
    _check(lib, "q8_block_absmax", rc)
    return out


def q8_quantize_shared(x, block_amax, block=128, codes=None, scales=None, stream=None):
    """q8_quantize_shared: int8 codes of x with the shared per-block maxima.

    Returns (codes int8 shaped like x, scales float32 [nblk]); pass scales=False to skip them.
    """
    lib = load()
    _need_cuda(x, block_amax, codes)
    if not x.is_contiguous() or not block_amax.is_contiguous() or block_amax.dtype != torch.float32:
        raise ValueError("x and block_amax (float32) must be contiguous")
    n = x.numel()
    nblk = (n + block - 1) // block
    if block_amax.numel() != nblk:
        raise ValueError(f"block_amax holds {block_amax.numel()} maxima, {nblk} needed")
    if codes is None:
        codes = torch.empty(x.shape, device=x.device, dtype=torch.int8)
    if scales is None:
        scales = torch.empty(nblk, device=x.device, dtype=torch.float32)
    scales = scales if scales is not False else None
    rc = lib.q8_quantize_shared(_ptr(x), _dtype_code(x.dtype), n, block, _ptr(block_amax), _ptr(codes),
                                _ptr(scales), _stream(stream))
    _check(lib, "q8_quantize_shared", rc)
    return codes, scales


def q8_sum_dequant(codes, scales, block=128, out=None, out_dtype=torch.float32, sums=None, stream=None):
    """q8_sum_dequant over P equal-shaped int8 code tensors with their shared scales.

    Returns (out, sums int32 [n]); pass sums=False to skip them.
    """
    lib = load()
    _need_cuda(*codes, scales, out)
    P = len(codes)
    shape = codes[0].shape
    for c in codes:
        if c.shape != shape or c.dtype != torch.int8 or not c.is_contiguous():
            raise ValueError("codes must be contiguous int8 tensors of one shape")
    n = codes[0].numel()
    dev = codes[0].device
    if out is None:
        out = torch.empty(shape, device=dev, dtype=out_dtype)
    if sums is None:
        sums = torch.empty(n, device=dev, dtype=torch.int32)
    sums = sums if sums is not False else None
    ptrs = (ctypes.c_void_p * P)(*[c.data_ptr() for c in codes])
    rc = lib.q8_sum_dequant(P, ctypes.cast(ptrs, ctypes.c_void_p), _ptr(scales), n, block, _ptr(out),
                            _dtype_code(out.dtype), _ptr(sums), _stream(stream))
    _check(lib, "q8_sum_dequant", rc)
    return out, sums


def device_status(clear: bool = True) -> int:
    """The device status word (OR of DEV_* bits); synchronises the device."""
    lib = load()
    v = ctypes.c_uint32(0)
    _check(lib, "ssm_device_status", lib.ssm_device_status(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def out_proj_partial(y, W, out=None, out_dtype=torch.bfloat16, block_amax=True, stream=None):
    """ssm_out_proj_partial: y [M, K] bf16 and W [N, K] bf16 (row views with stride-1 K).

    Returns (out [M, N], block_amax [M*N/128] float32 or None).
    """
    lib = load()
    _need_cuda(y, W, out)
    if y.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("y and W must be bfloat16")
    if y.dim() != 2 or W.dim() != 2 or y.stride(1) != 1 or W.stride(1) != 1 or y.shape[1] != W.shape[1]:
        raise ValueError("y [M, K] and W [N, K] must be 2-D with a stride-1 K dimension")
    M, K = y.shape
    N = W.shape[0]
    if out is None:
        out = torch.empty(M, N, device=y.device, dtype=out_dtype)
    if out.dim() != 2 or tuple(out.shape) != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with a stride-1 N dimension")
    amax = None
    if block_amax is True:
        amax = torch.empty((M * N + 127) // 128, device=y.device, dtype=torch.float32)
    elif block_amax is not None and block_amax is not False:
        amax = block_amax
    rc = lib.ssm_out_proj_partial(M, N, K, _ptr(y), y.stride(0), _ptr(W), W.stride(0), _dtype_code(out.dtype),
                                  _ptr(out), out.stride(0), _ptr(amax), _stream(stream))
    _check(lib, "ssm_out_proj_partial", rc)
    return out, amax


def selftest_expire_wait(limit_us: int = 50000, stream=None) -> None:
    """ssm_selftest_expire_wait: one kernel whose bounded wait expires after limit_us."""
    lib = load()
    _check(lib, "ssm_selftest_expire_wait", lib.ssm_selftest_expire_wait(int(limit_us), _stream(stream)))


# ------------------------------------------------------------------ SSD (Mamba-2-style) mixer
def _ssd_dims(n_heads, n_groups, head_dim=64, d_state=64):
    return n_heads * head_dim, n_heads * head_dim + 2 * n_groups * d_state


def ssd_prefill_workspace_bytes(batch: int, seqlen: int, n_heads: int, n_groups: int) -> int:
    """ssd_prefill_workspace_bytes: device bytes ssd_prefill needs."""
    return int(load().ssd_prefill_workspace_bytes(batch, seqlen, n_heads, n_groups))


def _ssd_params(conv_w, conv_b, A, D, dt_bias, H, Cx):
    _param(conv_w, (Cx, 4), "conv_w")
    _param(conv_b, (Cx,), "conv_b")
    for t, n in ((A, "A"), (D, "D"), (dt_bias, "dt_bias")):
        _param(t, (H,), n)


def _ssd_states(t, batch, H, Cx, name, conv):
    shape = (batch, 3, Cx) if conv else (batch, H, 64, 64)
    if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous float32 {shape}")


def ssd_prefill(xBC, z, dt, conv_w, conv_b, A, D, dt_bias, n_heads, n_groups, conv_state_in=None,
                ssm_state_in=None, out=None, out_dtype=torch.float32, conv_state_out=None, ssm_state_out=None,
                workspace=None, stream=None):
    """ssd_prefill: xBC [batch, L, 64 H + 128 G], z [batch, L, 64 H], dt [batch, L, H] bf16
    (channel-stride-1 views), head_dim = d_state = 64.  ``workspace`` (a CUDA uint8 tensor of at
    least ssd_prefill_workspace_bytes(batch, L, n_heads, n_groups) bytes) is allocated here with torch when not given.
    Returns (out [batch, L, 64 H], conv_state_out [batch, 3, Cx], ssm_state_out [batch, H, 64, 64])."""
    lib = load()
    _need_cuda(xBC, z, dt, conv_w, conv_b, A, D, dt_bias, conv_state_in, ssm_state_in)
    H, G = int(n_heads), int(n_groups)
    HP, Cx = _ssd_dims(H, G)
    batch, L, cx = xBC.shape
    if cx != Cx or tuple(z.shape) != (batch, L, HP) or tuple(dt.shape) != (batch, L, H):
        raise ValueError("xBC, z, dt shapes disagree with n_heads / n_groups")
    if z.dtype != xBC.dtype or dt.dtype != xBC.dtype:
        raise ValueError("xBC, z, dt must share one dtype")
    for t, n in ((xBC, "xBC"), (z, "z"), (dt, "dt")):
        _chan_contig(t, n)
    _ssd_params(conv_w, conv_b, A, D, dt_bias, H, Cx)
    dev = xBC.device
    if out is None:
        out = torch.empty(batch, L, HP, device=dev, dtype=out_dtype)
    _chan_contig(out, "out")
    if conv_state_out is None:
        conv_state_out = torch.empty(batch, 3, Cx, device=dev, dtype=torch.float32)
    if ssm_state_out is None:
        ssm_state_out = torch.empty(batch, H, 64, 64, device=dev, dtype=torch.float32)
    for t, n, c in ((conv_state_out, "conv_state_out", True), (ssm_state_out, "ssm_state_out", False),
                    (conv_state_in, "conv_state_in", True), (ssm_state_in, "ssm_state_in", False)):
        if t is not None:
            _ssd_states(t, batch, H, Cx, n, c)
    need = int(lib.ssd_prefill_workspace_bytes(batch, L, H, G))
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    _need_cuda(workspace)
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    rc = lib.ssd_prefill(batch, L, H, 64, G, 64, 4, _dtype_code(xBC.dtype), _dtype_code(out.dtype),
                         _ptr(xBC), xBC.stride(0), xBC.stride(1), _ptr(z), z.stride(0), z.stride(1),
                         _ptr(dt), dt.stride(0), dt.stride(1), _ptr(conv_w), _ptr(conv_b), _ptr(A), _ptr(D),
                         _ptr(dt_bias), _ptr(conv_state_in), _ptr(ssm_state_in), _ptr(out), out.stride(0),
                         out.stride(1), _ptr(conv_state_out), _ptr(ssm_state_out), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check(lib, "ssd_prefill", rc)
    return out, conv_state_out, ssm_state_out


def ssd_decode_step(xBC, z, dt, conv_w, conv_b, A, D, dt_bias, n_heads, n_groups, conv_state, ssm_state,
                    state_slot=None, out=None, out_dtype=torch.float32, stream=None):
    """ssd_decode_step: xBC [batch, Cx], z [batch, 64 H], dt [batch, H] (contiguous); the cached
    states conv_state [n_slots, 3, Cx] and ssm_state [n_slots, H, 64, 64] advance one token in
    place.  Returns out [batch, 64 H]."""
    lib = load()
    _need_cuda(xBC, z, dt, conv_w, conv_b, A, D, dt_bias, conv_state, ssm_state, state_slot)
    H, G = int(n_heads), int(n_groups)
    HP, Cx = _ssd_dims(H, G)
    batch = xBC.shape[0]
    if tuple(xBC.shape) != (batch, Cx) or tuple(z.shape) != (batch, HP) or tuple(dt.shape) != (batch, H):
        raise ValueError("xBC, z, dt shapes disagree with n_heads / n_groups")
    if z.dtype != xBC.dtype or dt.dtype != xBC.dtype:
        raise ValueError("xBC, z, dt must share one dtype")
    for t, n in ((xBC, "xBC"), (z, "z"), (dt, "dt")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _ssd_params(conv_w, conv_b, A, D, dt_bias, H, Cx)
    n_slots = conv_state.shape[0]
    _ssd_states(conv_state, n_slots, H, Cx, "conv_state", True)
    _ssd_states(ssm_state, n_slots, H, Cx, "ssm_state", False)
    if state_slot is not None and (state_slot.dtype != torch.int32 or tuple(state_slot.shape) != (batch,)
                                   or not state_slot.is_contiguous()):
        raise ValueError("state_slot must be contiguous int32 [batch]")
    if out is None:
        out = torch.empty(batch, HP, device=xBC.device, dtype=out_dtype)
    if not out.is_contiguous() or tuple(out.shape) != (batch, HP):
        raise ValueError("out must be contiguous [batch, 64 H]")
    rc = lib.ssd_decode_step(batch, H, 64, G, 64, 4, _dtype_code(xBC.dtype), _dtype_code(out.dtype),
                             _ptr(xBC), _ptr(z), _ptr(dt), _ptr(conv_w), _ptr(conv_b), _ptr(A), _ptr(D),
                             _ptr(dt_bias), _ptr(conv_state), _ptr(ssm_state), n_slots, _ptr(state_slot),
                             _ptr(out), _stream(stream))
    _check(lib, "ssd_decode_step", rc)
    return out
