"""Host-side checks of the C ABI that need no GPU.

* libssm.so builds for sm_103a and exports every function include/ssm.h declares;
* argument validation returns the documented status before any CUDA call
  (pointers here are fake and never dereferenced: every call is rejected first).
"""
import ctypes
import re
from pathlib import Path

import pytest

from selective_state_space_prefill_gb300 import binding, build

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "ssm.h"

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA = 0, -1, -2, -3, -4


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"^(?:int|size_t|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for fn in ("ssm_prefill", "ssm_decode_step", "q8_reduce_partials"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS)
    for fn in names:
        assert hasattr(lib, fn), fn
    assert lib.ssm_abi_version() == 108


FAKE = 0x10000  # 64 KiB-aligned fake device address, never dereferenced


def _prefill(lib, **kw):
    a = dict(batch=2, seqlen=16, d_inner=64, d_state=16, d_conv=4, in_dtype=1, out_dtype=0,
             x=FAKE, z=FAKE, dt=FAKE, in_stride_b=16 * 64, in_stride_t=64, B=FAKE, C=FAKE, A=FAKE,
             D=FAKE, dt_bias=FAKE, conv_w=FAKE, conv_b=FAKE, csi=None, ssi=None, ld=64, sb=64 * 16,
             out=FAKE, ob=16 * 64, ot=64, cso=FAKE, sso=FAKE, stream=None)
    a.update(kw)
    return lib.ssm_prefill(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), INVALID), (dict(seqlen=0), INVALID), (dict(d_inner=0), INVALID),
    (dict(in_dtype=7), INVALID), (dict(d_state=8), UNSUPPORTED), (dict(d_conv=3), UNSUPPORTED),
    (dict(d_inner=60, in_stride_t=60, ld=60, sb=960), UNSUPPORTED), (dict(x=None), INVALID),
    (dict(sso=None), INVALID), (dict(in_stride_t=32), INVALID), (dict(ob=64), INVALID),
    (dict(ld=32), INVALID), (dict(sb=100), INVALID), (dict(x=FAKE + 8), MISALIGNED),
    (dict(in_stride_t=68), MISALIGNED), (dict(A=FAKE + 4), MISALIGNED), (dict(sso=FAKE + 4), MISALIGNED),
])
def test_prefill_rejects_bad_arguments(lib, kw, code):
    assert _prefill(lib, **kw) == code
    assert lib.ssm_last_error().decode().startswith("ssm_prefill")


def _decode(lib, **kw):
    a = dict(batch=4, d_inner=64, d_state=16, d_conv=4, in_dtype=1, out_dtype=0, x=FAKE, z=FAKE,
             dt=FAKE, sx=64, B=FAKE, C=FAKE, A=FAKE, D=FAKE, dt_bias=FAKE, conv_w=FAKE, conv_b=FAKE,
             cs=FAKE, ss=FAKE, ld=64, sb=1024, n_slots=4, slot=None, out=FAKE, so=64, stream=None)
    a.update(kw)
    return lib.ssm_decode_step(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), INVALID), (dict(d_state=32), UNSUPPORTED), (dict(cs=None), INVALID),
    (dict(n_slots=2), INVALID), (dict(sx=32), INVALID), (dict(ss=FAKE + 8), MISALIGNED),
    (dict(B=FAKE + 2), MISALIGNED),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert _decode(lib, **kw) == code


def _q8(lib, P=4, ptrs=None, **kw):
    arr = (ctypes.c_void_p * max(P, 1))(*(ptrs or [FAKE] * max(P, 1)))
    a = dict(P=P, partials=ctypes.cast(arr, ctypes.c_void_p), dtype=1, n=4096, block=128, out=FAKE,
             out_dtype=1, sums=None, scales=None, stream=None)
    a.update(kw)
    return lib.q8_reduce_partials(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(P=0), UNSUPPORTED), (dict(P=9), UNSUPPORTED), (dict(n=0), INVALID), (dict(block=64), UNSUPPORTED),
    (dict(out=None), INVALID), (dict(ptrs=[FAKE, FAKE + 8, FAKE, FAKE]), MISALIGNED),
    (dict(partials=None), INVALID),
])
def test_q8_rejects_bad_arguments(lib, kw, code):
    assert _q8(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), INVALID), (dict(amax=None), INVALID), (dict(n=0), INVALID), (dict(block=256), UNSUPPORTED),
    (dict(dtype=5), INVALID), (dict(x=FAKE + 2), MISALIGNED),
])
def test_q8_block_absmax_rejects_bad_arguments(lib, kw, code):
    a = dict(x=FAKE, dtype=1, n=4096, block=128, amax=FAKE, stream=None)
    a.update(kw)
    assert lib.q8_block_absmax(*a.values()) == code
    assert lib.ssm_last_error().decode().startswith("q8_block_absmax")


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), INVALID), (dict(amax=None), INVALID), (dict(codes=None), INVALID), (dict(n=0), INVALID),
    (dict(block=64), UNSUPPORTED), (dict(dtype=3), INVALID), (dict(codes=FAKE + 8), MISALIGNED),
    (dict(x=FAKE + 4), MISALIGNED), (dict(scales=FAKE + 2), MISALIGNED),
])
def test_q8_quantize_shared_rejects_bad_arguments(lib, kw, code):
    a = dict(x=FAKE, dtype=1, n=4096, block=128, amax=FAKE, codes=FAKE, scales=None, stream=None)
    a.update(kw)
    assert lib.q8_quantize_shared(*a.values()) == code
    assert lib.ssm_last_error().decode().startswith("q8_quantize_shared")


def _q8_sum(lib, P=4, ptrs=None, **kw):
    arr = (ctypes.c_void_p * max(P, 1))(*(ptrs or [FAKE] * max(P, 1)))
    a = dict(P=P, codes=ctypes.cast(arr, ctypes.c_void_p), scales=FAKE, n=4096, block=128, out=FAKE,
             out_dtype=1, sums=None, stream=None)
    a.update(kw)
    return lib.q8_sum_dequant(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(P=0), UNSUPPORTED), (dict(P=9), UNSUPPORTED), (dict(n=0), INVALID), (dict(block=32), UNSUPPORTED),
    (dict(out=None), INVALID), (dict(scales=None), INVALID), (dict(codes=None), INVALID),
    (dict(ptrs=[FAKE, None, FAKE, FAKE]), INVALID), (dict(ptrs=[FAKE, FAKE + 1, FAKE, FAKE]), MISALIGNED),
    (dict(out_dtype=9), INVALID), (dict(sums=FAKE + 4), MISALIGNED),
])
def test_q8_sum_dequant_rejects_bad_arguments(lib, kw, code):
    assert _q8_sum(lib, **kw) == code
    assert lib.ssm_last_error().decode().startswith("q8_sum_dequant")


def test_valid_call_without_gpu_fails_cleanly(lib):
    """A well-formed call on a machine without a usable GPU returns SSM_ERR_CUDA, not a crash."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _prefill(lib) == CUDA


def _tokens(lib, **kw):
    a = dict(batch=4, T=3, d_inner=64, d_state=16, d_conv=4, in_dtype=1, out_dtype=0, x=FAKE, z=FAKE, dt=FAKE,
             sb=3 * 64, st=64, B=FAKE, C=FAKE, A=FAKE, D=FAKE, dt_bias=FAKE, conv_w=FAKE, conv_b=FAKE,
             cs=FAKE, ss=FAKE, ld=64, ssb=1024, n_slots=4, slot=None, out=FAKE, ob=3 * 64, ot=64, stream=None)
    a.update(kw)
    return lib.ssm_decode_tokens(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), INVALID), (dict(T=5000), INVALID), (dict(st=32), INVALID), (dict(ot=32), INVALID),
    (dict(ob=64), INVALID), (dict(sb=64), INVALID), (dict(d_state=8), UNSUPPORTED), (dict(ss=FAKE + 4), MISALIGNED),
])
def test_decode_tokens_rejects_bad_arguments(lib, kw, code):
    assert _tokens(lib, **kw) == code
    assert lib.ssm_last_error().decode().startswith("ssm_decode_tokens")


def _segmented(lib, seg_len=64, ws=FAKE, ws_bytes=1 << 20, **kw):
    a = dict(batch=2, seqlen=200, d_inner=64, d_state=16, d_conv=4, in_dtype=1, out_dtype=0,
             x=FAKE, z=FAKE, dt=FAKE, in_stride_b=200 * 64, in_stride_t=64, B=FAKE, C=FAKE, A=FAKE,
             D=FAKE, dt_bias=FAKE, conv_w=FAKE, conv_b=FAKE, csi=None, ssi=None, ld=64, sb=64 * 16,
             out=FAKE, ob=200 * 64, ot=64, cso=FAKE, sso=FAKE)
    a.update(kw)
    return lib.ssm_prefill_segmented(*a.values(), seg_len, ws, ws_bytes, None)


def test_prefill_workspace_bytes(lib):
    # (ceil(L / seg_len) - 1) segments x batch x d_inner x 32 floats
    assert lib.ssm_prefill_workspace_bytes(2, 200, 64, 64) == 3 * 2 * 64 * 128
    assert lib.ssm_prefill_workspace_bytes(1, 16384, 2048, 4096) == 3 * 2048 * 128
    assert lib.ssm_prefill_workspace_bytes(4, 128, 64, 128) == 0          # one segment
    assert lib.ssm_prefill_workspace_bytes(4, 128, 64, 4096) == 0
    assert lib.ssm_prefill_workspace_bytes(0, 128, 64, 64) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(seg_len=0), INVALID), (dict(seg_len=96), INVALID), (dict(seg_len=-64), INVALID),
    (dict(ws=None), INVALID), (dict(ws_bytes=3 * 2 * 64 * 128 - 1), INVALID),
    (dict(ws=FAKE + 8), MISALIGNED), (dict(batch=0), INVALID), (dict(d_state=8), UNSUPPORTED),
    (dict(seqlen=64 * 65536, in_stride_b=0, batch=1, ob=0), INVALID),     # 65536 segments
])
def test_prefill_segmented_rejects_bad_arguments(lib, kw, code):
    assert _segmented(lib, **kw) == code
    assert lib.ssm_last_error().decode().startswith("ssm_prefill_segmented")


def test_prefill_segmented_single_segment_needs_no_workspace(lib):
    """seg_len >= seqlen is the plain prefill: no workspace, and a valid call on a machine
    without a GPU fails with SSM_ERR_CUDA only after validation."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _segmented(lib, seg_len=256, ws=None, ws_bytes=0) == CUDA
    assert _segmented(lib, seg_len=64, ws=FAKE, ws_bytes=3 * 2 * 64 * 128) == CUDA


def _noalloc(lib, seg_len=64, **kw):
    a = dict(batch=2, seqlen=200, d_inner=64, d_state=16, d_conv=4, in_dtype=1, out_dtype=0,
             x=FAKE, z=FAKE, dt=FAKE, in_stride_b=200 * 64, in_stride_t=64, B=FAKE, C=FAKE, A=FAKE,
             D=FAKE, dt_bias=FAKE, conv_w=FAKE, conv_b=FAKE, csi=None, ssi=None, ld=64, sb=64 * 16,
             out=FAKE, ob=200 * 64, ot=64, cso=FAKE, sso=FAKE)
    a.update(kw)
    return lib.ssm_prefill_segmented_noalloc(*a.values(), seg_len, None)


@pytest.mark.parametrize("kw,code,words", [
    # a bad seg_len or shape is reported as such, even when the sizes would also overflow the array
    (dict(seg_len=1, seqlen=1 << 20, d_inner=8192, in_stride_t=8192, in_stride_b=(1 << 20) * 8192,
          ld=8192, sb=8192 * 16, ot=8192, ob=(1 << 20) * 8192), INVALID, "seg_len 1"),
    (dict(seg_len=96), INVALID, "seg_len 96"),
    (dict(d_state=8), UNSUPPORTED, "d_state 8"),
    (dict(in_stride_t=32), INVALID, "in_stride_t"),
    # valid arguments whose scratch exceeds the fixed array: the array's limit is named
    (dict(seqlen=64 * 6, batch=1, d_inner=8192, in_stride_t=8192, in_stride_b=0, ld=8192, sb=8192 * 16,
          ot=8192, ob=0), INVALID, "fixed array holds"),
])
def test_noalloc_validates_arguments_before_the_scratch_limit(lib, kw, code, words):
    assert _noalloc(lib, **kw) == code
    msg = lib.ssm_last_error().decode()
    assert msg.startswith("ssm_prefill_segmented_noalloc") and words in msg, msg


def test_suggest_seg_len():
    # 96 channel groups x 1 row on 152 SMs x 3 slots: 4 segments of 512 tokens
    assert binding.suggest_seg_len(1, 2048, 1536, 152) == 512
    assert binding.suggest_seg_len(4, 2048, 1536, 152) is None           # 384 CTAs already
    assert binding.suggest_seg_len(1, 16384, 2048, 152) == 5504          # 3 segments
    assert binding.suggest_seg_len(1, 100, 64, 152) == 64
    assert binding.suggest_seg_len(1, 64, 64, 152) is None               # a single chunk


def _out_proj(lib, **kw):
    a = dict(M=256, N=768, K=1536, y=FAKE, ldy=1536, W=FAKE, ldw=1536, out_dtype=1, out=FAKE, ldo=768,
             amax=None, stream=None)
    a.update(kw)
    return lib.ssm_out_proj_partial(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), INVALID), (dict(N=0), INVALID), (dict(K=0), INVALID), (dict(out_dtype=5), INVALID),
    (dict(y=None), INVALID), (dict(N=700, ldo=704), UNSUPPORTED), (dict(K=1540, ldy=1544, ldw=1544), UNSUPPORTED),
    (dict(ldy=1024), INVALID), (dict(ldo=700), INVALID), (dict(ldw=1540), MISALIGNED),
    (dict(y=FAKE + 8), MISALIGNED), (dict(out=FAKE + 4), MISALIGNED), (dict(M=65535 * 128 + 1), INVALID),
    (dict(M=65535 * 128, N=65536 * 128, ldo=65536 * 128, K=1 << 20, ldy=1 << 20, ldw=1 << 20), UNSUPPORTED),
])
def test_out_proj_rejects_bad_arguments(lib, kw, code):
    assert _out_proj(lib, **kw) == code
    assert lib.ssm_last_error().decode().startswith("ssm_out_proj_partial")


@pytest.mark.parametrize("limit", [0, -5, 2000001])
def test_selftest_rejects_bad_limits(lib, limit):
    assert lib.ssm_selftest_expire_wait(limit, None) == INVALID


def _ssd(lib, ws_bytes=1 << 30, **kw):
    H, G, L = 4, 1, 300
    Cx = 64 * H + 128 * G
    a = dict(batch=2, seqlen=L, H=H, P=64, G=G, N=64, W=4, in_dtype=1, out_dtype=0,
             xBC=FAKE, xsb=L * Cx, xst=Cx, z=FAKE, zsb=L * 64 * H, zst=64 * H, dt=FAKE, dsb=L * H, dst=H,
             conv_w=FAKE, conv_b=FAKE, A=FAKE, D=FAKE, dt_bias=FAKE, csi=None, ssi=None,
             out=FAKE, osb=L * 64 * H, ost=64 * H, cso=FAKE, sso=FAKE, ws=FAKE)
    a.update(kw)
    return lib.ssd_prefill(*a.values(), ws_bytes, None)


def test_ssd_workspace_bytes(lib):
    # 4 bf16 planes [B*G][L][64], 2 bf16 planes [B*G][64][Lp], 2 fp32 planes [B*H][Lp]
    # (Lp = L rounded up to 128; each part starts on a 256-byte boundary), then min(B*H, 256)
    # fp32 hand-off states [64][64] and as many uint32 flags (the total rounded up to 16 bytes)
    up = lambda v: (v + 255) // 256 * 256
    up16 = lambda v: (v + 15) // 16 * 16
    a = up(4 * 4 * 2048 * 64 * 2)
    b = up(a + 2 * 4 * 64 * 2048 * 2)
    c = up(b + 2 * 4 * 80 * 2048 * 4)
    assert lib.ssd_prefill_workspace_bytes(4, 2048, 80, 1) == up16(c + 256 * 64 * 64 * 4 + 256 * 4)
    a = up(4 * 2 * 300 * 128)
    b = up(a + 2 * 2 * 64 * 384 * 2)
    c = up(b + 2 * 4 * 384 * 4)
    assert lib.ssd_prefill_workspace_bytes(1, 300, 4, 2) == up16(c + 4 * 64 * 64 * 4 + 4 * 4)
    assert lib.ssd_prefill_workspace_bytes(0, 300, 4, 2) == 0
    assert lib.ssd_prefill_workspace_bytes(1, 300, 3, 2) == 0           # groups must divide heads


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), INVALID), (dict(seqlen=0), INVALID), (dict(H=0), INVALID), (dict(G=3), INVALID),
    (dict(P=32), UNSUPPORTED), (dict(N=128), UNSUPPORTED), (dict(W=3), UNSUPPORTED), (dict(in_dtype=0), UNSUPPORTED),
    (dict(out_dtype=4), INVALID), (dict(xBC=None), INVALID), (dict(ws=None), INVALID), (dict(xst=100), INVALID),
    (dict(ost=64), INVALID), (dict(dsb=3), INVALID), (dict(ws_bytes=1000), INVALID), (dict(xBC=FAKE + 8), MISALIGNED),
    (dict(xst=388, xsb=300 * 388), MISALIGNED), (dict(out=FAKE + 4), MISALIGNED), (dict(sso=FAKE + 8), MISALIGNED),
    (dict(ws=FAKE + 8), MISALIGNED),
])
def test_ssd_prefill_rejects_bad_arguments(lib, kw, code):
    assert _ssd(lib, **kw) == code
    assert lib.ssm_last_error().decode().startswith("ssd_prefill")


def test_ssd_prefill_refuses_a_workspace_without_the_handoff_slots(lib):
    # (batch 2, L 300, 4 heads, 1 group): the planes end at 528 384 bytes; the hand-off slots and
    # their flags follow. A workspace sized for the planes alone, or one byte short, is refused
    # on the host.
    up = lambda v: (v + 255) // 256 * 256
    planes = up(up(4 * 2 * 300 * 64 * 2) + 2 * 2 * 64 * 384 * 2) + 2 * 8 * 384 * 4
    need = lib.ssd_prefill_workspace_bytes(2, 300, 4, 1)
    assert planes == 528384 and need > planes
    for ws_bytes in (planes, need - 1):
        assert _ssd(lib, ws_bytes=ws_bytes) == INVALID
        assert "workspace" in lib.ssm_last_error().decode()


def _ssd_dec(lib, **kw):
    a = dict(batch=2, H=4, P=64, G=2, N=64, W=4, in_dtype=1, out_dtype=0, xBC=FAKE, z=FAKE, dt=FAKE,
             conv_w=FAKE, conv_b=FAKE, A=FAKE, D=FAKE, dt_bias=FAKE, cs=FAKE, ss=FAKE, n_slots=2, slot=None,
             out=FAKE, stream=None)
    a.update(kw)
    return lib.ssd_decode_step(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), INVALID), (dict(G=3), INVALID), (dict(N=16), UNSUPPORTED), (dict(cs=None), INVALID),
    (dict(n_slots=1), INVALID), (dict(ss=FAKE + 4), MISALIGNED), (dict(xBC=FAKE + 1), MISALIGNED),
])
def test_ssd_decode_rejects_bad_arguments(lib, kw, code):
    assert _ssd_dec(lib, **kw) == code
    assert lib.ssm_last_error().decode().startswith("ssd_decode_step")


def test_ssd_valid_call_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _ssd(lib) == CUDA
    assert _ssd_dec(lib) == CUDA
