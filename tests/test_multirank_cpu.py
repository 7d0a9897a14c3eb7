"""The N > 1 path on the CPU with gloo ranks (world size 2 and 4), no GPU.

* Channel sharding (the pages' Methodology 1-2: the mixer is split along the
  feature dimension and every shard keeps its own state): ranks run disjoint
  channel slices and the gathered result equals the unsplit run exactly.
* The quantized all-reduce (Methodology 4) carried out across ranks -- all-reduce
  MAX of the per-block absolute maxima, local int8 quantization, all-reduce SUM
  of the int32 codes, dequantization -- equals the local q8 reduction of the same
  P partials bit for bit (this is what q8_reduce_partials computes on one GPU).
* tp.q8_all_reduce, the exchange as the library runs it between GPUs (block maxima, MAX
  all-reduce, shared-scale int8 codes, all-gather of the codes, local sum), with its
  rank-local arithmetic injected from the oracle: equal to the local reduction on every rank.
* The benchmark's cross-rank timing: the slowest rank's time and the whole-job rate.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(world, fn, *args):
    port = _free_port()
    mp.start_processes(_entry, args=(world, port, fn, args), nprocs=world, start_method="spawn", join=True)


def _entry(rank, world, port, fn, args):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        fn(rank, world, *args)
    finally:
        dist.destroy_process_group()


def _shard_prefill(rank, world):
    import oracle
    from selective_state_space_prefill_gb300.inputs import make_mixer_inputs
    D = 32
    inp = make_mixer_inputs(2, 40, D, dtype=torch.bfloat16, seed=3)
    lo, hi = rank * D // world, (rank + 1) * D // world
    part = oracle.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                          inp.conv_b, channels=list(range(lo, hi)), n_threads=1)
    pieces = [torch.empty(2, 40, hi - lo, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(pieces, torch.from_numpy(part["out"]))
    states = [torch.empty(2, hi - lo, 16, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(states, torch.from_numpy(part["ssm_state"]))
    if rank == 0:
        full = oracle.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                              inp.conv_b, n_threads=1)
        assert np.array_equal(torch.cat(pieces, 2).numpy(), full["out"])
        assert np.array_equal(torch.cat(states, 1).numpy(), full["ssm_state"])


def _quantized_allreduce(rank, world):
    import oracle
    from selective_state_space_prefill_gb300.inputs import make_partials
    n, block = 4096 + 50, 128
    parts = make_partials(world, (n,), dtype=torch.bfloat16, seed=21)
    x = parts[rank].float().numpy()                       # this rank's partial, fp32
    nblk = (n + block - 1) // block
    pad = np.zeros(nblk * block, np.float32)
    pad[:n] = np.abs(x)
    amax = torch.from_numpy(pad.reshape(nblk, block).max(1))
    dist.all_reduce(amax, op=dist.ReduceOp.MAX)           # shared per-block scale
    amax = amax.numpy().astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, np.float32(127.0) / amax, np.float32(0.0)).astype(np.float32)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    q = np.rint((x * np.repeat(inv, block)[:n]).astype(np.float32))
    q = np.clip(q, -127, 127).astype(np.int32)
    s = torch.from_numpy(q)
    dist.all_reduce(s, op=dist.ReduceOp.SUM)              # the 8-bit codes travel, summed in int32
    out = (s.numpy().astype(np.float32) * np.repeat(scale, block)[:n]).astype(np.float32)
    ref = oracle.q8_reduce(parts, block)
    assert np.array_equal(s.numpy(), ref["sums"])
    assert np.array_equal(scale, ref["scales"])
    assert np.array_equal(out, ref["out_f32"])


class _OracleOps:
    """The rank-local arithmetic of tp.q8_all_reduce from the oracle (CPU), so the exchange's
    control flow -- which collective, on which buffers, in which order -- runs on gloo ranks."""

    @staticmethod
    def block_absmax(x):
        import oracle
        return torch.from_numpy(oracle.q8_block_absmax(x))

    @staticmethod
    def quantize_shared(x, amax):
        import oracle
        r = oracle.q8_quantize_shared(x, amax.numpy())
        return torch.from_numpy(r["codes"]).reshape(x.shape), torch.from_numpy(r["scales"])

    @staticmethod
    def sum_dequant(codes, scales, out_dtype):
        import oracle
        r = oracle.q8_sum_dequant([c.numpy() for c in codes], scales.numpy())
        if out_dtype == torch.bfloat16:
            out = torch.from_numpy(r["out_bf16"].view(np.int16)).view(torch.bfloat16)
        else:
            out = torch.from_numpy(r["out_f32"])
        return out, torch.from_numpy(r["sums"])


def _tp_q8_all_reduce(rank, world, out_dtype):
    import oracle
    from selective_state_space_prefill_gb300 import tp
    from selective_state_space_prefill_gb300.inputs import make_partials
    parts = make_partials(world, (3, 1, 1000), dtype=torch.bfloat16, seed=33)
    out, sums, scales = tp.q8_all_reduce(parts[rank], out_dtype=out_dtype, ops=_OracleOps)
    ref = oracle.q8_reduce([p.reshape(-1) for p in parts])
    assert out.shape == parts[rank].shape and out.dtype == out_dtype
    assert np.array_equal(sums.numpy(), ref["sums"])
    assert np.array_equal(scales.numpy(), ref["scales"])
    got = out.reshape(-1)
    if out_dtype == torch.bfloat16:
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), ref["out_bf16"])
    else:
        assert np.array_equal(got.numpy(), ref["out_f32"])
    # every rank ends with the same result
    mine = got.float().clone()
    total = mine.clone()
    dist.all_reduce(total)
    assert torch.equal(total, mine * world)


def _timing(rank, world):
    import bench
    t = bench.max_over_ranks(0.5 + rank)                  # rank r took 0.5 + r seconds
    assert t == 0.5 + (world - 1)
    assert bench.whole_job_rate(100.0, world, t) == world * 100.0 / t


@pytest.mark.parametrize("world", [2, 4])
def test_channel_shards_gather_to_unsplit(world):
    _run(world, _shard_prefill)


@pytest.mark.parametrize("world", [2, 4])
def test_quantized_allreduce_across_ranks_equals_local_q8(world):
    _run(world, _quantized_allreduce)


@pytest.mark.parametrize("world,out_dtype", [(2, torch.float32), (4, torch.bfloat16)])
def test_tp_q8_all_reduce_control_flow(world, out_dtype):
    """tp.q8_all_reduce on gloo ranks: MAX all-reduce of block maxima, shared-scale codes,
    all-gather of the int8 codes, local sum -- equal to the local reduction on every rank."""
    _run(world, _tp_q8_all_reduce, out_dtype)


def test_bench_cross_rank_timing():
    _run(2, _timing)
