"""The 8-bit quantized all-reduce of tensor-parallel partials across ranks.

"Scaling State-Space Models on Multiple GPUs with Tensor Parallelism", Methodology 4: the
ranks' partial outputs (one per channel slice of the mixer, after the output projection)
are quantized to 8 bits, summed across the ranks and dequantized.  With one scale per
block of 128 elements shared by every rank, the exchange is:

  1. each rank's block maxima of |partial|          (libssm q8_block_absmax, or the maxima
                                                     ssm_out_proj_partial emits)
  2. MAX all-reduce of the maxima                   (4 bytes per 128 elements)
  3. each rank's int8 codes with the shared scale   (libssm q8_quantize_shared)
  4. all-gather of the codes                        (1 byte per element and rank)
  5. every rank sums the P code buffers in int32 and dequantizes (libssm q8_sum_dequant)

so every rank ends with the same result, equal bit for bit to q8_reduce_partials over the P
partials held in one memory.  The collectives are torch.distributed's (NCCL between GPUs);
the arithmetic is libssm's.  This module orders the steps and moves the buffers.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

BLOCK = 128


class Kernels:
    """The rank-local arithmetic: libssm's kernels on CUDA tensors."""

    @staticmethod
    def block_absmax(x):
        from . import binding
        return binding.q8_block_absmax(x)

    @staticmethod
    def quantize_shared(x, amax):
        from . import binding
        return binding.q8_quantize_shared(x, amax)

    @staticmethod
    def sum_dequant(codes, scales, out_dtype):
        from . import binding
        return binding.q8_sum_dequant(codes, scales, out_dtype=out_dtype)


def q8_all_reduce(partial, group=None, out_dtype=None, block_amax=None, ops=Kernels):
    """Sum ``partial`` (contiguous, bf16 or fp32) over the ranks of ``group`` through int8 codes.

    ``block_amax`` may carry this rank's block maxima when the producer emitted them
    (ssm_out_proj_partial); ``ops`` supplies the rank-local arithmetic.
    Returns (out shaped like ``partial`` in ``out_dtype``, int32 sums [n], shared scales [nblk]).
    """
    if not partial.is_contiguous():
        raise ValueError("partial must be contiguous")
    world = dist.get_world_size(group)
    amax = (block_amax if block_amax is not None else ops.block_absmax(partial)).clone()
    dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)          # the shared maxima
    codes, scales = ops.quantize_shared(partial, amax)
    flat = codes.reshape(-1)
    gathered = [torch.empty_like(flat) for _ in range(world)]
    dist.all_gather(gathered, flat, group=group)                       # 1 byte per element
    out, sums = ops.sum_dequant(gathered, scales, out_dtype or partial.dtype)
    return out.reshape(partial.shape), sums, scales
