"""fp64 CPU oracle for the selective-SSM mixer, its SSD (Mamba-2-style) variant and the
output-projection partial (test infrastructure only).

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA path: the arithmetic
lives in ``ssm_oracle.c`` (plain C, double precision, sequential per channel)
and this module only marshals arrays into it.

Pinned against closed forms, invariants and brute force in
``tests/test_oracle_pins.py``; every oracle function there has at least one
pin that a dropped term, a wrong sign or index, or a swapped operand fails.
"""
from .oracle import (  # noqa: F401
    build,
    decode_step,
    lib_path,
    out_proj,
    prefill,
    q8_block_absmax,
    q8_quantize_shared,
    q8_reduce,
    q8_sum_dequant,
    scan_chunked,
    scan_sequential,
    ssd_prefill,
)
