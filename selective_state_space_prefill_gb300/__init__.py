"""GB300 (sm_103a) selective-SSM mixer: prefill, cached-state decode, 8-bit partial reduction.

The compute path is the C-ABI library ``libssm.so`` built from ``csrc/`` by
``selective_state_space_prefill_gb300.build``; ``binding`` marshals torch
tensors into it.  There is no CPU fallback: every call fails loudly when the
library or a CUDA device is missing.
"""
from .inputs import make_mixer_inputs  # noqa: F401
