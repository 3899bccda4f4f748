"""Medusa draft-and-verify decode step on one GB300 GPU (sm_103a CUDA kernels behind a C ABI).

The compute path is libmedusa.so (include/medusa.h); this package only builds it and
marshals arguments to it through ctypes.
"""
from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    Plan, MedusaError, lib, step, heads, tree_build, layer_qkv, tree_attention, layer_out,
    verify_logits, verify, kv_compact, tree_cartesian, tree_greedy, weights_struct, kv_struct,
    accept_struct, outputs_struct,
)
