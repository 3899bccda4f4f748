"""Seeded synthetic inputs for the Medusa decode step (shared by the oracle and the CUDA path)."""
from .inputs import (  # noqa: F401
    Workload, WORKLOADS, workload, vicuna33b, weights, hidden, kv_prefix, kv_cache, kv_cache_device,
    page_table, score_table, planted_weights, head_init_weights, uniforms, layer_weights,
)
