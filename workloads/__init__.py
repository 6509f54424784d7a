"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random bytes and numbers and packs them into the library's input
layouts (bf16 bit patterns, FP4 code bytes, per-expert blobs, router logits). It holds none
of the method's arithmetic: no routing, no cache policy, no FFN, no dequantisation. Both the
CUDA path and the oracle consume exactly the arrays produced here.
"""
from .gen import (  # noqa: F401
    CONFIGS, WorkloadConfig, config, expert_pool, router_weights, decode_trace,
    trace_step, tiny_inputs, prefill_inputs, predicted_picks, chained_inputs, pack_blob_bf16, pack_blob_fp4,
    f32_to_bf16_bits,
    cache_capacity, blob_layout,
)
