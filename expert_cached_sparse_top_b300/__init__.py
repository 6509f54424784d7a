"""expert_cached_sparse_top_b300: the routed MoE layer forward with a GPU-resident global-LRU
expert cache, as a C-ABI CUDA library (libftmoe.so, sm_103a) plus a ctypes binding.

    from expert_cached_sparse_top_b300 import ftmoe
    cache = ftmoe.MoECache(cfg, blob_ptrs, router_w)
    cache.forward(layer, x, T, out, logits=None)
"""
from . import ftmoe  # noqa: F401
