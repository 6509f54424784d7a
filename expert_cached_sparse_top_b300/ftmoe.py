"""ctypes binding of libftmoe.so (include/ftmoe.h). Argument marshalling only: every step of
the MoE layer runs in the library's CUDA kernels; nothing here computes.

Device buffers are passed as torch CUDA tensors (or raw integer device pointers), streams as
torch.cuda.Stream (or a raw cudaStream_t integer). If the shared library is missing this
module raises on import: there is no fallback path.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libftmoe.so")

FT_OK, FT_ERR_INVALID, FT_ERR_OOM, FT_ERR_CUDA, FT_ERR_TIMEOUT, FT_ERR_STATE = range(6)
FT_W_BF16, FT_W_MXFP4, FT_W_NVFP4 = 0, 1, 2
WFMT = {"bf16": FT_W_BF16, "mxfp4": FT_W_MXFP4, "nvfp4": FT_W_NVFP4}

# Every symbol include/ftmoe.h declares (checked by the CPU test suite).
EXPORTS = (
    "ft_status_str", "ft_expert_blob_bytes", "ft_moe_create", "ft_moe_forward",
    "ft_cache_resize", "ft_cache_stats", "ft_cache_snapshot", "ft_moe_set_timing",
    "ft_moe_timing", "ft_moe_last_error", "ft_moe_destroy", "ft_router_logits",
    "ft_topk_softmax", "ft_expert_ffn_noalloc", "ft_moe_prefill", "ft_cache_pin",
    "ft_cache_prefetch",
)


class FtMoeConfig(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("experts", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("wfmt", ctypes.c_int32), ("device", ctypes.c_int32),
                ("cache_slots", ctypes.c_int64), ("flags", ctypes.c_int32),
                ("max_prefill_tokens", ctypes.c_int32)]


class FtCacheStats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("misses", ctypes.c_uint64), ("bypassed", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("fill_bytes", ctypes.c_uint64),
                ("stage_bytes", ctypes.c_uint64), ("fill_ns", ctypes.c_uint64),
                ("capacity", ctypes.c_int64), ("resident", ctypes.c_int64),
                ("prefetches", ctypes.c_uint64), ("prefetch_fills", ctypes.c_uint64),
                ("prefetch_evictions", ctypes.c_uint64), ("prefetch_skipped", ctypes.c_uint64),
                ("prefetch_bytes", ctypes.c_uint64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class FtTiming(ctypes.Structure):
    _fields_ = [("route_ms", ctypes.c_double), ("ffn_hit_ms", ctypes.c_double),
                ("fill_ms", ctypes.c_double), ("ffn_miss_ms", ctypes.c_double),
                ("combine_ms", ctypes.c_double), ("total_ms", ctypes.c_double),
                ("forwards", ctypes.c_uint64), ("ffn_launches", ctypes.c_uint64),
                ("ffn_weight_bytes", ctypes.c_uint64), ("kernel_launches", ctypes.c_uint64),
                ("prefill_calls", ctypes.c_uint64), ("prefill_fill_ms", ctypes.c_double),
                ("prefill_compute_ms", ctypes.c_double), ("prefill_ffn_ms", ctypes.c_double),
                ("prefill_flops", ctypes.c_double), ("prefill_fill_bytes", ctypes.c_uint64),
                ("prefetch_fill_ms", ctypes.c_double), ("prefetch_wait_ms", ctypes.c_double),
                ("fill_lead_ms", ctypes.c_double), ("fill_lead_calls", ctypes.c_uint64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None


def lib():
    """Load libftmoe.so (built in-tree by expert_cached_sparse_top_b300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libftmoe.so is not built (run python -m expert_cached_sparse_top_b300.build)")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, I64, VP = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    sig = {
        "ft_status_str": (ctypes.c_char_p, [I32]),
        "ft_expert_blob_bytes": (ctypes.c_size_t, [ctypes.POINTER(FtMoeConfig)]),
        "ft_moe_create": (I32, [ctypes.POINTER(FtMoeConfig), ctypes.POINTER(VP), P,
                                ctypes.POINTER(VP)]),
        "ft_moe_forward": (I32, [VP, I32, P, I32, P, P, P, P, P]),
        "ft_cache_resize": (I32, [VP, I64]),
        "ft_cache_stats": (I32, [VP, ctypes.POINTER(FtCacheStats)]),
        "ft_cache_snapshot": (I32, [VP, P, P]),
        "ft_moe_set_timing": (I32, [VP, I32]),
        "ft_moe_timing": (I32, [VP, ctypes.POINTER(FtTiming), I32]),
        "ft_moe_last_error": (ctypes.c_char_p, [VP]),
        "ft_moe_destroy": (None, [VP]),
        "ft_router_logits": (I32, [P, I32, I32, P, I32, P, P]),
        "ft_topk_softmax": (I32, [P, I32, I32, I32, P, P, P]),
        "ft_expert_ffn_noalloc": (I32, [P, I32, I32, I32, P, I32, P, P]),
        "ft_moe_prefill": (I32, [VP, I32, P, I32, P, P, P]),
        "ft_cache_pin": (I32, [VP, P, I32]),
        "ft_cache_prefetch": (I32, [VP, I32, P, I32, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


class FtError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__("%s: %s" % (lib().ft_status_str(status).decode(), message))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


POLICY_GLOBAL_LRU, POLICY_LAYER_LRU, POLICY_STATIC = 0, 1, 2
FLAG_FUSED_DECODE = 0x100


def make_config(layers, experts, hidden, inter, top_k, max_tokens, wfmt, cache_slots, device=0,
                max_prefill_tokens=0, policy=POLICY_GLOBAL_LRU, fused_decode=False):
    """An ft_moe_config. policy: POLICY_*; fused_decode: every forward is one cooperative
    launch (FT_FLAG_FUSED_DECODE) and does not wait for the device; its errors surface on the
    next call or safe point (stats, snapshot, resize, pin, timing)."""
    flags = int(policy) | (FLAG_FUSED_DECODE if fused_decode else 0)
    return FtMoeConfig(layers, experts, hidden, inter, top_k, max_tokens,
                       WFMT.get(wfmt, wfmt), device, cache_slots, flags, max_prefill_tokens)


def blob_bytes(cfg):
    return int(lib().ft_expert_blob_bytes(ctypes.byref(cfg)))


def check(status, handle=None):
    if status != FT_OK:
        msg = lib().ft_moe_last_error(handle)
        raise FtError(status, (msg or b"").decode())


class MoECache:
    """One libftmoe handle: the MoE layer forward with a GPU expert cache."""

    def __init__(self, cfg, blob_ptrs, router_w=None):
        """cfg: FtMoeConfig. blob_ptrs: layers*experts host addresses (ints) of the expert
        blobs (caller-owned, must outlive this object). router_w: host fp32 numpy array
        [layers][experts][hidden] or None."""
        self.cfg = cfg
        n = cfg.layers * cfg.experts
        if len(blob_ptrs) != n:
            raise ValueError("need %d blob pointers" % n)
        self._ptrs = (ctypes.c_void_p * n)(*[int(p) for p in blob_ptrs])
        self._router = router_w
        rp = None
        if router_w is not None:
            import numpy as np
            self._router = np.ascontiguousarray(router_w, dtype=np.float32)
            rp = self._router.ctypes.data
        h = ctypes.c_void_p()
        st = lib().ft_moe_create(ctypes.byref(cfg), self._ptrs, rp, ctypes.byref(h))
        check(st, None)
        self.h = h

    def forward(self, layer, x, T, out, logits=None, topk_idx=None, topk_w=None, stream=None):
        st = lib().ft_moe_forward(self.h, int(layer), _ptr(x), int(T), _ptr(logits), _ptr(out),
                                  _ptr(topk_idx), _ptr(topk_w), _stream(stream))
        check(st, self.h)

    def forward_status(self, layer, x, T, out, logits=None, topk_idx=None, topk_w=None,
                       stream=None):
        """Same call, returning the raw status instead of raising."""
        return lib().ft_moe_forward(self.h, int(layer), _ptr(x), int(T), _ptr(logits),
                                    _ptr(out), _ptr(topk_idx), _ptr(topk_w), _stream(stream))

    def prefill(self, layer, x, T, out, logits=None, stream=None):
        check(lib().ft_moe_prefill(self.h, int(layer), _ptr(x), int(T), _ptr(logits), _ptr(out),
                                   _stream(stream)), self.h)

    def prefill_status(self, layer, x, T, out, logits=None, stream=None):
        return lib().ft_moe_prefill(self.h, int(layer), _ptr(x), int(T), _ptr(logits), _ptr(out),
                                    _stream(stream))

    def prefetch(self, layer, experts, n=None, stream=None):
        """Layer-ahead prefetch of `layer`'s predicted experts (dev int32 tensor); `stream` is
        the stream they are produced on."""
        n = int(experts.numel()) if n is None else int(n)
        check(lib().ft_cache_prefetch(self.h, int(layer), _ptr(experts), n, _stream(stream)), self.h)

    def pin(self, keys):
        """Place keys (layer * experts + expert) into the cache, first key least recent."""
        import numpy as np
        k = np.ascontiguousarray(keys, dtype=np.int32)
        check(lib().ft_cache_pin(self.h, k.ctypes.data if k.size else None, int(k.size)), self.h)

    def resize(self, new_slots):
        check(lib().ft_cache_resize(self.h, int(new_slots)), self.h)

    def resize_status(self, new_slots):
        return lib().ft_cache_resize(self.h, int(new_slots))

    def stats(self):
        s = FtCacheStats()
        check(lib().ft_cache_stats(self.h, ctypes.byref(s)), self.h)
        return s.as_dict()

    def snapshot(self):
        import numpy as np
        nkeys = self.cfg.layers * self.cfg.experts
        slot_of_key = np.empty(nkeys, dtype=np.int32)
        cap = self.stats()["capacity"]
        lru = np.empty(max(cap, 1), dtype=np.int32)
        check(lib().ft_cache_snapshot(self.h, slot_of_key.ctypes.data, lru.ctypes.data), self.h)
        return slot_of_key, lru[:cap]

    def set_timing(self, enable):
        check(lib().ft_moe_set_timing(self.h, 1 if enable else 0), self.h)

    def timing(self, reset=False):
        t = FtTiming()
        check(lib().ft_moe_timing(self.h, ctypes.byref(t), 1 if reset else 0), self.h)
        return t.as_dict()

    def last_error(self):
        return (lib().ft_moe_last_error(self.h) or b"").decode()

    def close(self):
        if getattr(self, "h", None):
            lib().ft_moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def router_logits(x, T, H, wr, E, logits, stream=None):
    check(lib().ft_router_logits(_ptr(x), int(T), int(H), _ptr(wr), int(E), _ptr(logits),
                                 _stream(stream)))


def topk_softmax(logits, T, E, k, idx, w, stream=None):
    check(lib().ft_topk_softmax(_ptr(logits), int(T), int(E), int(k), _ptr(idx), _ptr(w),
                                _stream(stream)))


def expert_ffn_noalloc(blob, wfmt, hidden, inter, x, T, y, stream=None):
    """Single-expert SwiGLU FFN with no device allocation (see include/ftmoe.h)."""
    check(lib().ft_expert_ffn_noalloc(_ptr(blob), int(WFMT.get(wfmt, wfmt)), int(hidden),
                                      int(inter), _ptr(x), int(T), _ptr(y), _stream(stream)))
