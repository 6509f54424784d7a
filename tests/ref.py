"""Test helpers: oracle-side expectations and device marshalling for the parity tests."""
from collections import OrderedDict

import numpy as np

from oracle import formats, lru, moe

TOL = {"bf16": 1e-2, "mxfp4": 2e-2, "nvfp4": 2e-2}   # normwise relative error on out


class OracleExperts:
    """key -> decoded fp64 (w1, w3, w2) from the same host blobs the GPU reads (memoised by
    physical image)."""

    def __init__(self, pool, max_cached=48):
        self.pool = pool
        self.cfg = pool.cfg
        self.memo = OrderedDict()
        self.max_cached = max_cached

    def __call__(self, key):
        img = self.pool.image_of(key)
        if img in self.memo:
            self.memo.move_to_end(img)
            return self.memo[img]
        w = formats.decode_blob(self.pool.blob(key), self.cfg.fmt, self.cfg.hidden, self.cfg.inter)
        self.memo[img] = w
        if len(self.memo) > self.max_cached:
            self.memo.popitem(last=False)
        return w


def oracle_call(experts, layer, x_bits, logits, k, tokens=None, ffn=None):
    """Expected (out, idx, w) for one forward call; ``tokens`` restricts to a sample; ``ffn``
    replaces the plain expert FFN (moe.expert_ffn)."""
    E = experts.cfg.experts
    x = formats.bf16_to_f64(x_bits)
    l = np.asarray(logits, dtype=np.float64)
    if tokens is not None:
        x, l = x[tokens], l[tokens]
    idx = moe.topk(l, k)
    w = moe.gate_weights(l, idx)
    out, _ = moe.layer_forward(x, idx, w, lambda e: experts(layer * E + e), ffn=ffn)
    return out, idx, w


def normwise_err(got, ref):
    """Normwise relative error of a whole call: ||got - ref||_F / ||ref||_F."""
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(np.asarray(got, dtype=np.float64) - ref) / max(den, 1e-30))


def token_err(got, ref):
    """Worst per-token normwise relative error: max over rows t of ||got_t - ref_t|| / ||ref_t||.
    A few wrong tokens in a large call stay under a whole-call bound; they do not stay under
    this one."""
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    ref2 = ref.reshape(ref.shape[0], -1)
    num = np.linalg.norm(got.reshape(ref2.shape) - ref2, axis=1)
    den = np.maximum(np.linalg.norm(ref2, axis=1), 1e-30)
    return float((num / den).max())


def out_err(got, ref):
    """The error the parity tests bound by TOL: the larger of the whole-call normwise error and
    the worst per-token normwise error (both at the same tolerance)."""
    return max(normwise_err(got, ref), token_err(got, ref))


def to_dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev_to_f64(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64)


class Runner:
    """Drives one MoECache and a mirror oracle LRU over calls, checking per-call cache
    counts bit-exactly."""

    def __init__(self, cache, cfg, capacity, sim=None):
        self.cache = cache
        self.cfg = cfg
        self.sim = sim if sim is not None else lru.LRUCache(capacity, cfg.experts)
        self.prev = cache.stats()

    def call(self, layer, x_bits, logits=None, T=None, check=True):
        import torch
        cfg = self.cfg
        T = x_bits.shape[0] if T is None else T
        x = to_dev_bf16(x_bits)
        out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
        idx = torch.full((max(T, 1), cfg.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((max(T, 1), cfg.top_k), dtype=torch.float32, device="cuda")
        lg = to_dev(np.asarray(logits, dtype=np.float32)) if logits is not None else None
        self.cache.forward(layer, x, T, out, logits=lg, topk_idx=idx, topk_w=w)
        torch.cuda.synchronize()
        idx_h = idx.cpu().numpy()[:T]
        if check:
            r = self.sim.call(layer, idx_h.reshape(-1))
            st = self.cache.stats()
            d = {k2: st[k2] - self.prev[k2] for k2 in ("hits", "misses", "bypassed", "evictions")}
            assert d == {"hits": len(r.hits), "misses": len(r.misses) + len(r.bypassed),
                         "bypassed": len(r.bypassed), "evictions": len(r.evicted)}, (d, layer)
            self.prev = st
        return out, idx_h, w.cpu().numpy()[:T]

    def resize(self, new_cap):
        self.cache.resize(new_cap)
        self.sim.resize(new_cap)
        self.prev = self.cache.stats()

    def check_state(self):
        slot_of_key, lru_keys = self.cache.snapshot()
        want_slots, want_lru = self.sim.snapshot(self.cfg.keys)
        assert slot_of_key.tolist() == want_slots
        assert lru_keys.tolist() == want_lru
