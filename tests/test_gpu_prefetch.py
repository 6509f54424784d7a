"""Layer-ahead prefetch (ft_cache_prefetch) on chained layers, through the C ABI, against the
oracle: a 4-layer chained decode (each layer's input is the previous layer's input plus its
output, rounded to bf16), with a prefetch of the next layer's predicted experts after every
forward call. Per-call and per-prefetch cache counts and the full cache state are checked
bit-exactly against the oracle's LRU simulator (which replays the same prefetches with the
same protection rule), outputs against the oracle's own chain within the BF16 tolerance, and
bit-for-bit against the same chain without prefetches (outputs never depend on cache state)."""
import numpy as np
import pytest

import workloads as W
from oracle import formats, lru, moe
from workloads.host import HostPool
from ref import TOL, OracleExperts, bf16_dev_to_f64, out_err, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ft():
    import torch
    from expert_cached_sparse_top_b300 import build
    build.build()
    from expert_cached_sparse_top_b300 import ftmoe
    ftmoe.lib()
    torch.cuda.init()
    return ftmoe


def _make(ft, cfg, pool, C, **kw):
    c = ft.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, cfg.t_max,
                       cfg.wfmt, C, **kw)
    return ft.MoECache(c, pool.ptrs, None)


def _chain(ft, cfg, pool, C, steps, prefetch, accuracy=0.75):
    """Run the chained trace; returns per-call outputs (bf16 tensors on the host) and checks
    cache counts against the simulator when `prefetch` is on."""
    import torch
    cache = _make(ft, cfg, pool, C)
    sim = lru.LRUCache(C, cfg.experts)
    protect = 0
    prev = cache.stats()
    outs = []
    for step in W.decode_trace(cfg, steps=steps):
        x = to_dev_bf16(step[0]["x"])
        T = step[0]["T"]
        for li, d in enumerate(step):
            out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
            idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
            cache.forward(li, x, T, out, logits=to_dev(d["logits"]), topk_idx=idx)
            torch.cuda.synchronize()
            r = sim.call(li, idx.cpu().numpy().reshape(-1))
            protect = len(r.hits) + len(r.misses)
            st = cache.stats()
            got = {k: st[k] - prev[k] for k in ("hits", "misses", "bypassed", "evictions")}
            assert got == {"hits": len(r.hits), "misses": len(r.misses) + len(r.bypassed),
                           "bypassed": len(r.bypassed), "evictions": len(r.evicted)}, (step[0]["step"], li)
            prev = st
            if prefetch and li + 1 < cfg.layers:
                nxt = step[li + 1]
                pred = W.predicted_picks(cfg, nxt["step"], li + 1, nxt["picks"], accuracy)
                cache.prefetch(li + 1, to_dev(pred))
                pr = sim.prefetch(li + 1, pred, protect=protect)
                protect += len(pr.inserted)
                st = cache.stats()
                got = {k: st[k] - prev[k] for k in ("prefetch_fills", "prefetch_evictions",
                                                     "prefetch_skipped", "hits", "misses")}
                assert got == {"prefetch_fills": len(pr.inserted), "prefetch_evictions": len(pr.evicted),
                               "prefetch_skipped": len(pr.skipped), "hits": 0, "misses": 0}, \
                    (step[0]["step"], li)
                prev = st
            outs.append(out.cpu())
            x = (x.float() + out.float()).to(torch.bfloat16)       # the chain's residual add
        if step[0]["step"] % 4 == 3:
            slot_of_key, lru_keys = cache.snapshot()
            want_slots, want_lru = sim.snapshot(cfg.keys)
            assert slot_of_key.tolist() == want_slots and lru_keys.tolist() == want_lru
    st = cache.stats()
    cache.close()
    return outs, st, sim


def test_prefetch_chained_trace_matches_oracle(ft):
    cfg = W.config("decode_chained", layers=4, hidden=256, inter=128)
    pool = HostPool(cfg)
    C = W.cache_capacity(cfg)
    steps = 24
    outs, st, sim = _chain(ft, cfg, pool, C, steps, prefetch=True)
    assert st["prefetch_fills"] > 0 and st["prefetch_evictions"] > 0 and st["prefetches"] == steps * 3
    assert st["prefetch_bytes"] == st["prefetch_fills"] * pool.blob_bytes
    # the oracle's own chain: x_{l+1} = bf16(x_l + bf16(out_l)), routing from the same logits
    experts = OracleExperts(pool, max_cached=cfg.keys)
    worst, i = 0.0, 0
    for step in W.decode_trace(cfg, steps=steps):
        x = formats.bf16_to_f64(step[0]["x"])
        for li, d in enumerate(step):
            logits = np.asarray(d["logits"], dtype=np.float64)
            idx = moe.topk(logits, cfg.top_k)
            w = moe.gate_weights(logits, idx)
            ref, _ = moe.layer_forward(x, idx, w, lambda e, L=li: experts(L * cfg.experts + e))
            worst = max(worst, out_err(outs[i].float().numpy(), ref))
            x = moe.bf16_round(x + moe.bf16_round(ref))
            i += 1
    assert worst <= TOL["bf16"], worst
    # the same chain without prefetches: bit-identical outputs, more misses
    outs2, st2, _ = _chain(ft, cfg, pool, C, steps, prefetch=False)
    import torch
    assert all(torch.equal(a, b) for a, b in zip(outs, outs2))
    assert st2["prefetches"] == 0 and st2["misses"] > st["misses"]


def test_prefetch_arguments(ft):
    import torch
    cfg = W.config("decode_chained", layers=2, hidden=256, inter=128)
    pool = HostPool(cfg)
    e = torch.zeros(4, dtype=torch.int32, device="cuda")
    cache = _make(ft, cfg, pool, 8)
    L = ft.lib()
    assert L.ft_cache_prefetch(cache.h, 2, e.data_ptr(), 4, None) == ft.FT_ERR_INVALID   # layer
    assert L.ft_cache_prefetch(cache.h, 0, e.data_ptr(), 10 ** 6, None) == ft.FT_ERR_INVALID
    assert L.ft_cache_prefetch(cache.h, 0, None, 4, None) == ft.FT_ERR_INVALID
    assert L.ft_cache_prefetch(cache.h, 0, e.data_ptr(), 0, None) == ft.FT_OK
    cache.prefetch(1, torch.tensor([3, 3, 5], dtype=torch.int32, device="cuda"))
    st = cache.stats()
    assert st["prefetch_fills"] == 2 and st["resident"] == 2 and st["hits"] == 0
    cache.close()
    for kw in ({"policy": ft.POLICY_LAYER_LRU}, {"fused_decode": True}):
        c2 = _make(ft, cfg, pool, 8, **kw)
        assert L.ft_cache_prefetch(c2.h, 0, e.data_ptr(), 4, None) == ft.FT_ERR_INVALID
        c2.close()
