"""Comparator cache policies through the engine (C ABI) vs the oracle's simulators: the
per-layer LRU and a static resident set give per-call hit / miss / bypass / eviction counts
and full cache snapshots bit-exact against oracle.policies, with outputs within tolerance;
ft_cache_pin places keys as the simulator does."""
import numpy as np
import pytest

import workloads as W
from workloads.host import HostPool
from oracle import lru, policies
from ref import TOL, OracleExperts, Runner, bf16_dev_to_f64, out_err, oracle_call

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


def _cfg():
    # 4 layers of the 284B layer's routing (256 experts, top-6), small expert shapes
    return W.config("decode_mxfp4", layers=4, hidden=64, inter=64, steps=24)


def _make(ft, cfg, pool, capacity, policy):
    c = ft.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, cfg.t_max,
                       cfg.wfmt, capacity, policy=policy)
    return ft.MoECache(c, pool.ptrs, None)


def test_layer_lru_matches_simulator(ft):
    cfg = _cfg()
    pool = HostPool(cfg, images=7)
    C = W.cache_capacity(cfg)                       # 20 % of 1024 keys: 204 slots, 51 per layer
    cache = _make(ft, cfg, pool, C, ft.POLICY_LAYER_LRU)
    run = Runner(cache, cfg, C, sim=policies.LayerLRU(C, cfg.experts, cfg.layers))
    experts = OracleExperts(pool, max_cached=7)
    worst = 0.0
    for s, step in enumerate(W.decode_trace(cfg)):
        for d in step:
            out, idx, _ = run.call(d["layer"], d["x"], d["logits"])
            if s % 6 == 0 and d["layer"] == 2:
                ref, ref_idx, _ = oracle_call(experts, d["layer"], d["x"], d["logits"], cfg.top_k)
                assert np.array_equal(idx, ref_idx)
                worst = max(worst, out_err(bf16_dev_to_f64(out), ref))
        if s % 4 == 0:
            run.check_state()
    run.check_state()
    assert worst <= TOL["mxfp4"], worst
    assert cache.resize_status(C // 2) != 0          # resize: global LRU only
    cache.close()


def test_static_set_matches_simulator(ft):
    cfg = _cfg()
    pool = HostPool(cfg, images=7)
    C = W.cache_capacity(cfg)
    steps = list(W.decode_trace(cfg))
    # the hot set: the C most selected keys over the first 8 steps (ties to the lower key)
    count = np.zeros(cfg.keys, dtype=np.int64)
    for step in steps[:8]:
        for d in step:
            for e in np.unique(d["picks"]):
                count[d["layer"] * cfg.experts + int(e)] += 1
    hot = [int(k) for k in np.lexsort((np.arange(cfg.keys), -count))[:C]]
    cache = _make(ft, cfg, pool, C, ft.POLICY_STATIC)
    cache.pin(hot)
    sim = policies.static_set(C, cfg.experts, hot)
    run = Runner(cache, cfg, C, sim=sim)
    run.check_state()
    before = cache.snapshot()[0].copy()
    experts = OracleExperts(pool, max_cached=7)
    worst = 0.0
    for s, step in enumerate(steps[8:]):
        for d in step:
            out, idx, _ = run.call(d["layer"], d["x"], d["logits"])
            if s % 6 == 0 and d["layer"] == 1:
                ref, _, _ = oracle_call(experts, d["layer"], d["x"], d["logits"], cfg.top_k)
                worst = max(worst, out_err(bf16_dev_to_f64(out), ref))
    run.check_state()
    assert np.array_equal(cache.snapshot()[0], before)   # the resident set never changes
    st = cache.stats()
    assert st["evictions"] == 0 and st["bypassed"] == st["misses"] and st["fill_bytes"] == 0
    assert worst <= TOL["mxfp4"], worst
    cache.close()


def test_pin_prewarms_the_global_lru(ft):
    cfg = _cfg()
    pool = HostPool(cfg, images=7)
    C = 40
    cache = _make(ft, cfg, pool, C, ft.POLICY_GLOBAL_LRU)
    keys = [5, 300, 7, 5, 1000]                      # 5 pinned twice: moves to the MRU end
    cache.pin(keys)
    sim = lru.LRUCache(C, cfg.experts)
    sim.pin(keys)
    slots, order = cache.snapshot()
    want_slots, want_order = sim.snapshot(cfg.keys)
    assert slots.tolist() == want_slots and order.tolist() == want_order
    assert cache.stats()["resident"] == 4 and cache.stats()["fill_bytes"] == 0
    run = Runner(cache, cfg, C, sim=sim)
    for step in list(W.decode_trace(cfg))[:3]:
        for d in step:
            run.call(d["layer"], d["x"], d["logits"])
    run.check_state()
    cache.close()
