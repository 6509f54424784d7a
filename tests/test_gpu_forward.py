"""Full MoE-layer forward through the cache (C ABI) vs the oracle: routing and cache state
bit-exact, outputs within the normwise tolerance, output independent of cache state."""
import os

import numpy as np
import pytest

import workloads as W
from workloads.host import HostPool
from ref import (TOL, OracleExperts, Runner, bf16_dev_to_f64, out_err, oracle_call,
                 to_dev_bf16)

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


def _make(ft, cfg, pool, capacity, max_tokens=None, router=None):
    mt = max_tokens or max(cfg.t_max, cfg.tokens, 1)
    c = ft.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, mt,
                       cfg.wfmt, capacity)
    return ft.MoECache(c, pool.ptrs, router)


@pytest.fixture(scope="module")
def bf16_pool():
    return HostPool(W.config("decode_bf16"))


# ---------------------------------------------------------------------------------------
def test_tiny_layer_router_in_the_loop(ft):
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    router = W.router_weights(cfg)
    cache = _make(ft, cfg, pool, capacity=cfg.experts, router=router)
    run = Runner(cache, cfg, cfg.experts)
    x = W.tiny_inputs(cfg)
    from oracle import formats, moe
    ref_logits = moe.router_logits(formats.bf16_to_f64(x), router[0])
    srt = np.sort(ref_logits, axis=1)[:, ::-1]
    assert np.all(srt[:, cfg.top_k - 1] - srt[:, cfg.top_k] > 1e-4)   # no near-ties
    experts = OracleExperts(pool)
    ref_out, ref_idx, ref_w = oracle_call(experts, 0, x, ref_logits, cfg.top_k)
    outs = []
    for _ in range(3):   # cold, then warm: every expert resident
        out, idx, w = run.call(0, x)
        assert np.array_equal(idx, ref_idx)
        assert np.max(np.abs(w - ref_w)) <= 2e-6
        outs.append(bf16_dev_to_f64(out))
        assert out_err(outs[-1], ref_out) <= TOL["bf16"]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    st = cache.stats()
    U = len(np.unique(ref_idx))
    assert st["misses"] == U and st["hits"] == 2 * U and st["resident"] == U
    run.check_state()
    cache.close()


def test_decode_bf16_trace_parity(ft, bf16_pool):
    cfg = W.config("decode_bf16")
    C = W.cache_capacity(cfg)
    cache = _make(ft, cfg, bf16_pool, C)
    run = Runner(cache, cfg, C)
    experts = OracleExperts(bf16_pool, max_cached=64)
    tr = W.decode_trace(cfg, steps=10)
    worst = 0.0
    for s, step in enumerate(tr):
        d = step[0]
        out, idx, w = run.call(0, d["x"], d["logits"])
        ref_out, ref_idx, ref_w = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
        assert np.array_equal(idx, ref_idx)
        worst = max(worst, out_err(bf16_dev_to_f64(out), ref_out))
        if s % 3 == 0:
            run.check_state()
    assert worst <= TOL["bf16"], worst
    st = cache.stats()
    assert st["bypassed"] > 0 or st["misses"] > 0
    cache.close()


@pytest.mark.parametrize("path", ["tcgen05", "tcgen05_two_launches", "simt"])
@pytest.mark.parametrize("T", [1, 16])
def test_decode_bf16_fixed_T(ft, bf16_pool, T, path, monkeypatch):
    """Both BF16 expert-FFN paths (tcgen05 grouped GEMM, CUDA-core GEMV) against the oracle."""
    if path == "simt":
        monkeypatch.setenv("FTMOE_FFN", "simt")
    if path == "tcgen05_two_launches":
        monkeypatch.setenv("FTMOE_TC_FUSED", "0")
    cfg = W.config("decode_bf16", t_min=T, t_max=T)
    C = W.cache_capacity(cfg)
    cache = _make(ft, cfg, bf16_pool, C, max_tokens=16)
    run = Runner(cache, cfg, C)
    experts = OracleExperts(bf16_pool, max_cached=64)
    for step in W.decode_trace(cfg, steps=4):
        d = step[0]
        out, idx, w = run.call(0, d["x"], d["logits"])
        ref_out, _, _ = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
        assert out_err(bf16_dev_to_f64(out), ref_out) <= TOL["bf16"]
    run.check_state()
    cache.close()


def test_output_independent_of_cache_state(ft, bf16_pool):
    """Cold cache, warm cache, capacity = pool and capacity 0 (everything bypassed from
    staging) give bit-identical outputs for the same inputs."""
    import torch
    cfg = W.config("decode_bf16")
    d = W.trace_step(cfg, 3, 0, 16)
    outs = []
    for C in (W.cache_capacity(cfg), cfg.experts, 0):
        cache = _make(ft, cfg, bf16_pool, C, max_tokens=16)
        run = Runner(cache, cfg, C)
        for _ in range(2):
            out, _, _ = run.call(0, d["x"], d["logits"])
            outs.append(out.clone())
        cache.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_full_trace_cache_state_small_shape(ft):
    """The whole 512-step trace (1..16 tokens/step, C = 37% of 128) at a reduced H/I: every
    call's hit/miss/bypass/eviction counts and periodic full snapshots match the oracle."""
    cfg = W.config("decode_bf16", hidden=64, inter=64)
    pool = HostPool(cfg)
    C = W.cache_capacity(cfg)
    cache = _make(ft, cfg, pool, C)
    run = Runner(cache, cfg, C)
    for s, step in enumerate(W.decode_trace(cfg)):
        d = step[0]
        run.call(0, d["x"], d["logits"])
        if s % 64 == 63:
            run.check_state()
    run.check_state()
    st = cache.stats()
    assert st["calls"] == cfg.steps
    cache.close()


def test_elastic_full_trace_small_shape(ft):
    """1024 steps with resizes 40% -> 15% -> 30% of the pool at steps 341 and 682."""
    cfg = W.config("elastic_nvfp4", hidden=64, inter=64)
    pool = HostPool(cfg)
    C = W.cache_capacity(cfg)
    cache = _make(ft, cfg, pool, C)
    run = Runner(cache, cfg, C)
    sched = dict(cfg.resize)
    for s, step in enumerate(W.decode_trace(cfg)):
        if s in sched:
            run.resize(W.cache_capacity(cfg, sched[s]))
            run.check_state()
        run.call(0, step[0]["x"], step[0]["logits"])
    run.check_state()
    assert cache.stats()["capacity"] == W.cache_capacity(cfg, 0.30)
    cache.close()


def test_elastic_nvfp4_full_size(ft):
    cfg = W.config("elastic_nvfp4")
    pool = HostPool(cfg)
    C = W.cache_capacity(cfg)
    cache = _make(ft, cfg, pool, C)
    run = Runner(cache, cfg, C)
    experts = OracleExperts(pool, max_cached=128)
    tr = W.decode_trace(cfg, steps=18)
    worst = 0.0
    for s, step in enumerate(tr):
        if s == 6:
            run.resize(W.cache_capacity(cfg, 0.15)); run.check_state()
        if s == 12:
            run.resize(W.cache_capacity(cfg, 0.30)); run.check_state()
        d = step[0]
        out, idx, _ = run.call(0, d["x"], d["logits"])
        if s % 2 == 0:
            ref_out, ref_idx, _ = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
            assert np.array_equal(idx, ref_idx)
            worst = max(worst, out_err(bf16_dev_to_f64(out), ref_out))
    assert worst <= TOL["nvfp4"], worst
    run.check_state()
    cache.close()


def test_mxfp4_43_layers_full_size(ft):
    """284B-shaped: 43 layers, one global LRU at 20% of 11008 keys (2201 slots). The host
    pool aliases 13 physical blobs (key -> key % 13); keys, cache and PCIe bytes are real."""
    cfg = W.config("decode_mxfp4")
    pool = HostPool(cfg, images=13)
    C = W.cache_capacity(cfg)
    assert C == 2201
    cache = _make(ft, cfg, pool, C)
    run = Runner(cache, cfg, C)
    experts = OracleExperts(pool, max_cached=13)
    worst = 0.0
    for s, step in enumerate(W.decode_trace(cfg, steps=3)):
        for d in step:
            out, idx, _ = run.call(d["layer"], d["x"], d["logits"])
            if d["layer"] in (0, 21, 42):
                ref_out, ref_idx, _ = oracle_call(experts, d["layer"], d["x"], d["logits"], cfg.top_k)
                assert np.array_equal(idx, ref_idx)
                worst = max(worst, out_err(bf16_dev_to_f64(out), ref_out))
        run.check_state()
    assert worst <= TOL["mxfp4"], worst
    cache.close()


def test_mxfp4_43_layers_full_trace_small_shape(ft):
    """The 284B-shaped cache over its whole trace: 256 steps x 43 layers (11,008 calls) into
    one global LRU of 2201 slots (20 % of 43 x 256 keys), at a reduced expert size (H = I =
    256). Every call's hits, misses, bypasses and evictions are checked against the oracle's
    LRU simulator, the full cache state every 32 steps and at the end, and sampled outputs
    against the oracle layer."""
    cfg = W.config("decode_mxfp4", hidden=256, inter=256)
    pool = HostPool(cfg, images=13)
    C = W.cache_capacity(cfg)
    assert C == 2201
    cache = _make(ft, cfg, pool, C)
    run = Runner(cache, cfg, C)
    experts = OracleExperts(pool, max_cached=13)
    worst = 0.0
    n = 0
    for s, step in enumerate(W.decode_trace(cfg)):
        for d in step:
            out, idx, _ = run.call(d["layer"], d["x"], d["logits"])
            n += 1
            if s % 32 == 0 and d["layer"] in (0, 42):
                ref_out, ref_idx, _ = oracle_call(experts, d["layer"], d["x"], d["logits"], cfg.top_k)
                assert np.array_equal(idx, ref_idx)
                worst = max(worst, out_err(bf16_dev_to_f64(out), ref_out))
        if s % 32 == 31:
            run.check_state()
    run.check_state()
    assert n == 256 * 43
    st = cache.stats()
    assert st["calls"] == n
    assert worst <= TOL["mxfp4"], worst
    cache.close()


def test_ragged_and_empty_calls(ft):
    import torch
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    cache = _make(ft, cfg, pool, capacity=3, max_tokens=16)
    run = Runner(cache, cfg, 3)
    experts = OracleExperts(pool)
    rng = np.random.default_rng(9)
    for T in (1, 5, 16, 11, 2):
        x = W.tiny_inputs(W.config("tiny", tokens=T))
        logits = rng.standard_normal((T, cfg.experts)).astype(np.float32)
        out, idx, _ = run.call(0, x, logits)
        ref_out, ref_idx, _ = oracle_call(experts, 0, x, logits, cfg.top_k)
        assert np.array_equal(idx, ref_idx)
        assert out_err(bf16_dev_to_f64(out), ref_out) <= TOL["bf16"]
    run.check_state()
    before = cache.stats()
    x = to_dev_bf16(W.tiny_inputs(cfg))
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    cache.forward(0, x, 0, out)                      # T = 0: no work
    assert cache.stats()["calls"] == before["calls"] + 1
    assert cache.forward_status(0, x, 17, out) == ft.FT_ERR_INVALID      # T > max_tokens
    assert cache.forward_status(1, x, 4, out) == ft.FT_ERR_INVALID       # bad layer
    assert cache.forward_status(0, x, 4, x) == ft.FT_ERR_INVALID         # out aliases x
    assert cache.forward_status(0, x, 4, out) == ft.FT_ERR_INVALID       # no router, no logits
    cache.close()


def test_nan_logit_is_reported(ft):
    import torch
    from ref import to_dev
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    cache = _make(ft, cfg, pool, capacity=8)
    x = to_dev_bf16(W.tiny_inputs(cfg))
    lg = np.zeros((16, 8), dtype=np.float32)
    lg[3, 5] = np.nan
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    assert cache.forward_status(0, x, 16, out, logits=to_dev(lg)) == ft.FT_ERR_INVALID
    lg[3, 5] = 0.0
    assert cache.forward_status(0, x, 16, out, logits=to_dev(lg)) == ft.FT_OK   # flag cleared
    cache.close()


def test_injected_alloc_failure_leaves_cache_intact(ft, monkeypatch):
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    monkeypatch.setenv("FTMOE_FAULT", "alloc_fail")
    cache = _make(ft, cfg, pool, capacity=4, max_tokens=16)
    run = Runner(cache, cfg, 4)
    rng = np.random.default_rng(1)
    x = W.tiny_inputs(cfg)
    for _ in range(3):
        run.call(0, x, rng.standard_normal((16, 8)).astype(np.float32))
    snap = cache.snapshot()
    assert cache.resize_status(2) == ft.FT_ERR_OOM
    snap2 = cache.snapshot()
    assert np.array_equal(snap[0], snap2[0]) and np.array_equal(snap[1], snap2[1])
    run.call(0, x, rng.standard_normal((16, 8)).astype(np.float32))   # still usable
    run.check_state()
    cache.close()


def test_injected_fill_failure(ft, monkeypatch):
    import torch
    from ref import to_dev
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    monkeypatch.setenv("FTMOE_FAULT", "fill_fail")
    cache = _make(ft, cfg, pool, capacity=4, max_tokens=16)
    x = to_dev_bf16(W.tiny_inputs(cfg))
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = to_dev(np.random.default_rng(2).standard_normal((16, 8)).astype(np.float32))
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_CUDA
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_STATE
    cache.close()


def test_host_wait_timeout(ft, monkeypatch):
    """A bounded host wait: the device is kept busy (a finite sleep kernel) longer than the
    wait limit, so the forward returns FT_ERR_TIMEOUT instead of blocking."""
    import torch
    from ref import to_dev
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    monkeypatch.setenv("FTMOE_WAIT_MS", "5")
    cache = _make(ft, cfg, pool, capacity=8, max_tokens=16)
    x = to_dev_bf16(W.tiny_inputs(cfg))
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = to_dev(np.zeros((16, 8), dtype=np.float32))
    torch.cuda._sleep(int(4e8))          # ~0.2 s of device time, then it ends by itself
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_STATE
    cache.close()


def test_miss_groups_match_single_miss_pass(ft, monkeypatch):
    """Misses run in two groups (all but the last copied, then the last) by default; the
    outputs are bit-identical to one FFN pass over all misses (FTMOE_MISS_GROUPS=0), and
    cache counts equal the oracle's."""
    import torch
    cfg = W.config("decode_bf16", hidden=512, inter=256, t_min=16, t_max=16)
    pool = HostPool(cfg)
    C = W.cache_capacity(cfg)
    outs = {}
    for groups in ("1", "0"):
        monkeypatch.setenv("FTMOE_MISS_GROUPS", groups)
        cache = _make(ft, cfg, pool, C)
        run = Runner(cache, cfg, C)
        outs[groups] = []
        for step in W.decode_trace(cfg, steps=12):
            d = step[0]
            out, _, _ = run.call(0, d["x"], d["logits"])
            outs[groups].append(out.clone())
        run.check_state()
        assert cache.stats()["misses"] > 2 * 12        # several misses per call: two groups
        cache.close()
    assert all(torch.equal(a, b) for a, b in zip(outs["1"], outs["0"]))
