"""The fused decode kernel (FT_FLAG_FUSED_DECODE: one cooperative launch per forward call
for top-k, lookup, row gather, expert FFN and combine; a host fill agent copies the misses
and sets their device flags, so the call never blocks) against the oracle and against the
default multi-launch path: routing, per-call cache counts and snapshots bit-exact against
the LRU simulators, outputs within the normwise tolerance of the oracle and bit-identical
to the default path's. Failures on the host end the kernel through its flags (no GPU
fault) and are reported by the next call on the handle."""
import time

import numpy as np
import pytest

import workloads as W
from workloads.host import HostPool
from oracle import lru, policies
from ref import (TOL, OracleExperts, Runner, bf16_dev_to_f64, out_err, oracle_call, to_dev,
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


def _make(ft, cfg, pool, capacity, fused, max_tokens=None, router=None, policy=0):
    mt = max_tokens or max(cfg.t_max, cfg.tokens, 1)
    c = ft.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, mt, cfg.wfmt,
                       capacity, policy=policy, fused_decode=fused)
    return ft.MoECache(c, pool.ptrs, router)


@pytest.fixture(scope="module")
def bf16_pool():
    return HostPool(W.config("decode_bf16"))


def _pair_call(runs, layer, x, logits, T=None):
    res = [r.call(layer, x, logits, T=T) for r in runs]
    (o0, i0, w0), (o1, i1, w1) = res
    assert np.array_equal(i0, i1)
    assert np.array_equal(w0, w1)
    assert bool((o0 == o1).all()), "fused output differs from the default path"
    return res[1]


def test_fused_decode_bf16_trace_parity(ft, bf16_pool):
    """35B-A3B-shaped layer, LRU at 37 %: 24 steps of 1..16 tokens. Counts per call and
    snapshots against the simulator, outputs against the oracle and bitwise against the
    default path."""
    cfg = W.config("decode_bf16")
    C = W.cache_capacity(cfg)
    runs = [Runner(_make(ft, cfg, bf16_pool, C, fused), cfg, C) for fused in (False, True)]
    experts = OracleExperts(bf16_pool, max_cached=64)
    worst = 0.0
    for s, step in enumerate(W.decode_trace(cfg, steps=24)):
        d = step[0]
        out, idx, w = _pair_call(runs, 0, d["x"], d["logits"])
        if s % 4 == 0:
            ref_out, ref_idx, ref_w = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
            assert np.array_equal(idx, ref_idx)
            assert np.max(np.abs(w - ref_w)) <= 2e-6
            worst = max(worst, out_err(bf16_dev_to_f64(out), ref_out))
            for r in runs:
                r.check_state()
    assert worst <= TOL["bf16"], worst
    assert runs[0].cache.stats() == runs[1].cache.stats()
    for r in runs:
        r.cache.close()


@pytest.mark.parametrize("T", [1, 16])
def test_fused_fixed_T_all_resident_and_cold(ft, bf16_pool, T):
    """A cold cache (every expert a miss, filled while the kernel runs), then warm calls
    (hits only), at T = 1 and T = 16."""
    cfg = W.config("decode_bf16", t_min=T, t_max=T)
    runs = [Runner(_make(ft, cfg, bf16_pool, cfg.experts, fused, max_tokens=16), cfg, cfg.experts)
            for fused in (False, True)]
    experts = OracleExperts(bf16_pool, max_cached=64)
    d = W.trace_step(cfg, 5, 0, T)
    ref_out, _, _ = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
    outs = []
    for _ in range(3):
        out, _, _ = _pair_call(runs, 0, d["x"], d["logits"])
        assert out_err(bf16_dev_to_f64(out), ref_out) <= TOL["bf16"]
        outs.append(out.clone())
    assert bool((outs[0] == outs[2]).all())
    st = runs[1].cache.stats()
    U = len(np.unique(d["picks"]))
    assert st["misses"] == U and st["hits"] == 2 * U
    for r in runs:
        r.check_state()
        r.cache.close()


def test_fused_output_independent_of_cache_state(ft, bf16_pool):
    """Cold, warm, capacity = pool and capacity 0 (all bypassed through staging): identical
    outputs, and identical to the default path's."""
    import torch
    cfg = W.config("decode_bf16")
    d = W.trace_step(cfg, 3, 0, 16)
    outs = []
    for fused in (False, True):
        for C in (W.cache_capacity(cfg), cfg.experts, 0):
            cache = _make(ft, cfg, bf16_pool, C, fused, max_tokens=16)
            run = Runner(cache, cfg, C)
            for _ in range(2):
                out, _, _ = run.call(0, d["x"], d["logits"])
                outs.append(out.clone())
            cache.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_fused_full_trace_cache_state_small_shape(ft):
    """The whole 512-step trace at reduced H / I through the fused kernel: every call's counts
    and periodic snapshots against the simulator."""
    cfg = W.config("decode_bf16", hidden=64, inter=64)
    pool = HostPool(cfg)
    C = W.cache_capacity(cfg)
    run = Runner(_make(ft, cfg, pool, C, True), cfg, C)
    for s, step in enumerate(W.decode_trace(cfg)):
        d = step[0]
        run.call(0, d["x"], d["logits"])
        if s % 64 == 0:
            run.check_state()
    run.check_state()
    run.cache.close()


def test_fused_multilayer_and_resize(ft):
    """4 layers sharing one global LRU with resizes between steps (elastic shape, BF16)."""
    cfg = W.config("elastic_nvfp4", wfmt="bf16", hidden=128, inter=64, layers=4, steps=60)
    pool = HostPool(cfg, images=9)
    C = 60
    runs = [Runner(_make(ft, cfg, pool, C, fused), cfg, C) for fused in (False, True)]
    for s, step in enumerate(W.decode_trace(cfg)):
        if s in (20, 40):
            for r in runs:
                r.resize(C // 3 if s == 20 else C)
        for d in step:
            _pair_call(runs, d["layer"], d["x"], d["logits"])
        if s % 10 == 0:
            for r in runs:
                r.check_state()
    for r in runs:
        r.check_state()
        r.cache.close()


@pytest.mark.parametrize("policy", ["layer_lru", "static"])
def test_fused_comparator_policies(ft, policy):
    cfg = W.config("decode_mxfp4", wfmt="bf16", layers=4, hidden=64, inter=64, steps=16)
    pool = HostPool(cfg, images=7)
    C = W.cache_capacity(cfg)
    pol = ft.POLICY_LAYER_LRU if policy == "layer_lru" else ft.POLICY_STATIC
    hot = list(range(0, cfg.keys, 5))[:C]
    runs = []
    for fused in (False, True):
        cache = _make(ft, cfg, pool, C, fused, policy=pol)
        if policy == "static":
            cache.pin(hot)
            sim = policies.static_set(C, cfg.experts, hot)
        else:
            sim = policies.LayerLRU(C, cfg.experts, cfg.layers)
        runs.append(Runner(cache, cfg, C, sim=sim))
    for step in W.decode_trace(cfg):
        for d in step:
            _pair_call(runs, d["layer"], d["x"], d["logits"])
    for r in runs:
        r.check_state()
        r.cache.close()


def test_fused_router_in_the_loop_and_ragged(ft):
    """Router logits computed from router weights (tiny layer), and T = 1..16 with T = 0."""
    import torch
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    router = W.router_weights(cfg)
    runs = [Runner(_make(ft, cfg, pool, 3, fused, max_tokens=16, router=router), cfg, 3)
            for fused in (False, True)]
    experts = OracleExperts(pool)
    from oracle import formats, moe
    for T in (16, 1, 5, 11, 2):
        x = W.tiny_inputs(W.config("tiny", tokens=T))
        lg = moe.router_logits(formats.bf16_to_f64(x), router[0])
        out, idx, _ = _pair_call(runs, 0, x, None)
        ref_out, _, _ = oracle_call(experts, 0, x, lg, cfg.top_k)
        assert out_err(bf16_dev_to_f64(out), ref_out) <= TOL["bf16"]
    for r in runs:
        r.check_state()
    cache = runs[1].cache
    before = cache.stats()
    xd = to_dev_bf16(W.tiny_inputs(cfg))
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    cache.forward(0, xd, 0, out)
    assert cache.stats()["calls"] == before["calls"] + 1
    for r in runs:
        r.cache.close()


def test_fused_nan_logit_is_reported(ft):
    import torch
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    cache = _make(ft, cfg, pool, 8, True, max_tokens=16)
    x = to_dev_bf16(W.tiny_inputs(cfg))
    lg = np.zeros((16, 8), dtype=np.float32)
    lg[3, 5] = np.nan
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    assert cache.forward_status(0, x, 16, out, logits=to_dev(lg)) == ft.FT_OK    # asynchronous
    torch.cuda.synchronize()
    lg[3, 5] = 0.0
    assert cache.forward_status(0, x, 16, out, logits=to_dev(lg)) == ft.FT_ERR_INVALID   # reported
    assert cache.forward_status(0, x, 16, out, logits=to_dev(lg)) == ft.FT_OK
    cache.stats()
    cache.close()


def test_fused_injected_fill_failure_ends_the_kernel(ft, monkeypatch):
    """The fill agent refuses to copy (injected): it marks every pending fill flag abandoned,
    the kernel's miss tiles see that and the kernel ends with an error code well before its
    wait bound; the next call reports the failure, the one after FT_ERR_STATE."""
    import torch
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    monkeypatch.setenv("FTMOE_FAULT", "fill_fail")
    cache = _make(ft, cfg, pool, 4, True, max_tokens=16)
    x = to_dev_bf16(W.tiny_inputs(cfg))
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = to_dev(np.random.default_rng(2).standard_normal((16, 8)).astype(np.float32))
    t0 = time.perf_counter()
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_OK             # launched
    torch.cuda.synchronize()                                 # the kernel ends by itself
    assert time.perf_counter() - t0 < 2.0
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_CUDA       # reported
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_STATE
    cache.close()


def test_fused_host_wait_timeout(ft, monkeypatch):
    """The device is kept busy (a finite sleep kernel) past the host's wait limit: the fill
    agent gives up on the call's routing, abandons its fill flags (so the kernel, once it
    runs, ends by itself), and the next call reports FT_ERR_TIMEOUT."""
    import torch
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    monkeypatch.setenv("FTMOE_WAIT_MS", "5")
    cache = _make(ft, cfg, pool, 8, True, max_tokens=16)
    x = to_dev_bf16(W.tiny_inputs(cfg))
    out = torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = to_dev(np.zeros((16, 8), dtype=np.float32))
    torch.cuda._sleep(int(4e8))          # ~0.2 s of device time
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_OK             # launched
    torch.cuda.synchronize()
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_TIMEOUT    # reported
    assert cache.forward_status(0, x, 16, out, logits=lg) == ft.FT_ERR_STATE
    cache.close()


def test_fused_rejects_unsupported_configs(ft):
    cfg = W.config("elastic_nvfp4", hidden=512, inter=256, t_max=17)
    pool = HostPool(cfg, images=4)
    with pytest.raises(ft.FtError) as e:
        _make(ft, cfg, pool, 8, True)          # FP4 weights, more than 16 tokens per call
    assert e.value.status == ft.FT_ERR_INVALID
    cfg = W.config("decode_mxfp4", wfmt="bf16", layers=1, hidden=64, inter=64, t_max=33)
    pool = HostPool(cfg, images=4)
    with pytest.raises(ft.FtError):
        _make(ft, cfg, pool, 8, True)          # BF16, more than 32 tokens per call


def test_fused_calls_queue_without_host_waits(ft, bf16_pool):
    """Forty calls issued back to back with no synchronisation in between (misses included):
    the final cache state, the statistics and the last outputs equal the default path's."""
    import torch
    cfg = W.config("decode_bf16")
    C = W.cache_capacity(cfg)
    caches = [_make(ft, cfg, bf16_pool, C, fused) for fused in (False, True)]
    steps = list(W.decode_trace(cfg, steps=40))
    xs = [(to_dev_bf16(st[0]["x"]), to_dev(st[0]["logits"]), st[0]["T"]) for st in steps]
    outs = [[torch.empty((16, cfg.hidden), dtype=torch.bfloat16, device="cuda") for _ in steps]
            for _ in caches]
    for ci, cache in enumerate(caches):
        for i, (x, lg, T) in enumerate(xs):
            cache.forward(0, x, T, outs[ci][i], logits=lg)
    torch.cuda.synchronize()
    for i, (_, _, T) in enumerate(xs):
        assert torch.equal(outs[0][i][:T], outs[1][i][:T])
    assert caches[0].stats() == caches[1].stats()
    s0, s1 = caches[0].snapshot(), caches[1].snapshot()
    assert np.array_equal(s0[0], s1[0]) and np.array_equal(s0[1], s1[1])
    for c in caches:
        c.close()


@pytest.mark.parametrize("name", ["decode_mxfp4", "elastic_nvfp4"])
def test_fused_fp4_matches_default_and_simulator(ft, name):
    """FP4 weights (block-scaled tcgen05 path) through the fused call: outputs bit-identical to
    the default path, per-call counts and snapshots against the simulator, one call per layer
    against the oracle. MXFP4: 4 layers of the 256-expert top-6 routing; NVFP4: resizes."""
    cfg = W.config(name, layers=4 if name == "decode_mxfp4" else 1, hidden=512, inter=256, steps=12)
    pool = HostPool(cfg, images=7)
    C = W.cache_capacity(cfg)
    runs = [Runner(_make(ft, cfg, pool, C, fused), cfg, C) for fused in (False, True)]
    experts = OracleExperts(pool, max_cached=7)
    worst = 0.0
    for s, step in enumerate(W.decode_trace(cfg)):
        if name == "elastic_nvfp4" and s in (4, 8):
            for r in runs:
                r.resize(C // 3 if s == 4 else C)
        for d in step:
            out, idx, _ = _pair_call(runs, d["layer"], d["x"], d["logits"])
            if s % 4 == 1 and d["layer"] == 0:
                ref, ref_idx, _ = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
                assert np.array_equal(idx, ref_idx)
                worst = max(worst, out_err(bf16_dev_to_f64(out), ref))
        if s % 4 == 0:
            for r in runs:
                r.check_state()
    assert worst <= TOL[cfg.wfmt], worst
    assert runs[0].cache.stats() == runs[1].cache.stats()
    for r in runs:
        r.check_state()
        r.cache.close()


def test_fused_fp4_full_size_mxfp4(ft):
    """The 284B-shaped MXFP4 layer at full size (H 4096, I 2048), 2 layers, 6 steps: fused and
    default outputs bit-identical, counts against the simulator."""
    cfg = W.config("decode_mxfp4", layers=2, steps=6)
    pool = HostPool(cfg, images=16)
    C = W.cache_capacity(cfg)
    runs = [Runner(_make(ft, cfg, pool, C, fused), cfg, C) for fused in (False, True)]
    for step in W.decode_trace(cfg):
        for d in step:
            _pair_call(runs, d["layer"], d["x"], d["logits"])
    for r in runs:
        r.check_state()
        r.cache.close()


@pytest.mark.parametrize("T", [17, 32])
def test_32_token_tiles_default_and_fused(ft, bf16_pool, T):
    """Calls of 17..32 tokens use 32-token N tiles (the BF16 kernel's second template): the
    default and fused paths against the oracle, bit-identical to each other, cold then warm."""
    cfg = W.config("decode_bf16", t_min=T, t_max=T)
    C = W.cache_capacity(cfg)
    runs = [Runner(_make(ft, cfg, bf16_pool, C, fused, max_tokens=32), cfg, C) for fused in (False, True)]
    experts = OracleExperts(bf16_pool, max_cached=64)
    for s, step in enumerate(W.decode_trace(cfg, steps=4)):
        d = step[0]
        out, idx, _ = _pair_call(runs, 0, d["x"], d["logits"])
        if s % 2 == 0:
            ref, ref_idx, _ = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
            assert np.array_equal(idx, ref_idx)
            assert out_err(bf16_dev_to_f64(out), ref) <= TOL["bf16"]
    for r in runs:
        r.check_state()
        r.cache.close()


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_fp4_32_token_tiles(ft, fmt):
    """FP4 calls of 32 tokens use 32-token tiles (four pieces: 128 N rows, one MMA issuer) on
    the default path: against the oracle and independent of the cache state."""
    import torch
    name = "decode_mxfp4" if fmt == "mxfp4" else "elastic_nvfp4"
    cfg = W.config(name, layers=1, hidden=512, inter=256, t_min=32, t_max=32)
    pool = HostPool(cfg, images=9)
    experts = OracleExperts(pool, max_cached=9)
    d = W.trace_step(cfg, 2, 0, 32)
    ref, _, _ = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
    outs = []
    for C in (W.cache_capacity(cfg), 0):
        run = Runner(_make(ft, cfg, pool, C, False, max_tokens=32), cfg, C)
        out, _, _ = run.call(0, d["x"], d["logits"])
        assert out_err(bf16_dev_to_f64(out), ref) <= TOL[fmt]
        outs.append(out.clone())
        run.cache.close()
    assert torch.equal(outs[0], outs[1])
