"""FP4 (MXFP4 / NVFP4) expert FFN through the cache (C ABI) vs the oracle: the block-scaled
tcgen05 path (activations split into E2M1 pieces) and the CUDA-core GEMV path, at one and
sixteen tokens per call; routing and cache state bit-exact, outputs within the FP4 normwise
tolerance and bit-identical across cache states."""
import numpy as np
import pytest

import workloads as W
from workloads.host import HostPool
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


def _cfg(fmt, T):
    if fmt == "nvfp4":   # the elastic layer's shape: H 2048, I 768, 128 experts top-8
        return W.config("elastic_nvfp4", t_min=T, t_max=T)
    # the 284B layer's experts (H 4096, I 2048, top-6 of 256) on one layer, cache 20 %
    return W.config("decode_mxfp4", layers=1, t_min=T, t_max=T)


_pools = {}


def _pool(fmt):
    if fmt not in _pools:
        cfg = _cfg(fmt, 1)
        _pools[fmt] = HostPool(cfg, images=8 if fmt == "mxfp4" else None)
    return _pools[fmt]


def _make(ft, cfg, pool, capacity, max_tokens=16):
    c = ft.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, max_tokens,
                       cfg.wfmt, capacity)
    return ft.MoECache(c, pool.ptrs, None)


@pytest.mark.parametrize("path", ["tcgen05", "simt"])
@pytest.mark.parametrize("T", [1, 16])
@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_fp4_decode_fixed_T(ft, fmt, T, path, monkeypatch):
    if path == "simt":
        monkeypatch.setenv("FTMOE_FFN", "simt")
    cfg = _cfg(fmt, T)
    pool = _pool(fmt)
    C = W.cache_capacity(cfg)
    cache = _make(ft, cfg, pool, C)
    run = Runner(cache, cfg, C)
    experts = OracleExperts(pool, max_cached=8 if fmt == "mxfp4" else 64)
    worst = 0.0
    for step in W.decode_trace(cfg, steps=8):
        d = step[0]
        out, idx, _ = run.call(0, d["x"], d["logits"])
        ref_out, ref_idx, _ = oracle_call(experts, 0, d["x"], d["logits"], cfg.top_k)
        assert np.array_equal(idx, ref_idx)
        worst = max(worst, out_err(bf16_dev_to_f64(out), ref_out))
    run.check_state()
    cache.close()
    print("%s %s T=%d worst normwise err %.3e" % (fmt, path, T, worst))
    assert worst <= TOL[fmt], worst
    if path == "tcgen05":
        # four E2M1 pieces carry the bf16 activations: the error stays near bf16 rounding
        assert worst <= 5e-3, worst


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_fp4_output_independent_of_cache_state(ft, fmt):
    """Cold, warm, whole pool resident and capacity 0 (all bypassed) give identical bits."""
    import torch
    cfg = _cfg(fmt, 16)
    pool = _pool(fmt)
    d = W.trace_step(cfg, 5, 0, 8)
    outs = []
    for C in (W.cache_capacity(cfg), cfg.experts, 0):
        cache = _make(ft, cfg, pool, C)
        run = Runner(cache, cfg, C)
        for _ in range(2):
            out, _, _ = run.call(0, d["x"], d["logits"])
            outs.append(out.clone())
        cache.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
