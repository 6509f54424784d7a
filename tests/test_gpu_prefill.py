"""Prefill-sized MoE layer forward with double-buffered full-layer streaming (C ABI) vs the
oracle: each layer's output within the normwise tolerance, refills bit-identical."""
import numpy as np
import pytest

import workloads as W
from workloads.host import HostPool
from ref import TOL, OracleExperts, bf16_dev_to_f64, out_err, oracle_call, to_dev, to_dev_bf16

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


def _make(ft, cfg, pool, T, router=None, capacity=1):
    c = ft.make_config(cfg.layers, cfg.experts, cfg.hidden, cfg.inter, cfg.top_k, 16, cfg.wfmt,
                       capacity, max_prefill_tokens=T)
    return ft.MoECache(c, pool.ptrs, router)


def _run(cache, cfg, layer, x_bits, logits=None):
    import torch
    T = x_bits.shape[0]
    out = torch.empty((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    lg = to_dev(logits) if logits is not None else None
    cache.prefill(layer, to_dev_bf16(x_bits), T, out, logits=lg)
    torch.cuda.synchronize()
    return out


def test_prefill_bf16_layers_in_order(ft):
    """35B-A3B-shaped layer (128 experts, top-8, ~256 tokens per expert), 4096 tokens, four
    layers streamed in order, then layer 0 again (a refill). Pool aliased onto 131 blobs so
    every layer has different weights."""
    import torch
    cfg = W.config("prefill_bf16")
    pool = HostPool(cfg, images=131)
    cache = _make(ft, cfg, pool, cfg.tokens)
    experts = OracleExperts(pool, max_cached=131)
    first = None
    for layer in (0, 1, 2, 3, 0):
        x, logits = W.prefill_inputs(cfg, layer)
        out = _run(cache, cfg, layer, x, logits)
        if layer == 0 and first is not None:
            assert torch.equal(out, first)            # refilled buffer, same result
            continue
        if layer == 0:
            first = out.clone()
        tokens = None if layer in (0, 3) else np.arange(0, cfg.tokens, 7)
        ref, _, _ = oracle_call(experts, layer, x, logits, cfg.top_k, tokens=tokens)
        got = bf16_dev_to_f64(out)
        if tokens is not None:
            got = got[tokens]
        assert out_err(got, ref) <= TOL["bf16"], layer
    st = cache.stats()
    assert st["hits"] == 0 and st["misses"] == 0          # the LRU is not consulted
    cache.close()


def test_prefill_ragged_token_counts(ft):
    """T far from a multiple of anything; few tokens per expert (small N tiles)."""
    cfg = W.config("prefill_bf16", layers=2)
    pool = HostPool(cfg, images=131)
    cache = _make(ft, cfg, pool, 1000)
    experts = OracleExperts(pool, max_cached=131)
    for layer, T in ((0, 1000), (1, 37), (0, 1)):
        x, logits = W.prefill_inputs(cfg, layer, tokens=T)
        out = _run(cache, cfg, layer, x, logits)
        ref, _, _ = oracle_call(experts, layer, x, logits, cfg.top_k)
        assert out_err(bf16_dev_to_f64(out), ref) <= TOL["bf16"], (layer, T)
    cache.close()


def test_prefill_mxfp4_full_shape(ft):
    """The 284B-shaped prefill layer at its full size: 4096 tokens, 256 experts top-6, MXFP4
    weights, ~96 routed rows per expert, so every expert spans several 32-token tiles (the
    kernel's N tiles) and the largest exceed 128 rows. The activations enter the block-scaled
    MMA as four E2M1 pieces: outputs within the FP4 tolerance of the plain oracle (no
    activation quantisation in the oracle), on a sample of tokens, for two layers streamed in
    order and a refill of the first (bit-identical)."""
    import torch
    cfg = W.config("prefill_mxfp4", layers=2)
    assert cfg.tokens == 4096
    pool = HostPool(cfg, images=13)
    cache = _make(ft, cfg, pool, cfg.tokens)
    experts = OracleExperts(pool, max_cached=13)
    first = None
    worst = 0.0
    for layer in (0, 1, 0):
        x, logits = W.prefill_inputs(cfg, layer)
        out = _run(cache, cfg, layer, x, logits)
        if first is not None and layer == 0:
            assert torch.equal(out, first)
            continue
        if layer == 0:
            first = out.clone()
        from oracle import moe
        idx = moe.topk(np.asarray(logits, dtype=np.float64), cfg.top_k)
        rows = np.bincount(idx.reshape(-1), minlength=cfg.experts)
        assert rows.min() > 32 and rows.max() > 96           # 2 to 5 N tiles per expert
        if layer == 0:
            assert rows.max() > 128                             # an entry of five N tiles
        sample = np.arange(layer, cfg.tokens, 16)
        ref, _, _ = oracle_call(experts, layer, x, logits, cfg.top_k, tokens=sample)
        err = out_err(bf16_dev_to_f64(out)[sample], ref)
        worst = max(worst, err)
        assert err <= TOL["mxfp4"], (layer, err)
    cache.close()
    print("MXFP4 prefill, 4096 tokens: worst error vs the plain oracle %.3e" % worst)
    # four pieces carry the bf16 activations: the error stays near the bf16 rounding level
    assert worst <= 5e-3, worst


@pytest.mark.parametrize("T", [1, 300, 1024])
def test_prefill_nvfp4_tensor_path(ft, T):
    """NVFP4 weights (the elastic layer's shape, H 2048, I 768, 128 experts top-8) on the
    block-scaled tensor path at prefill sizes, ragged T included, vs the plain oracle."""
    cfg = W.config("elastic_nvfp4", layers=2)
    pool = HostPool(cfg, images=64)
    cache = _make(ft, cfg, pool, 1024)
    experts = OracleExperts(pool, max_cached=64)
    for layer in (0, 1):
        x, logits = W.prefill_inputs(W.config("prefill_bf16"), layer, tokens=T)
        out = _run(cache, cfg, layer, x, logits)
        sample = np.arange(0, T, 3)
        ref, _, _ = oracle_call(experts, layer, x, logits, cfg.top_k, tokens=sample)
        assert out_err(bf16_dev_to_f64(out)[sample], ref) <= TOL["nvfp4"], (layer, T)
    cache.close()


def test_prefill_mxfp4_simt_path(ft, monkeypatch):
    """The CUDA-core FFN (FTMOE_FFN=simt: exact dequantisation, bf16 activations) at prefill
    size on the 284B-shaped layer, vs the plain oracle."""
    monkeypatch.setenv("FTMOE_FFN", "simt")
    cfg = W.config("prefill_mxfp4", layers=2)
    pool = HostPool(cfg, images=13)
    T = 512
    cache = _make(ft, cfg, pool, T)
    experts = OracleExperts(pool, max_cached=13)
    for layer in (0, 1):
        x, logits = W.prefill_inputs(cfg, layer, tokens=T)
        out = _run(cache, cfg, layer, x, logits)
        sample = np.arange(0, T, 5)
        ref, _, _ = oracle_call(experts, layer, x, logits, cfg.top_k, tokens=sample)
        assert out_err(bf16_dev_to_f64(out)[sample], ref) <= TOL["mxfp4"], layer
    cache.close()


def test_prefill_router_in_the_loop(ft):
    from oracle import formats, moe
    cfg = W.config("tiny", tokens=64)
    pool = HostPool(cfg)
    router = W.router_weights(cfg)
    cache = _make(ft, cfg, pool, 64, router=router)
    x = W.tiny_inputs(cfg)
    ref_logits = moe.router_logits(formats.bf16_to_f64(x), router[0])
    srt = np.sort(ref_logits, axis=1)[:, ::-1]
    keep = np.nonzero(srt[:, cfg.top_k - 1] - srt[:, cfg.top_k] > 1e-4)[0]
    out = _run(cache, cfg, 0, x)
    experts = OracleExperts(pool)
    ref, _, _ = oracle_call(experts, 0, x, ref_logits, cfg.top_k, tokens=keep)
    assert len(keep) > 48
    assert out_err(bf16_dev_to_f64(out)[keep], ref) <= TOL["bf16"]
    cache.close()


def test_prefill_errors(ft):
    import torch
    cfg = W.config("tiny")
    pool = HostPool(cfg)
    c = ft.make_config(1, 8, 256, 128, 2, 16, "bf16", 4)          # no prefill buffers
    cache = ft.MoECache(c, pool.ptrs, None)
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    lg = torch.zeros((16, 8), dtype=torch.float32, device="cuda")
    assert cache.prefill_status(0, x, 16, out, logits=lg) == ft.FT_ERR_STATE
    cache.close()
    cache = _make(ft, cfg, pool, 16)
    assert cache.prefill_status(0, x, 17, out, logits=lg) == ft.FT_ERR_INVALID
    assert cache.prefill_status(1, x, 16, out, logits=lg) == ft.FT_ERR_INVALID
    assert cache.prefill_status(0, x, 0, out, logits=lg) == ft.FT_OK
    cache.close()


def test_prefill_bf16_pair_and_single_cta_kernels(ft, monkeypatch):
    """The 4096-token 35B-A3B-shaped layer through the CTA-pair kernel (256 x 256 tiles over
    two CTAs, the default) and through the one-CTA kernel (FTMOE_PAIR=0): both within the
    normwise tolerance of the oracle on a token sample, and within it of each other."""
    import torch
    cfg = W.config("prefill_bf16", layers=1)
    pool = HostPool(cfg, images=131)
    experts = OracleExperts(pool, max_cached=131)
    x, logits = W.prefill_inputs(cfg, 0)
    outs = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("FTMOE_PAIR", mode)
        cache = _make(ft, cfg, pool, cfg.tokens)
        outs[mode] = _run(cache, cfg, 0, x, logits).clone()
        cache.close()
    tokens = np.arange(0, cfg.tokens, 5)
    ref, _, _ = oracle_call(experts, 0, x, logits, cfg.top_k, tokens=tokens)
    for mode, out in outs.items():
        assert out_err(bf16_dev_to_f64(out)[tokens], ref) <= TOL["bf16"], mode
    a, b = bf16_dev_to_f64(outs["1"]), bf16_dev_to_f64(outs["0"])
    assert out_err(a, b) <= TOL["bf16"]
    assert torch.isfinite(outs["1"].float()).all()
