"""Router logits and warp-per-token top-k: CUDA kernels (through the C ABI) vs the oracle."""
import numpy as np
import pytest

import workloads as W
from oracle import formats, moe

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


def _logits_gpu(ft, x_bits, wr):
    import torch
    from ref import to_dev, to_dev_bf16
    T, H = x_bits.shape
    E = wr.shape[0]
    out = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ft.router_logits(to_dev_bf16(x_bits), T, H, to_dev(wr), E, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", 16), ("decode_bf16", 13), ("decode_mxfp4", 8),
                                    ("decode_bf16", 64), ("decode_mxfp4", 1000), ("prefill_mxfp4", 4096)])
def test_router_logits_parity(ft, name, T):
    """Decode sizes (one warp per token-expert pair) and prefill sizes (the tiled kernel,
    T >= 64, ragged token tiles) against the oracle's fp64 logits."""
    cfg = W.config(name)
    wr = W.router_weights(cfg, layers=1)[0]
    x = W.tiny_inputs(W.config("tiny", hidden=cfg.hidden, tokens=T))
    got = _logits_gpu(ft, x, wr)
    ref = moe.router_logits(formats.bf16_to_f64(x), wr)
    # fp32 accumulation of H products: bound |err| by a few ulps of sum |x||w|
    bound = 8 * cfg.hidden * np.finfo(np.float32).eps * (np.abs(formats.bf16_to_f64(x)) @ np.abs(wr.T))
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


def _topk_gpu(ft, logits, k):
    import torch
    from ref import to_dev
    T, E = logits.shape
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ft.topk_softmax(to_dev(logits.astype(np.float32)), T, E, k, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def _check_topk(ft, logits, k):
    idx, w = _topk_gpu(ft, logits, k)
    ref_idx = moe.topk(logits.astype(np.float64), k)
    ref_w = moe.gate_weights(logits.astype(np.float64), ref_idx)
    assert np.array_equal(idx, ref_idx)
    assert np.max(np.abs(w - ref_w)) <= 2e-6
    assert np.allclose(w.sum(1), 1.0, atol=2e-6)


@pytest.mark.parametrize("name", ["decode_bf16", "decode_mxfp4", "elastic_nvfp4"])
def test_topk_on_trace_logits(ft, name):
    cfg = W.config(name)
    tr = W.decode_trace(cfg, steps=6)
    for step in tr:
        for d in step[:3]:
            _check_topk(ft, d["logits"], cfg.top_k)
            got, _ = _topk_gpu(ft, d["logits"], cfg.top_k)
            # the generator's picks are exactly the top-k set
            assert np.array_equal(np.sort(got, 1), np.sort(d["picks"], 1))


@pytest.mark.parametrize("E,k", [(1, 1), (7, 3), (32, 32), (33, 5), (256, 6), (1000, 17),
                                 (1024, 32), (1024, 1)])
def test_topk_shapes(ft, E, k):
    rng = np.random.default_rng(E * 100 + k)
    logits = rng.standard_normal((37, E)).astype(np.float32)
    _check_topk(ft, logits, k)


def test_topk_ties_and_prefill_size(ft):
    rng = np.random.default_rng(5)
    ties = rng.integers(-2, 3, size=(64, 128)).astype(np.float32)   # many exact ties
    _check_topk(ft, ties, 8)
    big = (rng.standard_normal((4096, 256)) * 0.5).astype(np.float32)
    _check_topk(ft, big, 6)
