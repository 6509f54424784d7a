"""ft_expert_ffn_noalloc: the single-expert FFN that allocates no device memory.

It is for callers that cannot allocate device memory at the moment they need an expert's
output: an engine that has already handed its whole VRAM budget to its own expert arena, or
a serving loop that forbids cudaMalloc/cudaFree after start-up because those calls can stall
or synchronise the device in the middle of a step. Its scratch is a fixed array compiled
into the library. This file checks, through the C ABI, that two calls in a row give the
same result as the oracle's expert FFN (the plain SwiGLU definition in fp64 on the decoded
blob) and as the cached forward (ft_moe_forward) over a one-expert, top-1 layer, within the
tolerance the other parity tests use. It is collected last on purpose.
"""
import numpy as np
import pytest

import workloads as W
from oracle import formats, moe
from workloads.host import HostPool

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "mxfp4": 2e-2, "nvfp4": 2e-2}


@pytest.fixture(scope="module")
def ft():
    import torch
    from expert_cached_sparse_top_b300 import build
    build.build()
    from expert_cached_sparse_top_b300 import ftmoe
    ftmoe.lib()
    torch.cuda.init()
    return ftmoe


def _x(cfg, T, seed):
    bits = W.tiny_inputs(W.config("tiny", hidden=cfg.hidden, tokens=T, seed=seed))
    import torch
    return bits, torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("name,H,I", [("decode_bf16", 256, 128), ("decode_mxfp4", 512, 256),
                                      ("elastic_nvfp4", 2048, 768)])
def test_noalloc_matches_oracle_and_cached_forward_twice(ft, name, H, I):
    import torch
    cfg = W.config(name, layers=1, experts=1, top_k=1, hidden=H, inter=I)
    pool = HostPool(cfg)
    blob = torch.from_numpy(pool.arr[0].copy()).cuda()
    c = ft.make_config(1, 1, H, I, 1, 16, cfg.wfmt, 1)
    cache = ft.MoECache(c, pool.ptrs, None)
    w1, w3, w2 = formats.decode_blob(pool.blob(0), cfg.fmt, H, I)
    for call, T in enumerate((16, 7)):                  # two calls in a row
        bits, x = _x(cfg, T, seed=10 + call)
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        ft.expert_ffn_noalloc(blob, cfg.wfmt, H, I, x, T, y)
        out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        logits = torch.zeros((T, 1), dtype=torch.float32, device="cuda")
        cache.forward(0, x, T, out, logits=logits)       # top-1 of one expert: weight 1
        torch.cuda.synchronize()
        got = y.double().cpu().numpy()
        assert np.isfinite(got).all()
        want, _ = moe.expert_ffn(w1, w3, w2, formats.bf16_to_f64(bits))
        err_oracle = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert err_oracle <= TOL[cfg.wfmt], (call, err_oracle)
        ref = out.double().cpu().numpy()
        err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert err <= TOL[cfg.wfmt], (call, err)
    cache.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(ft):
    import torch
    L = ft.lib()
    blob = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    too_many = 1025                                          # FT_NOALLOC_MAX_TOKENS + 1
    assert L.ft_expert_ffn_noalloc(blob.data_ptr(), 0, 256, 128, x.data_ptr(), too_many,
                                   y.data_ptr(), None) == ft.FT_ERR_INVALID
    # activation larger than the scratch: 1024 tokens x 8192 features x 2 bytes = 16 MiB
    assert L.ft_expert_ffn_noalloc(blob.data_ptr(), 0, 256, 8192, x.data_ptr(), 1024,
                                   y.data_ptr(), None) == ft.FT_ERR_INVALID
    assert L.ft_expert_ffn_noalloc(blob.data_ptr(), 0, 256, 128, x.data_ptr(), 0,
                                   y.data_ptr(), None) == ft.FT_OK
