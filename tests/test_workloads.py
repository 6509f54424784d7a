"""The seeded input generators (shared by the oracle and the CUDA path): reproducible draws,
decode logits whose top-k is exactly the generator's picks (with a margin), token counts in
range, step-to-step expert reuse, and the aliased host pool."""
import numpy as np

import workloads as W
from workloads.host import HostPool


def _steps(cfg, n):
    return list(W.decode_trace(cfg, steps=n))


def test_decode_trace_is_reproducible():
    cfg = W.config("decode_mxfp4", layers=3, hidden=64, inter=64)
    a, b = _steps(cfg, 5), _steps(cfg, 5)
    for sa, sb in zip(a, b):
        for da, db in zip(sa, sb):
            assert da["T"] == db["T"]
            assert np.array_equal(da["x"], db["x"])
            assert np.array_equal(da["logits"], db["logits"])
            assert np.array_equal(da["picks"], db["picks"])
    # a single (step, layer) draw does not depend on the rest of the trace for x
    one = W.trace_step(cfg, 3, 1, a[3][1]["T"])
    assert np.array_equal(one["x"], a[3][1]["x"])


def test_picks_are_exactly_the_top_k_with_a_margin():
    for name in ("decode_bf16", "decode_mxfp4", "elastic_nvfp4"):
        cfg = W.config(name, layers=min(2, W.config(name).layers), hidden=64, inter=64)
        for step in _steps(cfg, 8):
            for d in step:
                lg, picks = d["logits"], d["picks"]
                k = cfg.top_k
                assert picks.shape == (d["T"], k)
                order = np.argsort(-lg, axis=1, kind="stable")
                for t in range(d["T"]):
                    assert len(set(picks[t].tolist())) == k                  # distinct
                    assert set(order[t, :k].tolist()) == set(picks[t].tolist())
                    srt = np.sort(lg[t])[::-1]
                    assert srt[k - 1] - srt[k] >= 0.5                         # 3 + U vs <= 2.5


def test_token_counts_and_reuse():
    cfg = W.config("decode_bf16", hidden=64, inter=64)
    steps = _steps(cfg, 64)
    Ts = [s[0]["T"] for s in steps]
    assert min(Ts) >= cfg.t_min and max(Ts) <= cfg.t_max and len(set(Ts)) > 4
    reused, total = 0, 0
    for prev, cur in zip(steps, steps[1:]):
        pu = set(np.unique(prev[0]["picks"]).tolist())
        for e in cur[0]["picks"].reshape(-1):
            reused += int(e) in pu
            total += 1
    assert 0.5 <= reused / total <= 0.95       # reuse 0.6 plus Zipf overlap


def test_prefill_inputs_are_reproducible():
    cfg = W.config("prefill_bf16", hidden=64, inter=64)
    x1, l1 = W.prefill_inputs(cfg, 2, tokens=32)
    x2, l2 = W.prefill_inputs(cfg, 2, tokens=32)
    assert np.array_equal(x1, x2) and np.array_equal(l1, l2)
    assert x1.shape == (32, 64) and l1.shape == (32, cfg.experts)
    x3, _ = W.prefill_inputs(cfg, 3, tokens=32)
    assert not np.array_equal(x1, x3)


def test_aliased_pool_keeps_keys_distinct_in_address_only():
    cfg = W.config("decode_mxfp4", layers=2, hidden=256, inter=256)
    pool = HostPool(cfg, images=3, pinned=False)
    assert len(pool.ptrs) == cfg.keys
    assert pool.image_of(0) == pool.image_of(3) and pool.image_of(0) != pool.image_of(1)
    assert bytes(pool.blob(0)) == bytes(pool.blob(3))
    assert bytes(pool.blob(0)) != bytes(pool.blob(1))


def test_chained_inputs_and_predicted_picks():
    import numpy as np
    from oracle import formats
    cfg = W.config("decode_chained")
    a = W.chained_inputs(cfg, 6)
    b = W.chained_inputs(cfg, 6)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))             # seeded
    assert all(1 <= x.shape[0] <= 16 and x.shape[1] == cfg.hidden for x in a)
    x0, x1 = formats.bf16_to_f64(a[0]), formats.bf16_to_f64(a[1])
    n = min(x0.shape[0], x1.shape[0])
    r = np.corrcoef(x0[:n].ravel(), x1[:n].ravel())[0, 1]
    assert abs(r - cfg.x_corr) < 0.05                                  # AR(1) correlation
    picks = np.arange(64, dtype=np.int32).reshape(8, 8) % cfg.experts
    p1 = W.predicted_picks(cfg, 3, 2, picks, 1.0)
    assert np.array_equal(p1, picks.reshape(-1))
    p2 = W.predicted_picks(cfg, 3, 2, picks, 0.5)
    kept = (p2 == picks.reshape(-1)).mean()
    assert 0.3 < kept < 0.8 and p2.min() >= 0 and p2.max() < cfg.experts
