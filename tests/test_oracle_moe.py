"""Pins for the oracle's MoE layer definition (CPU only)."""
import itertools
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "moe_hand_example.txt")


def test_topk_brute_force():
    rng = np.random.default_rng(0)
    for E in range(1, 9):
        for k in range(1, E + 1):
            l = rng.standard_normal((5, E))
            idx = moe.topk(l, k)
            for t in range(5):
                best = max(itertools.combinations(range(E), k), key=lambda c: l[t, list(c)].sum())
                assert set(idx[t]) == set(best)
                vals = l[t, idx[t]]
                assert np.all(np.diff(vals) <= 0)      # rank order: descending


def test_topk_ties_go_to_lower_index():
    l = np.array([[1.0, 3.0, 3.0, 2.0], [0.5, 0.5, 0.5, 0.5], [2.0, -1.0, 2.0, 2.0]])
    assert moe.topk(l, 2).tolist() == [[1, 2], [0, 1], [0, 2]]
    assert moe.topk(l, 3).tolist()[2] == [0, 2, 3]


def test_topk_rejects_nan():
    with pytest.raises(ValueError):
        moe.topk(np.array([[0.0, np.nan]]), 1)


def test_gate_weights_closed_forms():
    rng = np.random.default_rng(1)
    l = rng.standard_normal((7, 16)) * 3
    for k in (1, 2, 6, 16):
        idx = moe.topk(l, k)
        w = moe.gate_weights(l, idx)
        assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
        ref = scipy.special.softmax(np.take_along_axis(l, idx, 1), axis=1)
        assert np.allclose(w, ref, rtol=1e-13, atol=0)
        if k == 1:
            assert np.all(w == 1.0)
    eq = np.zeros((3, 8))
    assert np.allclose(moe.gate_weights(eq, moe.topk(eq, 4)), 0.25)
    # full softmax then renormalisation over the chosen gives the same weights
    idx = moe.topk(l, 4)
    full = scipy.special.softmax(l, axis=1)
    ch = np.take_along_axis(full, idx, 1)
    assert np.allclose(moe.gate_weights(l, idx), ch / ch.sum(1, keepdims=True), rtol=1e-12)


def test_router_logits_vs_torch_linear():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((9, 64))
    wr = rng.standard_normal((12, 64)).astype(np.float32)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(wr.astype(np.float64))).numpy()
    assert np.allclose(moe.router_logits(x, wr), ref, rtol=1e-13, atol=1e-13)


def _rand_expert(rng, H, I):
    return (rng.standard_normal((I, H)) * 0.1, rng.standard_normal((I, H)) * 0.1,
            rng.standard_normal((H, I)) * 0.1)


def test_single_expert_is_plain_swiglu_mlp():
    rng = np.random.default_rng(3)
    H, I, T = 32, 24, 6
    w1, w3, w2 = _rand_expert(rng, H, I)
    x = rng.standard_normal((T, H))
    l = rng.standard_normal((T, 1))
    out, idx, w = moe.moe_forward(x, l, 1, lambda e: (w1, w3, w2))
    tx = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(tx @ torch.from_numpy(w1).T) * (tx @ torch.from_numpy(w3).T)) \
        @ torch.from_numpy(w2).T
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_k_equals_e_is_dense_weighted_sum():
    rng = np.random.default_rng(4)
    H, I, T, E = 16, 8, 5, 4
    experts = [_rand_expert(rng, H, I) for _ in range(E)]
    x = rng.standard_normal((T, H))
    l = rng.standard_normal((T, E))
    out, _, _ = moe.moe_forward(x, l, E, lambda e: experts[e])
    p = torch.softmax(torch.from_numpy(l), dim=1)
    tx = torch.from_numpy(x)
    ref = torch.zeros(T, H, dtype=torch.float64)
    for e, (w1, w3, w2) in enumerate(experts):
        ye = (torch.nn.functional.silu(tx @ torch.from_numpy(w1).T) * (tx @ torch.from_numpy(w3).T)) \
            @ torch.from_numpy(w2).T
        ref += p[:, e:e + 1] * ye
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def _golden_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rest = line.split(" ", 1)
        if key == "case":
            cur = {"name": rest}
            cases.append(cur)
        elif key == "router":
            cur["router"] = np.array([[float(v) for v in row.split()] for row in rest.split(";")])
        else:
            cur[key] = np.array([float(v) for v in rest.split()])
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_example(case):
    experts = {
        0: (np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]]), np.array([[1.0], [0.0]])),
        1: (np.array([[1.0, 1.0]]), np.array([[1.0, 1.0]]), np.array([[1.0], [1.0]])),
        2: (np.array([[0.0, 1.0]]), np.array([[1.0, 0.0]]), np.array([[0.0], [1.0]])),
    }
    x = np.array([[2.0, 1.0]])
    logits = moe.router_logits(x, case["router"].astype(np.float32))
    out, idx, w = moe.moe_forward(x, logits, 2, lambda e: experts[e])
    assert idx[0].tolist() == case["idx"].astype(int).tolist()
    assert np.allclose(w[0], case["w"], rtol=1e-15, atol=1e-16)
    assert np.allclose(out[0], case["out"], rtol=1e-15, atol=1e-15)


def test_plausible_mistakes_fail_a_pin():
    """Planted mistakes in a copy of the oracle's arithmetic must break the hand example."""
    case = _golden_cases()[1]
    x = np.array([[2.0, 1.0]])
    logits = moe.router_logits(x, case["router"].astype(np.float32))
    idx = moe.topk(logits, 2)
    w = moe.gate_weights(logits, idx)
    # wrong: sigmoid gate instead of softmax over chosen; W1/W3 swapped
    w_bad = 1 / (1 + np.exp(-np.take_along_axis(logits, idx, 1)))
    assert not np.allclose(w_bad, case["w"])
    e0 = (np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]]), np.array([[1.0], [0.0]]))
    y_ok, _ = moe.expert_ffn(*e0, x)
    y_swapped, _ = moe.expert_ffn(e0[1], e0[0], e0[2], x)
    assert not np.allclose(y_ok, y_swapped)


def test_bf16_round_matches_torch():
    import torch
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-6, 6, 5000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, -3.1415926]])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(moe.bf16_round(v), ref)
