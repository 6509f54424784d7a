"""The routed MoE layer forward, written out as its plain definition in fp64.

What the method computes: the pages state that the cached-expert engine returns exactly the
model's own MoE output: the router is left as it is, no expert is replaced by another and no
step runs at reduced precision ([MTP] §Key Takeaways); the parts of a step computed on the GPU
and on the CPU are summed without approximation ([MTP] §Three mechanisms, q* policy). So the
oracle is the plain routed-MoE definition, independent of where an expert lives:

1. router logits      l[t,e] = sum_h x[t,h] * Wr[e,h]                  (x is bf16, Wr fp32)
2. top-k              the k experts with the largest logits, in rank order
                      (logit descending, ties to the LOWER expert index: the pages are
                      silent on ties, this is the reading taken)
3. gate weights       softmax over the k chosen logits (renormalised over the chosen)
4. expert FFN         SwiGLU: g = W1 x, u = W3 x, a = silu(g) * u, y = W2 a
5. combine            out[t] = sum_{j<k} w[t,j] * y[t,j], summed in j order

The per-expert weights come from ``formats.decode_blob``. Everything is fp64; the GPU keeps
fp32 accumulators, stores a in bf16 and out in bf16, which the parity tolerance covers.

Pins (tests/test_oracle_moe.py): top-k against brute force over all C(E,k) subsets on tiny
inputs and crafted ties; gate weights against the closed forms (k=1 gives 1, equal logits
give 1/k) and the sum-to-one invariant; the FFN at E=1, k=1 against
torch.nn.functional.silu-based SwiGLU in fp64 (library routine); k=E with all experts
equal to the dense weighted sum; a hand-worked 3-expert example (tests/golden/); bf16
rounding against torch's bfloat16.
"""
import numpy as np

from . import formats


def router_logits(x_f64, wr_f32):
    """Step 1. x [T][H] (already exact fp64 of the bf16 input), Wr [E][H] fp32 -> [T][E]."""
    x = np.asarray(x_f64, dtype=np.float64)
    wr = np.asarray(wr_f32, dtype=np.float64)
    return x @ wr.T


def topk(logits, k):
    """Step 2. [T][E] logits -> idx [T][k] (int32, rank order).

    Order is (logit descending, expert index ascending); a stable sort on -logit keeps
    equal logits in ascending index order.
    """
    l = np.asarray(logits, dtype=np.float64)
    if np.isnan(l).any():
        raise ValueError("NaN router logit: precondition violated")
    if not 1 <= k <= l.shape[1]:
        raise ValueError("k out of range")
    order = np.argsort(-l, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gate_weights(logits, idx):
    """Step 3. softmax over the chosen logits (max-subtracted), per token."""
    l = np.asarray(logits, dtype=np.float64)
    chosen = np.take_along_axis(l, np.asarray(idx, dtype=np.int64), axis=1)
    m = chosen.max(axis=1, keepdims=True)
    e = np.exp(chosen - m)
    return e / e.sum(axis=1, keepdims=True)


def silu(g):
    return g / (1.0 + np.exp(-g))


def expert_ffn(w1, w3, w2, x):
    """Step 4. x [n][H] -> y [n][H]; also returns the SwiGLU activation a [n][I]."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ w1.T
    u = x @ w3.T
    a = silu(g) * u
    return a @ w2.T, a


def bf16_round(v):
    """Round to the nearest bf16 value (ties to even), returned in fp64."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def combine(w, y):
    """Step 5. w [T][k], y [T][k][H] -> out [T][H], summed over j in ascending order."""
    T, k = w.shape
    out = np.zeros((T, y.shape[2]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y[:, j, :]
    return out


def layer_forward(x_f64, idx, w, expert_weights, ffn=None):
    """Steps 4-5 for given routing. expert_weights(e) -> (w1, w3, w2) fp64; ffn (default
    expert_ffn) maps (w1, w3, w2, x) to y or (y, a).

    Returns out [T][H] and y [T][k][H]. Each (token, rank) pair goes through its expert's
    FFN; where the expert's bytes came from (cache slot, staging, host) does not enter.
    """
    x = np.asarray(x_f64, dtype=np.float64)
    T, k = idx.shape
    H = x.shape[1]
    y = np.zeros((T, k, H), dtype=np.float64)
    for e in np.unique(idx):
        rows, cols = np.nonzero(idx == e)
        w1, w3, w2 = expert_weights(int(e))
        if ffn is None:
            ye, _ = expert_ffn(w1, w3, w2, x[rows])
        else:
            ye = ffn(w1, w3, w2, x[rows])
        y[rows, cols, :] = ye
    return combine(w, y), y


def moe_forward(x_f64, logits, k, expert_weights):
    """Steps 2-5 from given logits: returns (out, idx, w)."""
    idx = topk(logits, k)
    w = gate_weights(logits, idx)
    out, _ = layer_forward(x_f64, idx, w, expert_weights)
    return out, idx, w


def blob_expert_weights(blob_of, fmt, hidden, inter):
    """Adapter: expert id -> decoded (w1, w3, w2) from a blob getter."""
    def get(e):
        return formats.decode_blob(blob_of(e), fmt, hidden, inter)
    return get
