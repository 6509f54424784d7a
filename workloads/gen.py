"""Seeded generators for the five workloads of the cached-expert MoE layer.

Every array is drawn from ``numpy.random.default_rng(SeedSequence([seed, tag, ...]))`` so
any (config, step, layer) can be regenerated on its own. Shapes and value distributions
follow the workload definitions; where they are not given, the choices made are stated
beside each generator below.
"""
import math
from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np

FMT_IDS = {"bf16": 0, "mxfp4": 1, "nvfp4": 2}

# Stream tags, so that draws for different purposes never share a generator.
_T_POOL, _T_ROUTER, _T_PERM, _T_TRACE, _T_X, _T_LEN, _T_PREFILL, _T_TINY, _T_PRED = range(1, 10)


def _rng(*tags):
    return np.random.default_rng(np.random.SeedSequence([int(t) for t in tags]))


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    layers: int
    experts: int
    hidden: int
    inter: int
    top_k: int
    wfmt: str
    seed: int
    steps: int = 1
    t_min: int = 1
    t_max: int = 1
    cache_frac: float = 1.0
    tokens: int = 0                     # fixed T (tiny, prefill)
    reuse: float = 0.6                  # step-to-step reuse probability (decode traces)
    zipf_s: float = 1.1
    resize: Tuple[Tuple[int, float], ...] = field(default_factory=tuple)
    logit_std: float = 0.5              # prefill router logits N(0, logit_std)
    x_corr: float = 0.0                 # chained decode: step-to-step correlation of a token's input

    @property
    def fmt(self):
        return FMT_IDS[self.wfmt]

    @property
    def keys(self):
        return self.layers * self.experts


CONFIGS = {
    # Tiny layer: all experts resident, router computed from x.
    "tiny": WorkloadConfig("tiny", 1, 8, 256, 128, 2, "bf16", seed=0, tokens=16,
                           cache_frac=1.0),
    # 35B-A3B-shaped decode layer, BF16, LRU at 37% of the pool, 1..16 tokens per step.
    "decode_bf16": WorkloadConfig("decode_bf16", 1, 128, 2048, 768, 8, "bf16", seed=2,
                                  steps=512, t_min=1, t_max=16, cache_frac=0.37),
    # 284B-shaped decode, 43 MoE layers, MXFP4, one global LRU at 20%, 1..8 tokens per step.
    "decode_mxfp4": WorkloadConfig("decode_mxfp4", 43, 256, 4096, 2048, 6, "mxfp4", seed=3,
                                   steps=256, t_min=1, t_max=8, cache_frac=0.20),
    # Prefill on the config-2 (35B-A3B-shaped) layer: 4096 tokens, logits N(0, 0.5).
    "prefill_bf16": WorkloadConfig("prefill_bf16", 4, 128, 2048, 768, 8, "bf16", seed=4,
                                   tokens=4096),
    # Prefill at the 256-expert top-6 shape (~96 tokens per expert), MXFP4.
    "prefill_mxfp4": WorkloadConfig("prefill_mxfp4", 4, 256, 4096, 2048, 6, "mxfp4", seed=4,
                                    tokens=4096),
    # Chained decode through 8 layers of the 35B-A3B shape (x_{l+1} = x_l + out_l), one global
    # LRU at 37% of the pool, 1..16 tokens per step: the layer-ahead prefetch workload.
    "decode_chained": WorkloadConfig("decode_chained", 8, 128, 2048, 768, 8, "bf16", seed=6,
                                     steps=128, t_min=1, t_max=16, cache_frac=0.37, x_corr=0.9),
    # Elastic NVFP4 decode, cache 40% -> 15% -> 30% at steps 0 / 341 / 682.
    "elastic_nvfp4": WorkloadConfig("elastic_nvfp4", 1, 128, 2048, 768, 8, "nvfp4", seed=5,
                                    steps=1024, t_min=1, t_max=16, cache_frac=0.40,
                                    resize=((341, 0.15), (682, 0.30))),
}


def config(name, **overrides):
    cfg = CONFIGS[name]
    if overrides:
        d = dict(cfg.__dict__)
        d.update(overrides)
        cfg = WorkloadConfig(**d)
    return cfg


def cache_capacity(cfg, frac=None):
    frac = cfg.cache_frac if frac is None else frac
    return int(math.floor(frac * cfg.layers * cfg.experts + 1e-9))


# ---------------------------------------------------------------------------------------
# bf16 bit patterns
# ---------------------------------------------------------------------------------------
def f32_to_bf16_bits(a):
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------------------
# Blob layout (the library's host layout of an expert; see include/ftmoe.h)
# ---------------------------------------------------------------------------------------
def _up(n, a=256):
    return (n + a - 1) // a * a


def blob_layout(fmt, H, I):
    """Section offsets {name: (offset, size)} and the blob size for one expert."""
    if fmt == 0:
        sizes = [("w13", 4 * I * H), ("w2", 2 * H * I)]
    else:
        B = 32 if fmt == 1 else 16
        sizes = [("w13", I * H), ("w2", H * I // 2),
                 ("w13_scale", _pad(2 * I, 128) * _pad(H // B, 4)),
                 ("w2_scale", _pad(H, 128) * _pad(I // B, 4))]
        if fmt == 2:
            sizes.append(("tensor_scale", 8))
    out, off = {}, 0
    for name, size in sizes:
        off = _up(off)
        out[name] = (off, size)
        off += size
    return out, _up(off)


def _pad(n, a):
    return (n + a - 1) // a * a


def scale_atoms(s):
    """[R][S] scale bytes -> the blob's scale-section bytes: 128-row x 4-block tiles of 512
    bytes (row band by row band, 4 blocks at a time), inside a tile byte
    (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4; padding is zero."""
    s = np.asarray(s, dtype=np.uint8)
    R, S = s.shape
    Rp, Sp = _pad(R, 128), _pad(S, 4)
    full = np.zeros((Rp, Sp), dtype=np.uint8)
    full[:R, :S] = s
    # [band][r1 (128//32)][r0 (32)][atom][j (4)] -> [band][atom][r0][r1][j]
    t = full.reshape(Rp // 128, 4, 32, Sp // 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(-1)


def _interleave_rows(w1, w3):
    rows, cols = w1.shape
    out = np.empty((2 * rows, cols), dtype=w1.dtype)
    out[0::2] = w1
    out[1::2] = w3
    return out


def pack_blob_bf16(w1_bits, w3_bits, w2_bits):
    """bf16 bit arrays W1 [I][H], W3 [I][H], W2 [H][I] -> one blob (uint8 array)."""
    I, H = w1_bits.shape
    secs, total = blob_layout(0, H, I)
    blob = np.zeros(total, dtype=np.uint8)
    w13 = _interleave_rows(w1_bits, w3_bits).astype(np.uint16)
    off, size = secs["w13"]
    blob[off:off + size] = w13.reshape(-1).view(np.uint8)
    off, size = secs["w2"]
    blob[off:off + size] = np.ascontiguousarray(w2_bits, dtype=np.uint16).reshape(-1).view(np.uint8)
    return blob


def _pack_nibbles(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def pack_blob_fp4(fmt, c1, c3, c2, s1, s3, s2, tensor_scales=None):
    """FP4 codes (one code 0..15 per element) and scale bytes -> one blob.

    c1, c3: [I][H] codes; c2: [H][I] codes; s1, s3: [I][H/B] scale bytes; s2: [H][I/B]
    (B = 32 for MXFP4, 16 for NVFP4); tensor_scales: (t13, t2) fp32 for NVFP4.
    """
    I, H = c1.shape
    secs, total = blob_layout(fmt, H, I)
    blob = np.zeros(total, dtype=np.uint8)

    def put(name, arr):
        off, size = secs[name]
        flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
        assert flat.size == size, (name, flat.size, size)
        blob[off:off + size] = flat

    put("w13", _pack_nibbles(_interleave_rows(c1, c3)))
    put("w2", _pack_nibbles(c2))
    put("w13_scale", scale_atoms(_interleave_rows(s1, s3)))
    put("w2_scale", scale_atoms(s2))
    if fmt == 2:
        put("tensor_scale", np.asarray(tensor_scales, dtype=np.float32))
    return blob


# ---------------------------------------------------------------------------------------
# Expert pool
# ---------------------------------------------------------------------------------------
# FP4 code distribution: magnitudes of block-quantised N(0, sigma) weights concentrate on
# the middle of the E2M1 grid; the shape below (magnitude codes 0..7) is the recipe's
# stand-in for quantised Gaussians. Sign is symmetric.
_MAG_P = np.array([0.06, 0.08, 0.15, 0.15, 0.15, 0.22, 0.12, 0.07])


def _code_lut():
    counts = np.round(_MAG_P * 128).astype(int)
    counts[-1] += 128 - counts.sum()
    mags = np.repeat(np.arange(8, dtype=np.uint8), counts)
    return np.concatenate([mags, mags | 8]).astype(np.uint8)   # 256 entries


_CODE_LUT = _code_lut()


def _fp4_codes(rng, shape):
    return _CODE_LUT[rng.integers(0, 256, size=shape, dtype=np.uint8)]


def _blob_for_image(cfg, image):
    rng = _rng(cfg.seed, _T_POOL, image)
    H, I, fmt = cfg.hidden, cfg.inter, cfg.fmt
    if fmt == 0:
        w1 = f32_to_bf16_bits(rng.standard_normal((I, H), dtype=np.float32) * np.float32(0.02))
        w3 = f32_to_bf16_bits(rng.standard_normal((I, H), dtype=np.float32) * np.float32(0.02))
        w2 = f32_to_bf16_bits(rng.standard_normal((H, I), dtype=np.float32) * np.float32(0.02))
        return pack_blob_bf16(w1, w3, w2)
    c1, c3 = _fp4_codes(rng, (I, H)), _fp4_codes(rng, (I, H))
    c2 = _fp4_codes(rng, (H, I))
    if fmt == 1:
        # E8M0 bytes 119..121: block scales 2^-8 .. 2^-6 (sigma 0.02 weights)
        s1 = rng.integers(119, 122, size=(I, H // 32), dtype=np.uint8)
        s3 = rng.integers(119, 122, size=(I, H // 32), dtype=np.uint8)
        s2 = rng.integers(119, 122, size=(H, I // 32), dtype=np.uint8)
        return pack_blob_fp4(fmt, c1, c3, c2, s1, s3, s2)
    # NVFP4: E4M3 block scales with exponent field 12..14 (32 .. 240), fp32 tensor scale
    def e4m3(shape):
        e = rng.integers(12, 15, size=shape, dtype=np.uint8)
        m = rng.integers(0, 8, size=shape, dtype=np.uint8)
        return ((e << 3) | m).astype(np.uint8)
    s1, s3, s2 = e4m3((I, H // 16)), e4m3((I, H // 16)), e4m3((H, I // 16))
    ts = (np.float32(8.0e-5) * (1 + np.float32(0.25) * rng.random(2, dtype=np.float32)))
    return pack_blob_fp4(fmt, c1, c3, c2, s1, s3, s2, ts.astype(np.float32))


def expert_pool(cfg, images=None, out=None):
    """Distinct expert blobs [P][blob_bytes] (uint8). Key (layer*E + e) uses image key % P.

    ``images`` defaults to the whole pool (layers * experts). A smaller P aliases the
    physical blobs; the keys, the cache and the PCIe bytes are unchanged. ``out`` may be a
    preallocated (e.g. pinned) uint8 array of the right shape.
    """
    P = cfg.keys if images is None else int(images)
    _, bb = blob_layout(cfg.fmt, cfg.hidden, cfg.inter)
    pool = np.empty((P, bb), dtype=np.uint8) if out is None else out
    assert pool.shape == (P, bb)
    for p in range(P):
        pool[p] = _blob_for_image(cfg, p)
    return pool


def router_weights(cfg, layers=None):
    """Router matrices [L][E][H] fp32, N(0, 0.02)."""
    L = cfg.layers if layers is None else layers
    rng = _rng(cfg.seed, _T_ROUTER)
    return (rng.standard_normal((L, cfg.experts, cfg.hidden), dtype=np.float32)
            * np.float32(0.02))


# ---------------------------------------------------------------------------------------
# Decode traces
# ---------------------------------------------------------------------------------------
def _zipf_p(E, s):
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** -s
    return p / p.sum()


class DecodeTrace:
    """Sequential generator of decode steps: per step a token count T, then for each layer
    the token activations x [T][H] (bf16 bits), router logits [T][E] (fp32) whose top-k
    are exactly the generator's picks, and the picks themselves.

    Picks: with probability ``reuse`` a pick is drawn uniformly from the previous step's
    union of selected experts for that layer (not yet picked for this token); otherwise a
    popularity rank r ~ Zipf(s) truncated to [1, E] names expert perm_l[r-1]; duplicates
    are redrawn. Logits: chosen experts get 3 + U(0,1), the rest N(0, 0.5) clipped to 2.5.
    """

    def __init__(self, cfg):
        self.cfg = cfg
        self.perm = [_rng(cfg.seed, _T_PERM, l).permutation(cfg.experts)
                     for l in range(cfg.layers)]
        self.prev_union = [np.zeros(0, dtype=np.int64) for _ in range(cfg.layers)]
        self.zipf_p = _zipf_p(cfg.experts, cfg.zipf_s)
        self.step = 0

    def tokens(self, step):
        cfg = self.cfg
        if cfg.t_min == cfg.t_max:
            return cfg.t_min
        return int(_rng(cfg.seed, _T_LEN, step).integers(cfg.t_min, cfg.t_max + 1))

    def layer(self, step, layer, T):
        cfg = self.cfg
        E, k, H = cfg.experts, cfg.top_k, cfg.hidden
        rng = _rng(cfg.seed, _T_TRACE, step, layer)
        prev = self.prev_union[layer]
        picks = np.empty((T, k), dtype=np.int32)
        for t in range(T):
            chosen = []
            while len(chosen) < k:
                avail = [e for e in prev if e not in chosen] if len(prev) else []
                if avail and rng.random() < cfg.reuse:
                    e = int(avail[rng.integers(0, len(avail))])
                else:
                    r = int(rng.choice(E, p=self.zipf_p))
                    e = int(self.perm[layer][r])
                if e not in chosen:
                    chosen.append(e)
            picks[t] = chosen
        logits = np.clip(rng.normal(0.0, 0.5, size=(T, E)), None, 2.5).astype(np.float32)
        chosen_vals = (3.0 + rng.random((T, k))).astype(np.float32)
        np.put_along_axis(logits, picks.astype(np.int64), chosen_vals, axis=1)
        xr = _rng(cfg.seed, _T_X, step, layer)
        x = f32_to_bf16_bits(xr.standard_normal((T, H), dtype=np.float32))
        self.prev_union[layer] = np.unique(picks).astype(np.int64)
        return dict(step=step, layer=layer, T=T, x=x, logits=logits, picks=picks)

    def __iter__(self):
        return self

    def __next__(self):
        """Yields one step: list over layers of the per-layer dicts."""
        if self.step >= self.cfg.steps:
            raise StopIteration
        s = self.step
        T = self.tokens(s)
        out = [self.layer(s, l, T) for l in range(self.cfg.layers)]
        self.step += 1
        return out


def decode_trace(cfg, steps=None):
    if steps is not None:
        cfg = WorkloadConfig(**{**cfg.__dict__, "steps": int(steps)})
    return DecodeTrace(cfg)


def trace_step(cfg, step, layer, T):
    """Stand-alone draw of one (step, layer) with no reuse history (tests of a single call)."""
    return DecodeTrace(cfg).layer(step, layer, T)


def chained_inputs(cfg, steps):
    """First-layer inputs of a chained decode, one [T][H] bf16 array per step. Token slot i
    follows an AR(1) process across steps, s_t = c s_{t-1} + sqrt(1 - c^2) e_t with
    c = cfg.x_corr and e_t ~ N(0, 1) (a decoding sequence's hidden state drifts from one step
    to the next, so its routing repeats in part); step t uses the first T_t slots."""
    c = float(cfg.x_corr)
    state = _rng(cfg.seed, _T_X, 0).standard_normal((cfg.t_max, cfg.hidden), dtype=np.float32)
    out = []
    for step in range(steps):
        if step:
            e = _rng(cfg.seed, _T_X, step).standard_normal((cfg.t_max, cfg.hidden), dtype=np.float32)
            state = np.float32(c) * state + np.float32(math.sqrt(max(0.0, 1.0 - c * c))) * e
        T = DecodeTrace(cfg).tokens(step)
        out.append(f32_to_bf16_bits(state[:T]))
    return out


def predicted_picks(cfg, step, layer, picks, accuracy):
    """A stand-in for a predictor of ``layer``'s routing at ``step``: each of the layer's true
    picks [T][k] is kept with probability ``accuracy`` and otherwise replaced by a uniformly
    drawn expert (duplicates possible). Returns int32 [T * k]."""
    rng = _rng(cfg.seed, _T_PRED, step, layer)
    p = np.asarray(picks, dtype=np.int32).reshape(-1).copy()
    swap = rng.random(p.size) >= accuracy
    p[swap] = rng.integers(0, cfg.experts, size=int(swap.sum()))
    return p


def tiny_inputs(cfg):
    """Tiny layer: x [T][H] bf16 bits ~N(0,1) (the router is router_weights(cfg))."""
    rng = _rng(cfg.seed, _T_TINY)
    return f32_to_bf16_bits(rng.standard_normal((cfg.tokens, cfg.hidden), dtype=np.float32))


def prefill_inputs(cfg, layer, tokens=None):
    """Prefill: x [T][H] bf16 bits ~N(0,1) and near-uniform logits N(0, logit_std) fp32."""
    T = cfg.tokens if tokens is None else tokens
    rng = _rng(cfg.seed, _T_PREFILL, layer)
    x = f32_to_bf16_bits(rng.standard_normal((T, cfg.hidden), dtype=np.float32))
    logits = (rng.standard_normal((T, cfg.experts), dtype=np.float32)
              * np.float32(cfg.logit_std))
    return x, logits
