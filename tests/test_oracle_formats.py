"""Pins for the oracle's number formats and blob parser (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import formats


def _generic_minifloat(code, ebits, mbits, bias, ieee_special):
    """Decode a sign/exponent/mantissa minifloat from its field definition.

    ieee_special: exponent all-ones is inf (mantissa 0) / NaN (e5m2 style). Otherwise only
    the 'fn' rule applies: all-ones exponent and all-ones mantissa is NaN (e4m3fn style),
    or no special values at all when ieee_special is None.
    """
    s = (code >> (ebits + mbits)) & 1
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    emax = (1 << ebits) - 1
    if ieee_special is True and e == emax:
        v = float("inf") if m == 0 else float("nan")
    elif ieee_special is False and e == emax and m == (1 << mbits) - 1:
        v = float("nan")
    elif e == 0:
        v = (m / (1 << mbits)) * 2.0 ** (1 - bias)
    else:
        v = (1 + m / (1 << mbits)) * 2.0 ** (e - bias)
    return -v if s else v


def _torch_decode(dtype, nbits=8):
    b = torch.arange(256, dtype=torch.uint8)
    return b.view(dtype).to(torch.float64).numpy()


def _same(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def test_generic_decoder_matches_torch_fp8():
    e4m3 = [_generic_minifloat(c, 4, 3, 7, False) for c in range(256)]
    e5m2 = [_generic_minifloat(c, 5, 2, 15, True) for c in range(256)]
    assert _same(e4m3, _torch_decode(torch.float8_e4m3fn))
    assert _same(e5m2, _torch_decode(torch.float8_e5m2))


def test_e2m1_table():
    generic = [_generic_minifloat(c, 2, 1, 1, None) for c in range(16)]
    assert _same(formats.E2M1_TABLE, generic)
    # the grid the MX spec lists: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives
    assert list(formats.E2M1_TABLE[:8]) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e8m0_table_vs_torch():
    assert _same(formats.E8M0_TABLE, _torch_decode(torch.float8_e8m0fnu))


def test_e4m3_table_vs_torch():
    assert _same(formats.E4M3_TABLE, _torch_decode(torch.float8_e4m3fn))


def test_bf16_vs_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(formats.bf16_to_f64(bits), ref)


H, I = 64, 64


def test_bf16_blob_parse_bytewise():
    secs, total = formats.blob_sections(formats.FMT_BF16, H, I)
    assert secs["w13"] == (0, 2 * I * H * 2) and secs["w2"][0] % 256 == 0
    rng = np.random.default_rng(0)
    w1 = rng.integers(-40, 40, size=(I, H)) / 8.0     # exactly representable in bf16
    w3 = rng.integers(-40, 40, size=(I, H)) / 16.0
    w2 = rng.integers(-40, 40, size=(H, I)) / 32.0
    blob = bytearray(total)

    def put_bf16(off, v):
        b = torch.tensor([v], dtype=torch.bfloat16).view(torch.int16).item() & 0xFFFF
        blob[off] = b & 0xFF
        blob[off + 1] = b >> 8

    base = secs["w13"][0]
    for i in range(I):
        for h in range(H):
            put_bf16(base + ((2 * i) * H + h) * 2, w1[i, h])
            put_bf16(base + ((2 * i + 1) * H + h) * 2, w3[i, h])
    base = secs["w2"][0]
    for h in range(H):
        for i in range(I):
            put_bf16(base + (h * I + i) * 2, w2[h, i])
    d1, d3, d2 = formats.decode_blob(bytes(blob), formats.FMT_BF16, H, I)
    assert np.array_equal(d1, w1) and np.array_equal(d3, w3) and np.array_equal(d2, w2)


@pytest.mark.parametrize("fmt", [formats.FMT_MXFP4, formats.FMT_NVFP4])
def test_fp4_blob_parse_bytewise(fmt):
    secs, total = formats.blob_sections(fmt, H, I)
    B = 32 if fmt == formats.FMT_MXFP4 else 16
    rng = np.random.default_rng(fmt)
    c1 = rng.integers(0, 16, size=(I, H))
    c3 = rng.integers(0, 16, size=(I, H))
    c2 = rng.integers(0, 16, size=(H, I))
    if fmt == formats.FMT_MXFP4:
        sb = lambda shape: rng.integers(100, 140, size=shape)
        sval = lambda b: 2.0 ** (int(b) - 127)
    else:
        sb = lambda shape: rng.integers(0, 0x7F, size=shape)       # finite E4M3 bytes
        sval = lambda b: torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()
    s1, s3, s2 = sb((I, H // B)), sb((I, H // B)), sb((H, I // B))
    t13, t2 = (0.75, 1.5) if fmt == formats.FMT_NVFP4 else (1.0, 1.0)
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    val = lambda c: (-1 if c & 8 else 1) * grid[c & 7]
    blob = bytearray(total)

    def put_codes(base, row, k, col, code):
        off = base + row * (k // 2) + col // 2
        if col % 2 == 0:
            blob[off] = (blob[off] & 0xF0) | code
        else:
            blob[off] = (blob[off] & 0x0F) | (code << 4)

    def put_scales(base, get, rows, blocks):
        # walk the section byte by byte: band, atom, r0 (32), r1 (4), j (4)
        pos = base
        for band in range((rows + 127) // 128):
            for atom in range((blocks + 3) // 4):
                for r0 in range(32):
                    for r1 in range(4):
                        for jj in range(4):
                            r, j = band * 128 + r1 * 32 + r0, atom * 4 + jj
                            if r < rows and j < blocks:
                                blob[pos] = get(r, j)
                            pos += 1

    for i in range(I):
        for h in range(H):
            put_codes(secs["w13"][0], 2 * i, H, h, c1[i, h])
            put_codes(secs["w13"][0], 2 * i + 1, H, h, c3[i, h])
    put_scales(secs["w13_scale"][0], lambda r, j: (s1 if r % 2 == 0 else s3)[r // 2, j], 2 * I, H // B)
    for h in range(H):
        for i in range(I):
            put_codes(secs["w2"][0], h, I, i, c2[h, i])
    put_scales(secs["w2_scale"][0], lambda r, j: s2[r, j], H, I // B)
    if fmt == formats.FMT_NVFP4:
        blob[secs["tensor_scale"][0]:secs["tensor_scale"][0] + 8] = np.array([t13, t2], np.float32).tobytes()
    d1, d3, d2 = formats.decode_blob(bytes(blob), fmt, H, I)
    for i in range(0, I, 7):
        for h in range(0, H, 5):
            assert d1[i, h] == val(c1[i, h]) * sval(s1[i, h // B]) * t13
            assert d3[i, h] == val(c3[i, h]) * sval(s3[i, h // B]) * t13
            assert d2[h, i] == val(c2[h, i]) * sval(s2[h, i // B]) * t2


def test_scale_atom_offsets_hand_traced():
    """Scale-section offsets worked out by hand for a section with 8 blocks per row (two
    atoms per 128-row band, 1024 bytes per band)."""
    cases = {(0, 0): 0, (0, 1): 1, (0, 3): 3, (1, 0): 16, (31, 2): 31 * 16 + 2,
             (32, 0): 4, (64, 1): 9, (127, 3): 31 * 16 + 12 + 3, (0, 4): 512, (5, 6): 512 + 80 + 2,
             (128, 0): 1024, (200, 5): 1024 + 512 + 8 * 16 + 2 * 4 + 1}
    for (r, j), off in cases.items():
        assert formats.sf_offset(r, j, 8) == off, (r, j)
    # padding: 6 blocks per row pad to 8, 130 rows pad to 256
    assert formats.sf_padded(130, 6) == (256, 8)
    assert formats.sf_offset(129, 5, 6) == 1024 + 512 + 16 + 1


def test_generator_blobs_roundtrip_through_oracle():
    """The generator's packer and the oracle's parser are separate code; they must agree."""
    import workloads as W
    cfg = W.config("tiny")
    pool = W.expert_pool(cfg, images=1)
    assert pool.shape[1] == formats.blob_bytes(cfg.fmt, cfg.hidden, cfg.inter)
    for name, hh, ii in (("decode_mxfp4", 128, 64), ("elastic_nvfp4", 128, 64),
                         ("decode_mxfp4", 64, 64), ("elastic_nvfp4", 320, 192)):
        c = W.config(name, hidden=hh, inter=ii)
        p = W.expert_pool(c, images=1)
        assert p.shape[1] == formats.blob_bytes(c.fmt, c.hidden, c.inter)
        w1, w3, w2 = formats.decode_blob(p[0], c.fmt, c.hidden, c.inter)
        assert np.isfinite(w1).all() and 0.005 < w1.std() < 0.08
