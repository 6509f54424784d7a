"""Weight formats and the per-expert blob layout, decoded exactly into fp64.

The pages name three weight precisions for the served models: BF16 (35B-A3B on the RTX
5090), MXFP4 (DeepSeek-V4-Flash) and NVFP4 (35B on the 8 GB laptop GPU) ([MTP] §Results;
[LN]). They also say each expert is laid out in host memory once, in the form that is
copied to the GPU, and that memory is page-locked ([MTP] §Three mechanisms, elastic
memory management). The pages do not print a layout; the one decoded here is this
library's own host layout (one contiguous blob per expert, so that one DMA fills one cache
slot):

    section            BF16               MXFP4                 NVFP4
    s0  W13            [2I][H] bf16       [2I][H/2] E2M1 x2     [2I][H/2] E2M1 x2
    s1  W2             [H][I]  bf16       [H][I/2]  E2M1 x2     [H][I/2]  E2M1 x2
    s2  W13 scales     -                  SF(2I, H/32) E8M0     SF(2I, H/16) E4M3
    s3  W2 scales      -                  SF(H, I/32)  E8M0     SF(H, I/16)  E4M3
    s4  tensor scales  -                  -                     fp32 [2] (W13, W2)

* SF(R, S) holds the scale of row r, block j (j < S) in tiles ("atoms") of 128 rows x 4
  blocks, 512 bytes each: R and S are padded to multiples of 128 and 4 (padding bytes are
  zero), atoms follow each other 4 blocks at a time along a row band, then band after band,
  and inside an atom the byte of (r, j) sits at (r mod 32) * 16 + ((r mod 128) div 32) * 4
  + (j mod 4). This is the order in which the block-scaled tensor-core MMA takes its scale
  factors, so a cache slot can feed them to it without any rearrangement.

* Row 2i of W13 is W1 row i (gate projection), row 2i+1 is W3 row i (up projection).
* W1, W3 are [I][H] and W2 is [H][I] (out x in, so y = W2 a).
* Two E2M1 codes per byte; the LOW nibble holds the even-indexed element.
* Each section starts on a 256-byte boundary; the blob size is rounded up to 256 bytes.

Decoding definitions (OCP Microscaling formats v1.0, the standard the MXFP4/NVFP4 names
refer to):

* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0. Exponent 0 is subnormal:
  value = m * 0.5. Otherwise value = (1 + m/2) * 2^(e-1). No inf/NaN.
* E8M0: value = 2^(s-127); s = 255 is NaN.
* E4M3 (the "fn" variant): sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
  subnormal m/8 * 2^-6; exponent 15 with mantissa 7 is NaN; no inf.

Pins (tests/test_oracle_formats.py): all 256 E8M0 values and all 256 E4M3 values against
torch's float8_e8m0fnu / float8_e4m3fn conversions (library routines); E2M1 via a generic
minifloat decoder that is itself checked against torch's E4M3 and E5M2 conversions; blob
parsing against blobs assembled byte by byte in the test.
"""
import numpy as np

FMT_BF16, FMT_MXFP4, FMT_NVFP4 = 0, 1, 2
FMT_NAMES = {FMT_BF16: "bf16", FMT_MXFP4: "mxfp4", FMT_NVFP4: "nvfp4"}
_ALIGN = 256


def _round_up(n, a=_ALIGN):
    return (n + a - 1) // a * a


def e2m1_value(code):
    """Value of one 4-bit E2M1 code (scalar, exact)."""
    code = int(code)
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        v = 0.5 * m
    else:
        v = (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -v if s else v


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def e8m0_value(byte):
    """Value of one E8M0 scale byte: 2^(s-127); 255 is NaN."""
    byte = int(byte)
    if byte == 255:
        return float("nan")
    return 2.0 ** (byte - 127)


E8M0_TABLE = np.array([e8m0_value(b) for b in range(256)], dtype=np.float64)


def e4m3_value(byte):
    """Value of one E4M3 (fn) byte; exponent 15 with mantissa 7 is NaN, there is no inf."""
    byte = int(byte)
    s = (byte >> 7) & 1
    e = (byte >> 3) & 15
    m = byte & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        v = (m / 8.0) * 2.0 ** -6
    else:
        v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -v if s else v


E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def bf16_to_f64(u16):
    """bf16 bit patterns (uint16 array) -> fp64 values (exact: bf16 is the top half of fp32)."""
    u16 = np.asarray(u16, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (u16.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def unpack_e2m1(packed, k):
    """[rows][k/2] bytes -> [rows][k] codes; low nibble = even element."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows = packed.shape[0]
    codes = np.empty((rows, k), dtype=np.uint8)
    codes[:, 0::2] = packed & 0x0F
    codes[:, 1::2] = packed >> 4
    return codes


def sf_padded(rows, blocks):
    """Padded (rows, blocks) of a scale section: multiples of 128 and 4."""
    return (rows + 127) // 128 * 128, (blocks + 3) // 4 * 4


def sf_offset(r, j, blocks):
    """Byte offset of the scale of row r, block j in a scale section with `blocks` blocks
    per row (before padding). Works elementwise on integer arrays."""
    s_pad = (blocks + 3) // 4 * 4
    atom = (r // 128) * (s_pad // 4) + j // 4
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4


def blob_sections(fmt, hidden, inter):
    """Byte offsets and sizes of the sections of one expert blob, and the blob size."""
    H, I = hidden, inter
    if H % 64 or I % 64:
        raise ValueError("hidden and inter must be multiples of 64")
    secs = {}
    off = 0
    if fmt == FMT_BF16:
        sizes = [("w13", 2 * I * H * 2), ("w2", H * I * 2)]
    elif fmt in (FMT_MXFP4, FMT_NVFP4):
        B = 32 if fmt == FMT_MXFP4 else 16
        r13, s13 = sf_padded(2 * I, H // B)
        r2, s2 = sf_padded(H, I // B)
        sizes = [("w13", 2 * I * H // 2), ("w2", H * I // 2),
                 ("w13_scale", r13 * s13), ("w2_scale", r2 * s2)]
        if fmt == FMT_NVFP4:
            sizes.append(("tensor_scale", 8))
    else:
        raise ValueError("unknown format %r" % (fmt,))
    for name, size in sizes:
        off = _round_up(off)
        secs[name] = (off, size)
        off += size
    return secs, _round_up(off)


def blob_bytes(fmt, hidden, inter):
    return blob_sections(fmt, hidden, inter)[1]


def read_scales(section, rows, blocks):
    """Scale section (atom order) -> [rows][blocks] bytes."""
    r = np.arange(rows)[:, None]
    j = np.arange(blocks)[None, :]
    return np.asarray(section, dtype=np.uint8)[sf_offset(r, j, blocks)]


def _dequant_fp4(codes_packed, scales, rows, k, fmt, tensor_scale):
    codes = unpack_e2m1(codes_packed.reshape(rows, k // 2), k)
    vals = E2M1_TABLE[codes]
    if fmt == FMT_MXFP4:
        s = E8M0_TABLE[read_scales(scales, rows, k // 32)]
        vals = vals * np.repeat(s, 32, axis=1)
    else:
        s = E4M3_TABLE[read_scales(scales, rows, k // 16)]
        vals = vals * np.repeat(s, 16, axis=1) * tensor_scale
    return vals


def decode_blob(blob, fmt, hidden, inter):
    """One expert blob (bytes / uint8 array) -> (W1 [I][H], W3 [I][H], W2 [H][I]) in fp64."""
    H, I = hidden, inter
    b = np.frombuffer(bytes(blob), dtype=np.uint8) if not isinstance(blob, np.ndarray) else blob
    b = np.asarray(b, dtype=np.uint8).reshape(-1)
    secs, total = blob_sections(fmt, H, I)
    if b.size < total:
        raise ValueError("blob too short: %d < %d" % (b.size, total))

    def sec(name):
        off, size = secs[name]
        return b[off:off + size]

    if fmt == FMT_BF16:
        w13 = bf16_to_f64(sec("w13").view(np.uint16).reshape(2 * I, H))
        w2 = bf16_to_f64(sec("w2").view(np.uint16).reshape(H, I))
    else:
        if fmt == FMT_NVFP4:
            ts = sec("tensor_scale").view(np.float32).astype(np.float64)
            t13, t2 = float(ts[0]), float(ts[1])
        else:
            t13 = t2 = 1.0
        w13 = _dequant_fp4(sec("w13"), sec("w13_scale"), 2 * I, H, fmt, t13)
        w2 = _dequant_fp4(sec("w2"), sec("w2_scale"), H, I, fmt, t2)
    w1 = w13[0::2]
    w3 = w13[1::2]
    return w1, w3, w2
