"""Oracle block decoders (fp64).  TEST INFRASTRUCTURE ONLY.

The pages name the formats and their bits per weight but print no layout:
  * PTQ1_0: ternary {-1, 0, +1}, "5 trits/byte", 1.75 bpw
    (Strata 4090 post, section 1 and the section 5.1 format table);
  * Q2_0: 2.25 bpw, the budget-neutral reference format (section 5.1);
  * Q3_K: 3.44 bpw (section 5.1);
  * FP4 experts with per-32 weight blocks (DeepSeek-V4.1-Flash 4xL20 field
    report, header and section 2: "single expert = 3 x 5120 x 2304 x 0.5 B");
  * an NVFP4 checkpoint of the model (the news digest): FP4 codes in blocks
    of 16 with an FP8 E4M3 scale each, the plainest reading of NVIDIA's
    published NVFP4 (the pages give no layout; no per-tensor scale here).
The block layouts decoded here are this library's specification of those
formats (one block per bpw figure: 56 B / 256, 18 B / 64, 110 B / 256,
17 B / 32, 9 B / 16).  Every value is exact in fp64, so decoding is exact.

Functions take an array of canonical blocks of shape (..., block_bytes) as
uint8 and return float64 weights of shape (..., block_weights).
"""
from __future__ import annotations

import numpy as np

TQ1, Q2_0, Q3_K, MXFP4, NVFP4 = 1, 2, 3, 4, 5
BLOCK = {TQ1: (256, 56), Q2_0: (64, 18), Q3_K: (256, 110), MXFP4: (32, 17), NVFP4: (16, 9)}


def fp16_to_f64(lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    """IEEE 754 binary16 (little-endian bytes lo, hi) to float64, written out:
    sign, 5-bit exponent with bias 15, 10-bit fraction, subnormals when the
    exponent field is 0, inf/NaN when it is 31."""
    bits = lo.astype(np.int64) | (hi.astype(np.int64) << 8)
    sign = (bits >> 15) & 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    mag = np.where(e == 0, f * 2.0 ** -24, (1.0 + f / 1024.0) * np.exp2(e.astype(np.float64) - 15.0))
    mag = np.where(e == 31, np.where(f == 0, np.inf, np.nan), mag)
    return np.where(sign == 1, -mag, mag)


def e2m1_to_f64(code: np.ndarray) -> np.ndarray:
    """OCP E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
    Exponent field 0 is subnormal: value = mantissa * 0.5."""
    c = code.astype(np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.exp2(e.astype(np.float64) - 1.0) * (1.0 + 0.5 * m))
    return np.where(s == 1, -mag, mag)


def ue8m0_to_f64(e: np.ndarray) -> np.ndarray:
    """UE8M0 scale byte: 2^(E - 127); 0xFF is NaN."""
    e = e.astype(np.int64)
    return np.where(e == 255, np.nan, np.exp2(e.astype(np.float64) - 127.0))


def e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
    mantissa; exponent field 0 is subnormal (mantissa / 8 x 2^-6); exponent
    15 with mantissa 7 is NaN (the format has no infinities)."""
    b = b.astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def dequant_nvfp4(blocks: np.ndarray) -> np.ndarray:
    """9-byte block of 16 weights: byte i (0..7) holds weight 2i in its low
    nibble and 2i+1 in its high nibble (E2M1); byte 8 is the E4M3 scale.
    w = e2m1(code) * e4m3(scale)."""
    b = blocks.astype(np.int64)
    codes = b[..., :8]
    nib = np.stack([codes & 0xF, (codes >> 4) & 0xF], axis=-1).reshape(*b.shape[:-1], 16)
    return e2m1_to_f64(nib) * e4m3_to_f64(b[..., 8])[..., None]


def dequant_mxfp4(blocks: np.ndarray) -> np.ndarray:
    """17-byte block of 32 weights: byte i (0..15) holds weight 2i in its low
    nibble and weight 2i+1 in its high nibble; byte 16 is the UE8M0 exponent E.
    w = e2m1(code) * 2^(E-127)."""
    b = blocks.astype(np.int64)
    codes = b[..., :16]
    nib = np.stack([codes & 0xF, (codes >> 4) & 0xF], axis=-1).reshape(*b.shape[:-1], 32)
    return e2m1_to_f64(nib) * ue8m0_to_f64(b[..., 16])[..., None]


def dequant_q2_0(blocks: np.ndarray) -> np.ndarray:
    """18-byte block of 64 weights: weight j has the 2-bit code q at bits
    2(j mod 4).. of byte j div 4; bytes 16..17 are d (fp16).  w = d * (2q - 3),
    i.e. d times one of {-3, -1, +1, +3}."""
    b = blocks.astype(np.int64)
    j = np.arange(64)
    q = (b[..., j // 4] >> (2 * (j % 4))) & 3
    d = fp16_to_f64(b[..., 16], b[..., 17])
    return d[..., None] * (2 * q - 3)


def tq1_digits(byte_values: np.ndarray, ndigits: int = 5) -> np.ndarray:
    """Base-3 digits of each byte, least significant first (digit r = byte // 3^r mod 3)."""
    v = byte_values.astype(np.int64)
    return np.stack([(v // 3 ** r) % 3 for r in range(ndigits)], axis=-1)


def dequant_tq1(blocks: np.ndarray) -> np.ndarray:
    """56-byte block of 256 ternary weights.  Bytes 0..50 each hold 5 weights as
    base-3 digits (weight 5i+r is digit r of byte i, digit = t + 1, least
    significant first); byte 51 holds weight 255 as a single digit; bytes
    52..53 are d (fp16); bytes 54..55 are zero padding.  w = d * t, t in {-1,0,1}."""
    b = blocks.astype(np.int64)
    t = tq1_digits(b[..., :51]).reshape(*b.shape[:-1], 255) - 1
    t255 = (b[..., 51] % 3)[..., None] - 1
    t = np.concatenate([t, t255], axis=-1)
    d = fp16_to_f64(b[..., 52], b[..., 53])
    return d[..., None] * t


def q3k_subscales(blocks: np.ndarray) -> np.ndarray:
    """Sixteen unsigned 6-bit sub-scales packed little-endian in bytes 96..107:
    s_j occupies bits 6j..6j+5 of that 96-bit string."""
    b = blocks.astype(np.int64)[..., 96:108]
    out = []
    for j in range(16):
        bit = 6 * j
        lo = b[..., bit // 8]
        hi = b[..., bit // 8 + 1] if bit // 8 + 1 < 12 else np.zeros_like(lo)
        out.append(((lo | (hi << 8)) >> (bit % 8)) & 63)
    return np.stack(out, axis=-1)


def dequant_q3k(blocks: np.ndarray) -> np.ndarray:
    """110-byte block of 256 weights: bytes 0..63 hold the low two bits of q
    (weight j: byte j div 4, bits 2(j mod 4)..), bytes 64..95 the high bit
    (weight j: byte 64 + j div 8, bit j mod 8), so q = lo + 4*hi in 0..7;
    bytes 96..107 the sixteen 6-bit sub-scales; bytes 108..109 d (fp16).
    Weight j belongs to sub-block j div 16:  w = d * s_(j div 16) * (q - 4)."""
    b = blocks.astype(np.int64)
    j = np.arange(256)
    lo = (b[..., j // 4] >> (2 * (j % 4))) & 3
    hi = (b[..., 64 + j // 8] >> (j % 8)) & 1
    q = lo + 4 * hi
    s = q3k_subscales(blocks)[..., j // 16]
    d = fp16_to_f64(b[..., 108], b[..., 109])
    return d[..., None] * s * (q - 4)


DECODERS = {TQ1: dequant_tq1, Q2_0: dequant_q2_0, Q3_K: dequant_q3k, MXFP4: dequant_mxfp4, NVFP4: dequant_nvfp4}


def dequant_matrix(fmt: int, packed: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Row-major matrix whose rows are consecutive canonical blocks along the
    input dimension -> float64 (rows, cols)."""
    bw, bb = BLOCK[fmt]
    assert cols % bw == 0
    nb = cols // bw
    blocks = np.asarray(packed, dtype=np.uint8).reshape(rows, nb, bb)
    return DECODERS[fmt](blocks).reshape(rows, cols)


def split_expert(fmt: int, packed: np.ndarray, hidden: int, inter: int):
    """Canonical expert bytes W1 | W3 | W2 -> three packed matrices."""
    bw, bb = BLOCK[fmt]
    n13 = inter * (hidden // bw) * bb
    n2 = hidden * (inter // bw) * bb
    p = np.asarray(packed, dtype=np.uint8)
    assert p.size == 2 * n13 + n2
    return p[:n13], p[n13:2 * n13], p[2 * n13:]


def dequant_expert(fmt: int, packed: np.ndarray, hidden: int, inter: int):
    """Exact fp64 W1 (inter x hidden), W3 (inter x hidden), W2 (hidden x inter)."""
    p1, p3, p2 = split_expert(fmt, packed, hidden, inter)
    return (dequant_matrix(fmt, p1, inter, hidden),
            dequant_matrix(fmt, p3, inter, hidden),
            dequant_matrix(fmt, p2, hidden, inter))
