"""Plain, slow, fp64 CPU oracle of the orthogonally rotated 3-bit KV cache
(and its 2- and 4-bit variants).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The library (CUDA kernels and C ABI)
never calls it, and it shares no code with the library: it is the
specification written out step by step, with dense matrices where the library
uses butterflies.

Sources (page titles with the section they come from):
  [OMC]  "Orthogonally mixed 3-bit KV cache" (synthcore idea 1973):
         Mathematical statement (U = B H_d, SO(4) blocks, the symmetric
         quantiser with eps), Key formulas, Implementation notes (write path,
         read path, codes packed into bytes with only codes and scales kept,
         q1 = U q, y = U^T y1).
  [OIQ]  "Orthogonal Invariance in Activation Space: Fast Walsh-Hadamard
         Transforms for KV Quantization": section 3.1 (normalised H_d,
         self-inverse), 3.2 (random sign flip D before the FWHT, generated once
         and kept fixed), 3.3 (store / retrieve / attention), 3.4 (per-group
         scales, g = 32), 4.2 (record = scale header + packed data).
  [HFF]  "Hardware-Fused Fast Hadamard Transforms Enable Lossless 3-Bit
         KV-Cache Compression at 128K Context": 64-element sub-blocks with an
         FP8 scale header (3.125 bits per element).

Readings where the pages are silent or disagree (all written into the C
header of the library as well):
  * U = B . H_d . D: sign flip first, then the normalised Hadamard transform in
    natural (Sylvester) order, then the SO(4) blocks.
  * Each SO(4) block is the left-multiplication matrix of one unit quaternion
    and acts on the contiguous coordinates 4i..4i+3.
  * Seed -> parameters: SplitMix64; d sign draws first, then one point of S^3
    per block by Marsaglia's 1972 method.
  * Scale: s = (max|x| + eps)/3 in the block, rounded to nearest even into the
    scale's storage type (fp32, fp16 or FP8-E4M3, the last two saturating to
    their largest finite value); codes use the stored scale:
    c = clip(round_half_even(x/s_q), -3, 3), and c = 0 where s_q = 0.
  * Codes are 3-bit two's complement in a little-endian bit stream: element j
    of a vector at bits 3j..3j+2 of its 3d/8-byte code string.
  * The asymmetric variant of [HFF] (scale kind "e4m3zp"): per block an E4M3
    scale s = (max - min + eps)/(2^b - 1) and an E4M3 zero point z = min,
    stored as two bytes, and unsigned codes u = clip(round((x - z_q)/s_q), 0,
    2^b - 1); x_hat = s_q u + z_q.  The page's "FP8 scale and zero-point
    header" is taken as one byte each (3.25 bits per element at m = 64); its
    3.125-bit figure fits a single header byte and is not followed.
  * Other bit widths b = 2 and 4 ([OIQ] 3.3, 4.2 and 5.1 evaluate them; the
    quantiser of [OMC] Key formulas is written for any b): divisor and clip
    bound 2^(b-1) - 1, b-bit two's-complement codes in the same bit stream
    (element j at bits b*j..b*j+b-1), code strings of b*d/8 bytes.
  * Cache layout: see :class:`Layout`.
  * Attention: logits = (q1 . k1_hat) * sm_scale with sm_scale = 1/sqrt(d),
    softmax over positions [0, seq_len), output U^T y1 in fp32; an empty
    sequence gives a zero output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

MASK64 = (1 << 64) - 1
# "e4m3zp": the asymmetric variant of [HFF] -- an E4M3 scale byte and an
# E4M3 zero-point byte per block, unsigned codes (see quantize_asym)
SCALE_BYTES = {"f32": 4, "f16": 2, "e4m3": 1, "e4m3zp": 2}

# Device-status bits (the library's dev_status word uses the same meaning).
ST_BAD_SEQ = 1
ST_BAD_POS = 2
ST_BAD_PAGE = 4
ST_BAD_LEN = 8


# ---------------------------------------------------------------------------
# Seed -> rotation parameters
# ---------------------------------------------------------------------------
class SplitMix64:
    """SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): state += golden gamma,
    then the xor-shift/multiply finaliser.  Written out with Python integers."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)

    def uniform_pm1(self) -> float:
        """A uniform number in [-1, 1): the top 53 bits scaled to [0, 1), times
        2, minus 1 (all steps exact in fp64)."""
        return (self.next() >> 11) * (2.0 ** -53) * 2.0 - 1.0


def marsaglia_s3(rng: SplitMix64):
    """A uniform point on the unit sphere S^3 (a unit quaternion) by
    Marsaglia, "Choosing a point from the surface of a sphere", Ann. Math.
    Stat. 43 (1972): two pairs drawn uniformly in the open unit disk (pairs
    with s >= 1 or s == 0 are rejected), then
    (x1, x2, x3*sqrt((1-s1)/s2), x4*sqrt((1-s1)/s2))."""
    while True:
        x1, x2 = rng.uniform_pm1(), rng.uniform_pm1()
        s1 = x1 * x1 + x2 * x2
        if 0.0 < s1 < 1.0:
            break
    while True:
        x3, x4 = rng.uniform_pm1(), rng.uniform_pm1()
        s2 = x3 * x3 + x4 * x4
        if 0.0 < s2 < 1.0:
            break
    f = math.sqrt((1.0 - s1) / s2)
    return (x1, x2, x3 * f, x4 * f)


def rotation_params(d: int, seed: int, use_sign: bool = True, use_so4: bool = True):
    """(signs[d] in {+1,-1}, quats[d/4][4]) for a rotation seed.  [OIQ] 3.2:
    D is drawn once and kept as a fixed parameter; [OMC] Implementation notes:
    fixed random SO(4) rotations parameterised by normalised quaternions.
    The d sign draws come first (sign -1 when the top bit is set), then one
    quaternion per block; flags only decide whether the draws are used."""
    rng = SplitMix64(seed)
    signs = np.array([-1 if (rng.next() >> 63) else 1 for _ in range(d)], dtype=np.int8)
    quats = np.array([marsaglia_s3(rng) for _ in range(d // 4)], dtype=np.float64).reshape(d // 4, 4)
    if not use_sign:
        signs[:] = 1
    if not use_so4:
        quats[:] = (1.0, 0.0, 0.0, 0.0)
    return signs, quats


def rotation_params_pair(d: int, seed: int, use_sign: bool = True):
    """(signs, quats, quats_r) of the two-quaternion rotation: the draws of
    :func:`rotation_params` (signs, then the left quaternion p_i of every
    block), followed by one more point of S^3 per block, the right quaternion
    q_i of R_i = L(p_i) R(conj q_i)."""
    rng = SplitMix64(seed)
    signs = np.array([-1 if (rng.next() >> 63) else 1 for _ in range(d)], dtype=np.int8)
    quats = np.array([marsaglia_s3(rng) for _ in range(d // 4)], dtype=np.float64).reshape(d // 4, 4)
    quats_r = np.array([marsaglia_s3(rng) for _ in range(d // 4)], dtype=np.float64).reshape(d // 4, 4)
    if not use_sign:
        signs[:] = 1
    return signs, quats, quats_r


# ---------------------------------------------------------------------------
# The orthogonal transform U = B . H_d . D
# ---------------------------------------------------------------------------
def hadamard_matrix(d: int) -> np.ndarray:
    """Normalised Walsh-Hadamard matrix in natural (Sylvester) order,
    H[i, j] = (-1)^popcount(i & j) / sqrt(d).  [OIQ] 3.1, [OMC] Key formulas."""
    assert d >= 1 and d & (d - 1) == 0
    idx = np.arange(d)
    par = np.zeros((d, d), dtype=np.int64)
    a = idx[:, None] & idx[None, :]
    while a.any():
        par ^= a & 1
        a = a >> 1
    return np.where(par == 1, -1.0, 1.0) / math.sqrt(d)


def fwht_recursive(x: np.ndarray) -> np.ndarray:
    """Normalised fast Walsh-Hadamard transform by the recursive butterfly of
    [OMC] Implementation notes: H_{2n} x = [H_n a + H_n b, H_n a - H_n b]/sqrt 2
    with x = [a, b].  Used only to pin :func:`hadamard_matrix`."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    if n == 1:
        return x.copy()
    a = fwht_recursive(x[..., : n // 2])
    b = fwht_recursive(x[..., n // 2:])
    return np.concatenate([a + b, a - b], axis=-1) / math.sqrt(2.0)


def quat_left_matrix(p) -> np.ndarray:
    """Matrix of x -> p (x) x (Hamilton product) for p = (a, b, c, e) =
    a + b i + c j + e k.  It is orthogonal with det |p|^4, so a unit quaternion
    gives an element of SO(4) ([OMC] Mathematical statement)."""
    a, b, c, e = (float(t) for t in p)
    return np.array([[a, -b, -c, -e],
                     [b, a, -e, c],
                     [c, e, a, -b],
                     [e, -c, b, a]], dtype=np.float64)


def quat_right_matrix(q) -> np.ndarray:
    """Matrix of x -> x (x) q (Hamilton product with q on the right) for
    q = (a, b, c, e).  Orthogonal with det |q|^4."""
    a, b, c, e = (float(t) for t in q)
    return np.array([[a, -b, -c, -e],
                     [b, a, e, -c],
                     [c, -e, a, b],
                     [e, c, -b, a]], dtype=np.float64)


def quat_conj(q) -> np.ndarray:
    a, b, c, e = (float(t) for t in q)
    return np.array([a, -b, -c, -e], dtype=np.float64)


def so4_pair_matrix(p, q) -> np.ndarray:
    """The general element of SO(4) as a pair of unit quaternions:
    x -> p (x) x (x) conj(q), i.e. L(p) R(conj q) (every rotation of R^4 has
    this form, and (p, q) and (-p, -q) give the same one).  The block form
    R_i in SO(4) of [OMC] Mathematical statement; q = 1 gives L(p)."""
    return quat_left_matrix(p) @ quat_right_matrix(quat_conj(q))


def block_so4_matrix(quats: np.ndarray, quats_r=None) -> np.ndarray:
    """B = diag(R_1, ..., R_{d/4}), R_i acting on coordinates 4i..4i+3:
    R_i = L(p_i), or L(p_i) R(conj q_i) when right quaternions are given."""
    n = len(quats)
    B = np.zeros((4 * n, 4 * n))
    for i, p in enumerate(quats):
        R = quat_left_matrix(p) if quats_r is None else so4_pair_matrix(p, quats_r[i])
        B[4 * i:4 * i + 4, 4 * i:4 * i + 4] = R
    return B


def rotation_matrix(signs: np.ndarray, quats: np.ndarray, quats_r=None) -> np.ndarray:
    """Dense U = B . H_d . D ([OMC] U = B H_d; [OIQ] 3.2 puts D before H)."""
    d = len(signs)
    return block_so4_matrix(quats, quats_r) @ hadamard_matrix(d) @ np.diag(signs.astype(np.float64))


# ---------------------------------------------------------------------------
# Scale storage types
# ---------------------------------------------------------------------------
def round_e4m3(s):
    """Round non-negative fp64 values to OCP FP8 E4M3 (bias 7, 3 mantissa bits,
    subnormal quantum 2^-9, largest finite 448): round half to even, saturating
    to 448 (the "satfinite" rule).  The quantum of the binade is found with
    frexp, so every step is exact in fp64."""
    s = np.asarray(s, dtype=np.float64)
    _, E = np.frexp(s)                      # s = f * 2^E, f in [0.5, 1)
    e = np.maximum(E - 1, -6)               # binade exponent; subnormals share -6
    quantum = np.ldexp(1.0, e - 3)
    q = np.rint(s / quantum) * quantum      # np.rint rounds half to even
    return np.minimum(np.where(s == 0, 0.0, q), 448.0)


def round_e4m3_signed(v):
    """E4M3 rounding of signed values: the sign, then round_e4m3 of |v|."""
    v = np.asarray(v, dtype=np.float64)
    return np.sign(v) * round_e4m3(np.abs(v))


def encode_e4m3_signed(q):
    """Bytes of exactly representable E4M3 values of either sign (sign bit 0x80)."""
    q = np.asarray(q, dtype=np.float64)
    return (encode_e4m3(np.abs(q)) | np.where(q < 0, 0x80, 0)).astype(np.uint8)


def encode_e4m3(q):
    """Bytes of exactly representable non-negative E4M3 values."""
    q = np.asarray(q, dtype=np.float64)
    _, E = np.frexp(q)
    e = np.maximum(E - 1, -6)
    sub = q < 2.0 ** -6
    m_sub = q / 2.0 ** -9
    m_nrm = (q / np.ldexp(1.0, e) - 1.0) * 8.0
    byte = np.where(sub, m_sub, (e + 7) * 8 + m_nrm)
    assert np.all(byte == np.floor(byte)) and np.all(byte <= 126)
    return byte.astype(np.uint8)


def decode_e4m3(byte):
    """fp64 values of E4M3 bytes (0x7F / 0xFF are NaN)."""
    byte = np.asarray(byte, dtype=np.int64)
    sgn = np.where(byte & 0x80, -1.0, 1.0)
    e = (byte >> 3) & 0xF
    m = (byte & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sgn * val


def round_f16(s):
    """IEEE binary16 round to nearest even (numpy's conversion), saturating to
    65504 instead of overflowing to infinity."""
    s = np.asarray(s, dtype=np.float64)
    return np.where(s >= 65520.0, 65504.0, np.minimum(s, 65504.0).astype(np.float16).astype(np.float64))


def round_scale(s, kind: str):
    """Round fp64 scales to their storage type (fp32 / fp16 / E4M3), RNE."""
    s = np.asarray(s, dtype=np.float64)
    if kind == "f32":
        return s.astype(np.float32).astype(np.float64)
    if kind == "f16":
        return round_f16(s)
    if kind == "e4m3":
        return round_e4m3(s)
    raise ValueError(kind)


def scale_midpoint_distance(s, kind: str):
    """Relative distance from each fp64 scale s to the nearest rounding
    midpoint of the storage type.  A block whose s lies within 1e-6 of one may
    legitimately be stored as either neighbour by a correct fp32 computation.
    Infinite for fp32 (one unit in the last place is already below the 1e-6
    scale tolerance) and beyond the largest finite value."""
    s = np.asarray(s, dtype=np.float64)
    if kind == "f32":
        return np.full(s.shape, np.inf)
    _, E = np.frexp(s)
    if kind == "f16":
        quantum = np.ldexp(1.0, np.maximum(E - 1, -14) - 10)
        top = 65504.0
    else:
        quantum = np.ldexp(1.0, np.maximum(E - 1, -6) - 3)
        top = 448.0
    mid = (np.floor(s / quantum) + 0.5) * quantum
    with np.errstate(divide="ignore", invalid="ignore"):
        dist = np.abs(s - mid) / s
    return np.where((s == 0) | (s >= top), np.inf, dist)


def encode_scales(q: np.ndarray, kind: str) -> np.ndarray:
    """Stored scale values (..., n) -> little-endian bytes (..., n*sb).  For
    "e4m3zp" q is (..., n, 2): (scale, zero point) of each block, stored as
    the scale byte then the zero-point byte."""
    q = np.asarray(q, dtype=np.float64)
    if kind == "e4m3zp":
        b = np.stack([encode_e4m3(q[..., 0]), encode_e4m3_signed(q[..., 1])], axis=-1)
        return b.reshape(q.shape[:-2] + (-1,))
    if kind == "f32":
        b = q.astype("<f4").view(np.uint8)
    elif kind == "f16":
        b = q.astype("<f2").view(np.uint8)
    else:
        b = encode_e4m3(q)
    return b.reshape(q.shape[:-1] + (-1,))


def decode_scales(buf: np.ndarray, kind: str) -> np.ndarray:
    """Scale bytes (uint8, ..., n*sb) -> fp64 values (..., n); for "e4m3zp"
    (..., n, 2) pairs (scale, zero point)."""
    buf = np.ascontiguousarray(buf)
    if kind == "e4m3zp":
        return decode_e4m3(buf.reshape(buf.shape[:-1] + (-1, 2)))
    if kind == "f32":
        return buf.view("<f4").astype(np.float64)
    if kind == "f16":
        return buf.view("<f2").astype(np.float64)
    return decode_e4m3(buf)


# ---------------------------------------------------------------------------
# Quantiser and packing
# ---------------------------------------------------------------------------
BIT_WIDTHS = (2, 3, 4)


def qmax(bits: int) -> int:
    """Largest code magnitude of the b-bit symmetric quantiser, 2^(b-1) - 1
    ([OMC] Key formulas; the method fixes b = 3, [OIQ] 3.3 and 5.1 use b = 2,
    3 and 4): 1, 3 or 7."""
    if bits not in BIT_WIDTHS:
        raise ValueError(f"bit width {bits} not in {BIT_WIDTHS}")
    return (1 << (bits - 1)) - 1


def quantize(x: np.ndarray, block: int, eps: float, kind: str, bits: int = 3):
    """Blockwise symmetric b-bit quantiser ([OMC] Key formulas): per block of
    ``block`` consecutive coordinates, s = (max|x| + eps)/(2^(b-1) - 1),
    stored as s_q = round(s) in the scale type, codes
    c = clip(round_half_even(x/s_q), -(2^(b-1) - 1), 2^(b-1) - 1)
    (c = 0 where s_q = 0).
    x: fp64 [n][d].  Returns (codes int8 [n][d], s_q fp64 [n][d/block],
    s fp64 [n][d/block])."""
    n, d = x.shape
    qm = qmax(bits)
    xb = x.reshape(n, d // block, block)
    s = (np.abs(xb).max(axis=-1, initial=0.0) + eps) / float(qm)
    sq = round_scale(s, kind)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sq[..., None] > 0, xb / sq[..., None], 0.0)
    c = np.clip(np.rint(r), -qm, qm).astype(np.int8)
    return c.reshape(n, d), sq, s


def quantize_asym(x: np.ndarray, block: int, eps: float, bits: int = 3):
    """The asymmetric variant of [HFF] (each 64-element sub-block keeps
    unsigned 3-bit codes and an FP8 header with a scale and a zero point):
    per block, z = min x and s = (max x - min x + eps)/(2^b - 1), both
    stored in E4M3 (round half to even, saturating; z keeps its sign), and
    unsigned codes u = clip(round_half_even((x - z_q)/s_q), 0, 2^b - 1)
    (u = 0 where s_q = 0).  Dequantisation: x_hat = s_q u + z_q.
    x: fp64 [n][d].  Returns (codes uint8 [n][d], (s_q, z_q) fp64
    [n][d/block][2], s fp64 [n][d/block])."""
    qmax(bits)
    n, d = x.shape
    top = (1 << bits) - 1
    xb = x.reshape(n, d // block, block)
    lo, hi = xb.min(axis=-1), xb.max(axis=-1)
    s = (hi - lo + eps) / float(top)
    sq = round_e4m3(s)
    zq = round_e4m3_signed(lo)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sq[..., None] > 0, (xb - zq[..., None]) / sq[..., None], 0.0)
    u = np.clip(np.rint(r), 0, top).astype(np.uint8)
    return u.reshape(n, d), np.stack([sq, zq], axis=-1), s


def calib_sse(x: np.ndarray, signs: np.ndarray, quats: np.ndarray, block: int, kind: str,
              bits: int = 3, eps: float = 1e-6, quats_r=None) -> np.ndarray:
    """Objective of the SO(4) calibration ([OMC] Implementation notes:
    reconstruction MSE after quantisation, SO(4) blocks as normalised
    quaternions): per quantisation block j, the sum over the sample vectors
    x (fp64 [n][d]) and the coordinates of block j of (y - y_hat)^2, with
    y = B H D x for these signs and quaternions (SO(4) blocks applied) and
    y_hat its quantised value (symmetric codes, or the asymmetric variant for
    kind "e4m3zp").  With quats_r, the blocks are the two-quaternion
    R_i = L(p_i) R(conj q_i).  Returns fp64 [d/block]."""
    U = rotation_matrix(np.asarray(signs), np.asarray(quats, dtype=np.float64),
                        None if quats_r is None else np.asarray(quats_r, dtype=np.float64))
    y = np.asarray(x, dtype=np.float64) @ U.T
    n, d = y.shape
    eps = float(np.float32(eps))
    if kind == "e4m3zp":
        u, sz, _ = quantize_asym(y, block, eps, bits)
        yh = (u.reshape(n, d // block, block) * sz[..., 0:1] + sz[..., 1:2]).reshape(n, d)
    else:
        c, sq, _ = quantize(y, block, eps, kind, bits)
        yh = (c.reshape(n, d // block, block) * sq[..., None]).reshape(n, d)
    return ((y - yh) ** 2).reshape(n, d // block, block).sum(axis=(0, 2))


def pack_codes(codes: np.ndarray, bits: int = 3) -> np.ndarray:
    """b-bit two's-complement codes [..., d] -> bytes [..., b*d/8]: element j
    at bits b*j..b*j+b-1 of a little-endian bit stream (bit k of the stream is
    bit k % 8 of byte k // 8) ([OMC] Implementation notes: codes packed into
    bytes; [OIQ] 4.2: INT3/INT4 packed values after the scale header)."""
    qmax(bits)
    d = codes.shape[-1]
    c = codes.astype(np.int64) & ((1 << bits) - 1)
    bs = np.stack([(c >> i) & 1 for i in range(bits)], axis=-1)      # [..., d, b]
    bs = bs.reshape(codes.shape[:-1] + (bits * d,)).astype(np.uint8)
    return np.packbits(bs, axis=-1, bitorder="little")


def unpack_codes(buf: np.ndarray, d: int, bits: int = 3, signed: bool = True) -> np.ndarray:
    """Inverse of :func:`pack_codes` (the value -2^(b-1), which the quantiser
    never writes, reads as itself); signed=False reads the unsigned codes of
    the asymmetric variant."""
    qmax(bits)
    bs = np.unpackbits(np.asarray(buf, dtype=np.uint8), axis=-1, bitorder="little")
    bs = bs.reshape(buf.shape[:-1] + (d, bits)).astype(np.int64)
    v = sum(bs[..., i] << i for i in range(bits))
    if not signed:
        return v.astype(np.uint8)
    half = 1 << (bits - 1)
    return np.where(v >= half, v - 2 * half, v).astype(np.int8)


# ---------------------------------------------------------------------------
# Cache layout ([OIQ] 4.2 header + packed data; [OMC] Kcache.append)
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Layout:
    """Byte layout of the packed cache.

    The pool is an array of pages of ``page_size`` (P) token slots.  A page
    holds, for kv heads 0..Hkv-1 in order, a K record then a V record.  A
    record is its scale header -- P*(d/block) scales, token-major
    (slot t, block j at index t*(d/block)+j), each in the scale type,
    little-endian -- followed by P code strings of b*d/8 bytes (slot t at
    t*b*d/8; b = ``bits``, 3 unless stated).  Token position ``pos`` of
    sequence ``b`` lives in slot pos % P of
    logical page pos // P; the physical page is page_table[b][pos // P], or
    b*max_pages_per_seq + pos // P for a contiguous cache (no page table)."""
    d: int
    num_kv_heads: int
    block: int
    scale: str
    page_size: int
    batch: int
    max_pages_per_seq: int
    num_pages: int
    bits: int = 3

    @property
    def nb(self) -> int:
        return self.d // self.block

    @property
    def sb(self) -> int:
        return SCALE_BYTES[self.scale]

    @property
    def code_bytes(self) -> int:
        return self.bits * self.d // 8

    @property
    def record_bytes(self) -> int:
        return self.page_size * (self.nb * self.sb + self.code_bytes)

    @property
    def page_bytes(self) -> int:
        return self.num_kv_heads * 2 * self.record_bytes

    @property
    def pool_bytes(self) -> int:
        return self.num_pages * self.page_bytes

    def page_id(self, page_table, b: int, logical: int) -> int:
        if page_table is None:
            return b * self.max_pages_per_seq + logical
        return int(page_table[b][logical])

    def record_offset(self, page: int, kv_head: int, which: int) -> int:
        return page * self.page_bytes + (kv_head * 2 + which) * self.record_bytes

    def scale_offset(self, page, kv_head, which, slot):
        return self.record_offset(page, kv_head, which) + slot * self.nb * self.sb

    def code_offset(self, page, kv_head, which, slot):
        return (self.record_offset(page, kv_head, which) + self.page_size * self.nb * self.sb
                + slot * self.code_bytes)


def locate(layout: Layout, page_table, b, pos):
    """Physical page, slot and status bits of positions ``pos`` of sequences
    ``b`` (arrays of equal shape).  Status bits are set where the sequence
    index, the position or the page id is out of range (page -1 there)."""
    b = np.asarray(b, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    st = np.zeros(b.shape, np.int64)
    st |= np.where((b < 0) | (b >= layout.batch), ST_BAD_SEQ, 0)
    cap = layout.max_pages_per_seq * layout.page_size
    st |= np.where((st == 0) & ((pos < 0) | (pos >= cap)), ST_BAD_POS, 0)
    ok = st == 0
    logical = np.where(ok, pos // layout.page_size, 0)
    bb = np.where(ok, b, 0)
    if page_table is None:
        page = bb * layout.max_pages_per_seq + logical
    else:
        page = np.asarray(page_table, dtype=np.int64)[bb, logical] if b.size else np.zeros(0, np.int64)
    st |= np.where(ok & ((page < 0) | (page >= layout.num_pages)), ST_BAD_PAGE, 0)
    page = np.where(st == 0, page, -1)
    return page, np.where(st == 0, pos % layout.page_size, -1), st


def _gather_index(base: np.ndarray, nbytes: int) -> np.ndarray:
    return base[:, None] + np.arange(nbytes)[None, :]


# ---------------------------------------------------------------------------
# Write path: rotate, quantise, pack, store   ([OMC] Implementation notes)
# ---------------------------------------------------------------------------
def write(pool: np.ndarray, layout: Layout, U: np.ndarray, k: np.ndarray, v: np.ndarray,
          seq_idx: np.ndarray, pos: np.ndarray, page_table=None, eps: float = 1e-6) -> int:
    """For every token i, kv head h and K/V ([OMC] "On every new token, compute
    k1 = U(k) and v1 = U(v) ... Store only packed codes and scales"):
    x = U @ fp64(vector); scales and codes per block; the code string and the
    scales are stored in the slot of (seq_idx[i], pos[i]).  Tokens without a
    valid slot are skipped and reported in the returned status bits.
    k, v: fp16 [n_tok][Hkv][d]; pool: uint8, updated in place."""
    eps = float(np.float32(eps))
    n_tok = k.shape[0]
    H = layout.num_kv_heads
    page, slot, st = locate(layout, page_table, seq_idx, pos)
    status = int(np.bitwise_or.reduce(st)) if n_tok else 0
    ok = np.nonzero(st == 0)[0]
    for which, src in ((0, k), (1, v)):
        x = src[ok].astype(np.float64).reshape(len(ok) * H, layout.d) @ U.T
        if layout.scale == "e4m3zp":
            codes, sq, _ = quantize_asym(x, layout.block, eps, layout.bits)
        else:
            codes, sq, _ = quantize(x, layout.block, eps, layout.scale, layout.bits)
        packed = pack_codes(codes, layout.bits)                 # [n*H, cb]
        hdr = encode_scales(sq, layout.scale)                   # [n*H, nb*sb]
        heads = np.tile(np.arange(H), len(ok))
        pg = np.repeat(page[ok], H)
        sl = np.repeat(slot[ok], H)
        rec = pg * layout.page_bytes + (heads * 2 + which) * layout.record_bytes
        so = rec + sl * layout.nb * layout.sb
        co = rec + layout.page_size * layout.nb * layout.sb + sl * layout.code_bytes
        pool[_gather_index(so, layout.nb * layout.sb)] = hdr
        pool[_gather_index(co, layout.code_bytes)] = packed
    return status


def read_rotated(pool: np.ndarray, layout: Layout, b: int, kv_head: int, which: int,
                 t0: int, nt: int, page_table=None):
    """Stored codes and scales of positions t0..t0+nt-1 of sequence b,
    dequantised in the rotated domain: x_hat = s_q * c ([OMC] Key formulas),
    or s_q * u + z_q for the asymmetric variant ("e4m3zp").
    Returns (x_hat fp64 [nt][d], codes int8 [nt][d] (uint8 for "e4m3zp"),
    scales fp64 [nt][d/m] ([nt][d/m][2] (scale, zero point) for "e4m3zp"))."""
    pos = np.arange(t0, t0 + nt)
    page, slot, st = locate(layout, page_table, np.full(nt, b), pos)
    if np.any(st):
        raise IndexError(f"sequence {b}: positions without a slot in [{t0}, {t0 + nt})")
    rec = page * layout.page_bytes + (kv_head * 2 + which) * layout.record_bytes
    so = rec + slot * layout.nb * layout.sb
    co = rec + layout.page_size * layout.nb * layout.sb + slot * layout.code_bytes
    sc = decode_scales(pool[_gather_index(so, layout.nb * layout.sb)], layout.scale)
    if layout.scale == "e4m3zp":     # x_hat = s_q u + z_q
        cs = unpack_codes(pool[_gather_index(co, layout.code_bytes)], layout.d, layout.bits, signed=False)
        cb = cs.reshape(nt, layout.nb, layout.block).astype(np.float64)
        xh = (cb * sc[..., 0:1] + sc[..., 1:2]).reshape(nt, layout.d)
        return xh, cs, sc
    cs = unpack_codes(pool[_gather_index(co, layout.code_bytes)], layout.d, layout.bits)
    xh = (cs.reshape(nt, layout.nb, layout.block) * sc[..., None]).reshape(nt, layout.d)
    return xh, cs, sc


# ---------------------------------------------------------------------------
# Read path: rotated-query attention over the packed cache
# ---------------------------------------------------------------------------
def attention_rotated(U: np.ndarray, q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray,
                      sm_scale: float) -> np.ndarray:
    """One query head against dequantised rotated keys/values ([OMC]
    Implementation notes, read path): q1 = U q; logits = (q1 . k_hat_t) *
    sm_scale; p = softmax(logits); y1 = p @ v_hat; y = U^T y1.  fp64
    throughout; no keys gives a zero output."""
    if k_hat.shape[0] == 0:
        return np.zeros(U.shape[0])
    q1 = U @ q.astype(np.float64)
    logits = (k_hat @ q1) * sm_scale
    p = np.exp(logits - logits.max())
    p /= p.sum()
    return U.T @ (p @ v_hat)


def decode(pool: np.ndarray, layout: Layout, U: np.ndarray, q: np.ndarray,
           seq_lens: np.ndarray, page_table=None, sm_scale: float = 0.0,
           heads=None) -> np.ndarray:
    """Decode attention for q [B][Hq][d] over positions [0, seq_lens[b]) of
    each sequence; query head h reads kv head h // (Hq/Hkv).  Returns fp64
    [B][Hq][d] (only the (b, h) pairs listed in ``heads`` if given, zeros
    elsewhere)."""
    B, Hq, d = q.shape
    G = Hq // layout.num_kv_heads
    if sm_scale <= 0:
        sm_scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, Hq, d))
    want = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    last = (None, None)
    for b, h in want:
        g = h // G
        if last[0] != (b, g):
            n = int(seq_lens[b])
            kh = read_rotated(pool, layout, b, g, 0, 0, n, page_table)[0]
            vh = read_rotated(pool, layout, b, g, 1, 0, n, page_table)[0]
            last = ((b, g), (kh, vh))
        kh, vh = last[1]
        out[b, h] = attention_rotated(U, q[b, h], kh, vh, sm_scale)
    return out


def prefill(pool: np.ndarray, layout: Layout, U: np.ndarray, q: np.ndarray, seq: int, pos0: int,
            page_table=None, sm_scale: float = 0.0) -> np.ndarray:
    """Chunked-prefill attention over the packed cache: query token i of
    q [n][Hq][d] sits at position pos0 + i of sequence ``seq`` and attends
    causally to positions [0, pos0 + i] -- exactly one decode step of the
    sequence truncated after its own position (the reading taken for the
    pages' prefill-phase attention: [OMC] read path, Key formulas with a
    causal mask).  Query head h reads kv head h // (Hq/Hkv).  Returns fp64
    [n][Hq][d]."""
    n, Hq, d = q.shape
    G = Hq // layout.num_kv_heads
    if sm_scale <= 0:
        sm_scale = 1.0 / math.sqrt(d)
    out = np.zeros((n, Hq, d))
    L = pos0 + n
    for g in range(layout.num_kv_heads):
        kh = read_rotated(pool, layout, seq, g, 0, 0, L, page_table)[0]
        vh = read_rotated(pool, layout, seq, g, 1, 0, L, page_table)[0]
        for i in range(n):
            m = pos0 + i + 1
            for gh in range(G):
                h = g * G + gh
                out[i, h] = attention_rotated(U, q[i, h], kh[:m], vh[:m], sm_scale)
    return out


def attention_plain(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float) -> np.ndarray:
    """softmax(k q * sm_scale) v for one query head in fp64 ([OMC] Key
    formulas, Attn(Q, K, V)); the reference that rotated attention must equal
    when nothing is quantised."""
    logits = (k.astype(np.float64) @ q.astype(np.float64)) * sm_scale
    p = np.exp(logits - logits.max())
    p /= p.sum()
    return p @ v.astype(np.float64)
