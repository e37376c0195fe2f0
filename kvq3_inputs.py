"""Seeded synthetic inputs for the rotated 3-bit KV cache (keys, values, queries,
sequence lengths and page tables).

This module is shared by the CPU oracle, the tests and the benchmark.  It holds
none of the method's arithmetic (no rotation, no quantisation, no packing): it
only draws numbers.  Everything is counter based, so any slice of any tensor can
be regenerated on its own, on the host (numpy) or on a CUDA device (torch), with
the same bits.

Generator (SplitMix64, Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): the i-th output (i = 0, 1, ...) of the stream seeded
with ``s`` is ``mix(s + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64)`` where ``mix``
is the published finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift
27, multiply 0x94D049BB133111EB, xor-shift 31).

Distribution (what the pages describe for real key/value activations):
  * standard normal entries by the Box-Muller transform in float64
    (u1 in (0, 1], u2 in [0, 1), z0 = sqrt(-2 ln u1) cos(2 pi u2),
    z1 = sqrt(-2 ln u1) sin(2 pi u2)); entry 2i takes z0 of pair i, entry 2i+1
    takes z1 -- Orthogonal Invariance in Activation Space, section 2.1
    (sparse extreme outliers in 2-5 % of dimensions);
  * a seeded set of outlier channels per (kv head, K or V), chosen by a partial
    Fisher-Yates shuffle, multiplied by a factor (x20 or x30);
  * keys only: magnitude decays with position as 1/sqrt(1 + pos/256)
    (same page, section 2.1, pattern 2);
  * queries: plain N(0, 1);
  * everything is rounded to fp16 (round to nearest even) at the end.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

# stream tags: which tensor a stream feeds
TAG_K, TAG_V, TAG_Q, TAG_CH_K, TAG_CH_V, TAG_LENS, TAG_PAGES = 1, 2, 3, 4, 5, 6, 7


def _mix_int(z: int) -> int:
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def splitmix64_at(seed: int, i: int) -> int:
    """i-th output (0-based) of the SplitMix64 stream seeded with ``seed``."""
    return _mix_int((seed + (i + 1) * GOLDEN) & MASK64)


def stream_seed(data_seed: int, tag: int, a: int = 0, b: int = 0) -> int:
    """Seed of the stream feeding tensor ``tag`` at index (a, b).

    Derived by drawing one SplitMix64 output from a key made of the fields,
    so streams of different tensors are unrelated."""
    key = (data_seed * 0x100000001B3 + tag * 0x1000193 + a * 0x10001 + b * 0x101) & MASK64
    return splitmix64_at(key, 0)


# ---------------------------------------------------------------- numpy side
def _mix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def splitmix64_np(seed: int, idx: np.ndarray) -> np.ndarray:
    """Outputs number ``idx`` (uint64 array) of the stream seeded with ``seed``."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (idx.astype(np.uint64) + np.uint64(1)) * np.uint64(GOLDEN)
        return _mix_np(z)


def normal_np(seed: int, start: int, count: int) -> np.ndarray:
    """Entries [start, start+count) of the N(0,1) stream ``seed`` (float64)."""
    if count <= 0:
        return np.zeros(0, np.float64)
    p0 = start // 2
    p1 = (start + count + 1) // 2
    pairs = np.arange(p0, p1, dtype=np.uint64)
    r1 = splitmix64_np(seed, 2 * pairs)
    r2 = splitmix64_np(seed, 2 * pairs + np.uint64(1))
    u1 = ((r1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (r2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * math.pi * u2
    z = np.empty(2 * len(pairs), np.float64)
    z[0::2] = rad * np.cos(ang)
    z[1::2] = rad * np.sin(ang)
    off = start - 2 * p0
    return z[off:off + count]


def outlier_channels(data_seed: int, which: int, kv_head: int, d: int, frac: float) -> np.ndarray:
    """Outlier channel indices of (kv_head, K|V): round-half-even(frac*d) of
    them, the first entries of a seeded partial Fisher-Yates shuffle of [0, d)."""
    n = int(np.rint(frac * d))
    s = stream_seed(data_seed, TAG_CH_K if which == 0 else TAG_CH_V, kv_head)
    perm = list(range(d))
    for i in range(n):
        j = i + splitmix64_at(s, i) % (d - i)
        perm[i], perm[j] = perm[j], perm[i]
    return np.array(sorted(perm[:n]), dtype=np.int64)


@dataclass(frozen=True)
class DataSpec:
    """Distribution of one synthetic workload's K/V/q (see module docstring)."""
    d: int
    num_kv_heads: int
    seed: int
    outlier_frac: float = 0.03
    outlier_factor: float = 20.0
    # kv heads that use ``outlier_frac_hi`` instead (the "middle half" of heads)
    hi_heads: tuple = field(default_factory=tuple)
    outlier_frac_hi: float = 0.0
    key_decay: bool = True

    def frac(self, kv_head: int) -> float:
        return self.outlier_frac_hi if kv_head in self.hi_heads else self.outlier_frac


def kv_rows_np(spec: DataSpec, which: int, b: int, kv_head: int, pos0: int, n: int) -> np.ndarray:
    """fp16 [n][d] rows of K (which=0) or V (which=1) for sequence b, kv head
    ``kv_head``, positions pos0..pos0+n-1."""
    d = spec.d
    s = stream_seed(spec.seed, TAG_K if which == 0 else TAG_V, b, kv_head)
    x = normal_np(s, pos0 * d, n * d).reshape(n, d)
    ch = outlier_channels(spec.seed, which, kv_head, d, spec.frac(kv_head))
    x[:, ch] *= spec.outlier_factor
    if which == 0 and spec.key_decay:
        pos = np.arange(pos0, pos0 + n, dtype=np.float64)
        x *= (1.0 / np.sqrt(1.0 + pos / 256.0))[:, None]
    return x.astype(np.float16)


def q_np(spec: DataSpec, batch: int, num_q_heads: int, step: int = 0) -> np.ndarray:
    """fp16 [batch][Hq][d] queries of decode step ``step``."""
    out = np.empty((batch, num_q_heads, spec.d), np.float16)
    for b in range(batch):
        for h in range(num_q_heads):
            s = stream_seed(spec.seed, TAG_Q, b * 65536 + h, step)
            out[b, h] = normal_np(s, 0, spec.d).astype(np.float16)
    return out


def seq_lens_np(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """int32 lengths drawn uniformly from [lo, hi] (inclusive)."""
    s = stream_seed(seed, TAG_LENS)
    span = hi - lo + 1
    return np.array([lo + splitmix64_at(s, i) % span for i in range(batch)], dtype=np.int32)


def shuffled_page_ids_np(seed: int, n: int) -> np.ndarray:
    """A seeded Fisher-Yates shuffle of [0, n) (int32)."""
    s = stream_seed(seed, TAG_PAGES)
    perm = np.arange(n, dtype=np.int64)
    r = splitmix64_np(s, np.arange(n, dtype=np.uint64))
    for i in range(n - 1, 0, -1):
        j = int(r[n - 1 - i] % np.uint64(i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm.astype(np.int32)


def page_table_np(seed: int, seq_lens: np.ndarray, page_size: int, max_pages_per_seq: int):
    """Page table [batch][max_pages_per_seq] (int32, -1 where unused) that hands
    the shuffled ids of [0, sum ceil(L_b/P)) to the sequences in order.
    Returns (table, num_pages)."""
    need = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    total = sum(need)
    ids = shuffled_page_ids_np(seed, total)
    table = np.full((len(seq_lens), max_pages_per_seq), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = ids[o:o + n]
        o += n
    return table, total


# ---------------------------------------------------------------- torch side
def _torch():
    import torch
    return torch


def _mix_torch(z):
    """SplitMix64 finaliser on int64 tensors (two's complement wrap-around,
    logical right shifts emulated by masking)."""
    torch = _torch()

    def shr(x, k):
        return (x >> k) & ((1 << (64 - k)) - 1)

    m1 = torch.tensor(M1 - (1 << 64), dtype=torch.int64, device=z.device)
    m2 = torch.tensor(M2 - (1 << 64), dtype=torch.int64, device=z.device)
    z = (z ^ shr(z, 30)) * m1
    z = (z ^ shr(z, 27)) * m2
    return z ^ shr(z, 31)


def _to_i64(u: int) -> int:
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def normal_torch(seed: int, start: int, count: int, device):
    """Same numbers as :func:`normal_np`, computed on ``device`` (float64)."""
    torch = _torch()
    p0 = start // 2
    p1 = (start + count + 1) // 2
    pairs = torch.arange(p0, p1, dtype=torch.int64, device=device)
    g = torch.tensor(_to_i64(GOLDEN), dtype=torch.int64, device=device)
    s = torch.tensor(_to_i64(seed), dtype=torch.int64, device=device)
    r1 = _mix_torch(s + (2 * pairs + 1) * g)
    r2 = _mix_torch(s + (2 * pairs + 2) * g)
    top = (1 << 53) - 1
    u1 = (((r1 >> 11) & top).to(torch.float64) + 1.0) * (2.0 ** -53)
    u2 = ((r2 >> 11) & top).to(torch.float64) * (2.0 ** -53)
    rad = torch.sqrt(-2.0 * torch.log(u1))
    ang = 2.0 * math.pi * u2
    z = torch.stack([rad * torch.cos(ang), rad * torch.sin(ang)], dim=1).reshape(-1)
    off = start - 2 * p0
    return z[off:off + count]


def _round_fp16_torch(x):
    """float64 -> float16 with a single round-to-nearest-even (as numpy's
    conversion does).  A plain .to(float16) may pass through float32 and
    round twice; here the value is first rounded to the fp16 grid in float64
    (quantum 2^(e-10), subnormal quantum 2^-24), which the cast then keeps."""
    torch = _torch()
    _, E = torch.frexp(x)
    quantum = torch.ldexp(torch.ones_like(x), torch.clamp(E - 1, min=-14) - 10)
    return (torch.round(x / quantum) * quantum).to(torch.float16)


def kv_rows_torch(spec: DataSpec, which: int, b: int, kv_head: int, pos0: int, n: int, device):
    """Same rows as :func:`kv_rows_np`, generated on ``device`` (fp16 [n][d])."""
    torch = _torch()
    d = spec.d
    s = stream_seed(spec.seed, TAG_K if which == 0 else TAG_V, b, kv_head)
    x = normal_torch(s, pos0 * d, n * d, device).reshape(n, d)
    ch = outlier_channels(spec.seed, which, kv_head, d, spec.frac(kv_head))
    if len(ch):
        idx = torch.as_tensor(ch, device=device)
        x[:, idx] *= spec.outlier_factor
    if which == 0 and spec.key_decay:
        pos = torch.arange(pos0, pos0 + n, dtype=torch.float64, device=device)
        x *= (1.0 / torch.sqrt(1.0 + pos / 256.0))[:, None]
    return _round_fp16_torch(x)


# ---------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    """One of the five seeded workloads of the rotated 3-bit KV cache."""
    name: str
    batch: int
    num_kv_heads: int
    num_q_heads: int
    d: int
    block: int
    scale: str            # "f32" | "f16" | "e4m3"
    rot_flags: int        # 1 = sign flip, 2 = SO(4) blocks (H_d is always on)
    page_size: int
    paged: bool
    seq_len: int          # attended length (uniform workloads)
    len_range: tuple      # (lo, hi) for ragged workloads, else ()
    data: DataSpec
    rot_seed: int = 42
    decode: bool = True
    eps: float = 1e-6
    chunk: int = 0        # prefill-attention workloads: query tokens of the chunk
    bits: int = 3         # code width b (2, 3 or 4)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def workloads():
    """The five workloads: data seed 1000 + index, rotation seed 42."""
    return {
        "tiny": Workload("tiny", 1, 4, 4, 128, 64, "f32", 3, 64, False, 1024, (),
                         DataSpec(128, 4, 1000, 0.03, 20.0)),
        "llama8b": Workload("llama8b", 16, 8, 32, 128, 64, "f16", 3, 128, False, 32768, (),
                            DataSpec(128, 8, 1001, 0.03, 20.0)),
        "long70b": Workload("long70b", 8, 8, 64, 128, 64, "e4m3", 3, 128, False, 131072, (),
                            DataSpec(128, 8, 1002, 0.03, 20.0, hi_heads=(2, 3, 4, 5),
                                     outlier_frac_hi=0.08)),
        "prefill": Workload("prefill", 1, 8, 8, 128, 32, "f32", 1, 64, False, 131072, (),
                            DataSpec(128, 8, 1003, 0.03, 20.0), decode=False),
        "prefill_attn": Workload("prefill_attn", 1, 8, 32, 128, 64, "f16", 3, 128, False, 32768, (),
                                 DataSpec(128, 8, 1005, 0.03, 20.0), decode=False, chunk=2048),
        "ragged": Workload("ragged", 64, 4, 16, 256, 64, "f16", 3, 16, True, 0, (1024, 65536),
                           DataSpec(256, 4, 1004, 0.05, 30.0)),
    }
