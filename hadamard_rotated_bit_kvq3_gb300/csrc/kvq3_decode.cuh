// Fused split-K decode attention over the packed 3-bit cache.
//
// "Orthogonally mixed 3-bit KV cache", Implementation notes (read path):
// q1 = U(q); unpack and scale keys inside the dot product; logits from q1 and
// the reconstructed transformed keys; softmax; multiply by the reconstructed
// transformed values; rotate the output back with U^T; unpacking, scale
// multiplication and accumulation fused so full fp16 K/V never exist.
// Key formulas: Attn = softmax(QK^T/sqrt d)V.  "Orthogonal Invariance in
// Activation Space", 4.3: dequantisation fused into the attention kernel.
//
// Design (one GPU, HBM-bound):
//  * Work = the flattened list of chunks of every (sequence, kv head) unit (a
//    chunk is up to ceil(kChunk/P) consecutive pages of the unit: fewer when
//    two stages of them would not fit in a resident CTA's share of shared
//    memory).  A persistent grid of 4-warp CTAs splits the list into equal
//    contiguous ranges.
//  * Each chunk's K and V records stream into a ring of shared-memory stages
//    with cp.async.bulk (mbarrier completion, L2 evict-first), one warp
//    issuing a chunk with lane i copying page i; the four warps share every
//    stage, one 16-token step each, meet at one barrier per chunk, and one
//    of them then refills the stage just released with the chunk S places
//    ahead.
//  * Each warp keeps an online-softmax state per unit; at the end of a unit
//    the four states merge (max, rescale, sum) into one fp32 partial
//    (o1[G][d] unnormalised, max, sum) at workspace slot (cta + unit), unique
//    because CTA ranges and units are both ordered.  A second kernel merges
//    the partials of each (sequence, query head) with the log-sum-exp rule
//    and applies U^T.
//  * QK^T and PV run on tensor cores (mma.sync m16n8k16, fp16 in, fp32
//    accumulate).  A b-bit field (b = 2, 3, 4) placed in the mantissa of a
//    half with a zero exponent is an exact subnormal; with its sign bit
//    flipped it reads (c + 2^(b-1)) 2^(k-24).  Keys take one LOP3 per pair of
//    codes and the offset enters as a per-block constant seeded into the
//    logit accumulator; values take a byte permute per 2-4 fields, a mask
//    and one half2 subtraction.  The powers of two are folded into q1 (keys)
//    or into the output (values).  The asymmetric variant's unsigned codes
//    need neither the flip nor the offset; its zero points add z_k * sum q1
//    per block to the logits and sum p z_v per block to the outputs.  q1 is
//    split into hi + lo fp16 halves (two columns per head) so the logits
//    keep ~fp32 accuracy; the probabilities are split the same way with fp32
//    value scales, at up to 4 heads per kv head and in the asymmetric
//    variant.  Per-(token, block) scales multiply the per-block partial dot
//    products (keys) or the probabilities (values).
#pragma once

#include <float.h>

#include <type_traits>

#include "kvq3_internal.h"

namespace kvq3 {

constexpr int kChunk = 192;      // minimum tokens per chunk (smaller pages are grouped)
constexpr int kMaxPagesPerChunk = kChunk / 16;
constexpr int kWarps = 4;        // consumer warps per CTA
constexpr int kMaxStages = 8;

struct DecodeParams {
  CacheGeom g;
  const uint8_t* pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const __half* q;        // [B][Hq][D]
  float* ws;              // partial slots
  int32_t* unit_cta;      // [units][2]: first and last CTA holding chunks of each unit
  int32_t* status;
  int32_t G;              // query heads per kv head
  int32_t Hq;
  float qk_scale;         // sm_scale * log2(e)
  float inv_sqrt_d;
  int32_t stages;         // ring depth
  uint32_t stage_bytes;   // bytes per stage
  int32_t chunk_tokens;   // tokens per chunk: max(64, P)
  int32_t pages_per_chunk;
  int32_t ctas;
  uint32_t slot_floats;   // floats per partial slot: G*(D+2)
  uint32_t smem_bytes;    // dynamic shared memory of a CTA (checked builds)
  int64_t slots;          // partial slots of the workspace (checked builds)
  uint32_t wait_limit;    // bound on mbarrier polls
  // Chunked prefill (pf_n > 0): the "sequences" are tiles of sequence
  // pf_seq: tile b holds query tokens tb*pf_qt .. (tb = b / pf_hb) and the
  // head block hb = b % pf_hb of pf_hpb query heads of each kv head; column
  // c of a unit is query token tb*pf_qt + c / pf_hpb and query head
  // hb*pf_hpb + c % pf_hpb of the kv head (when < pf_gkv).  Query token i sits
  // at position pf_pos0 + i and attends to positions [0, pf_pos0 + i].
  int32_t pf_n;           // query tokens (0: decode)
  int32_t pf_qt;          // query tokens per tile
  int32_t pf_hb;          // head blocks per kv head
  int32_t pf_hpb;         // query heads per head block
  int32_t pf_gkv;         // query heads per kv head
  int32_t pf_seq;         // the sequence
  int64_t pf_pos0;        // position of query token 0
};

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ int64_t seq_len_checked(const DecodeParams& p, int b, bool flag) {
  if (p.pf_n > 0) {   // query tile b attends up to its last token (checked on the host)
    const int64_t last = min((int64_t)(b / p.pf_hb + 1) * p.pf_qt, (int64_t)p.pf_n);
    return p.pf_pos0 + last;
  }
  const int64_t len = p.seq_lens[b];
  const int64_t cap = (int64_t)p.g.max_pages * p.g.page_size;
  if (len < 0 || len > cap) {
    if (flag) set_status(p.status, KVQ3_DEV_BAD_LEN);
    return 0;
  }
  return len;
}

__device__ __forceinline__ int64_t seq_chunks(const DecodeParams& p, int b, bool flag) {
  // lengths are int32, so the rounded-up sum stays below 2^32
  return (int64_t)(((uint32_t)seq_len_checked(p, b, flag) + (uint32_t)(p.chunk_tokens - 1)) /
                   (uint32_t)p.chunk_tokens);
}

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Total chunks over all (sequence, kv head) units.
__device__ __forceinline__ int64_t total_chunks(const DecodeParams& p, bool flag) {
  const int lane = threadIdx.x & 31;
  int64_t acc = 0;
  for (int b0 = 0; b0 < p.g.batch; b0 += 32) {
    const int b = b0 + lane;
    acc += warp_sum64(b < p.g.batch ? seq_chunks(p, b, flag) : 0);
  }
  return acc * p.g.hkv;
}

// Position in the flattened chunk list: sequence b, kv head, chunk c of nc.
struct Cursor {
  int b, kvh;
  int64_t c, nc;
};

__device__ __forceinline__ Cursor cursor_at(const DecodeParams& p, int64_t idx) {
  const int lane = threadIdx.x & 31;
  int64_t acc = 0;
  Cursor cur{p.g.batch, 0, 0, 0};
  for (int b0 = 0; b0 < p.g.batch; b0 += 32) {
    const int b = b0 + lane;
    const int64_t n = b < p.g.batch ? seq_chunks(p, b, false) * p.g.hkv : 0;
    int64_t incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t excl = incl - n;
    const unsigned hit = __ballot_sync(kFull, n > 0 && acc + excl <= idx && idx < acc + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const int64_t base = acc + __shfl_sync(kFull, excl, src);
      const int64_t ncb = __shfl_sync(kFull, n, src) / p.g.hkv;
      const int64_t within = idx - base;
      cur.b = b0 + src;
      cur.nc = ncb;
      cur.kvh = (int)(within / ncb);
      cur.c = within % ncb;
      return cur;
    }
    acc += __shfl_sync(kFull, incl, 31);
  }
  return cur;
}

__device__ __forceinline__ void cursor_next(const DecodeParams& p, Cursor& cur) {
  if (++cur.c < cur.nc) return;
  cur.c = 0;
  if (++cur.kvh < p.g.hkv) return;
  cur.kvh = 0;
  do {
    ++cur.b;
    cur.nc = cur.b < p.g.batch ? seq_chunks(p, cur.b, false) : 0;
  } while (cur.b < p.g.batch && cur.nc == 0);
}

// Compile-time loop: f(integral_constant<int, 0>) ... f(integral_constant<int, N-1>).
template <int I, int N, typename F>
__device__ __forceinline__ void static_for_impl(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for_impl<I + 1, N>(f);
  }
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  static_for_impl<0, N>(f);
}

// half2 subtraction on raw bits
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a);
  const __half2 y = *reinterpret_cast<const __half2*>(&b);
  x = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&x);
}

// ---- codes -> fp16, as subnormal halves.  A b-bit field u placed at
// mantissa bit k of a half with a zero exponent is the exact fp16 value
// u * 2^(k-24).  With the field's sign bit flipped, u = c + 2^(b-1) (c the
// two's-complement code), so the half is (c + 2^(b-1)) 2^(k-24): the power of
// two is folded into q1 (keys) or the output (values), and the offset is
// either removed per half (values) or, for keys, becomes the per-block
// constant 2^(b-1) * sum_d 2^k_d q1_d that seeds the logit accumulators (so
// the key path is one mask per half2).

// Key pairs: a lane's FQ consecutive fields (FQ = 16 or 8; field 0 at bit 0 of
// the 64-bit window lo:hi) -> FQ/2 half2 values, each holding field fl(P) at
// mantissa bit kl(P) of the low half and field fh(P) at bit kh(P) of the high
// half (a b-bit field at bit k of a half with a zero exponent needs
// k + b <= 10).
//
// 3-bit fields: pair P cuts the window (lo:hi) >> o(P), so 3 fl - o = kl and
// 3 fh - o - 16 = kh; the pairings use four shifted windows for 16 fields
// (found by exhaustive search over window offsets) and two for 8.
//                                                  P:  0   1  2   3   4   5   6   7
__host__ __device__ constexpr int kp3_o(int FQ, int P) {
  return FQ == 16 ? (P == 0 ? -7 : P == 1 ? -4 : P == 2 ? 0 : P < 5 ? 14 : 23)
                  : (P < 2 ? -4 : P == 2 ? 0 : 2);
}
__host__ __device__ constexpr int kp3_fl(int FQ, int P) {
  return FQ == 16 ? (P == 0 ? 0 : P == 1 ? 1 : P == 2 ? 2 : P == 3 ? 5 : P + 3) : P;
}
__host__ __device__ constexpr int kp3_fh(int FQ, int P) {
  return FQ == 16 ? (P == 0 ? 3 : P == 1 ? 4 : P == 2 ? 6 : P + 8) : P + 4;
}
// 4-bit fields: word w = P/4 of the window holds fields 8w..8w+7 at nibbles;
// pair P = (8w + a, 8w + a + 4), a = P % 4, from the word shifted right by 8
// when a >= 2: both halves at bit 4 (a % 2).
// 2-bit fields: byte pair g = P/4 holds fields 8g..8g+7; a byte permute puts
// byte 2g in the low half and byte 2g+1 in the high half: pair P =
// (8g + a, 8g + a + 4) at bit 2a of each half.
__host__ __device__ constexpr int kp_fl(int NBIT, int FQ, int P) {
  return NBIT == 3 ? kp3_fl(FQ, P) : 8 * (P / 4) + P % 4;
}
__host__ __device__ constexpr int kp_fh(int NBIT, int FQ, int P) {
  return NBIT == 3 ? kp3_fh(FQ, P) : 8 * (P / 4) + P % 4 + 4;
}
__host__ __device__ constexpr int kp_kl(int NBIT, int FQ, int P) {
  return NBIT == 3 ? 3 * kp3_fl(FQ, P) - kp3_o(FQ, P) : NBIT == 4 ? 4 * (P % 2) : 2 * (P % 4);
}
__host__ __device__ constexpr int kp_kh(int NBIT, int FQ, int P) {
  return NBIT == 3 ? 3 * kp3_fh(FQ, P) - kp3_o(FQ, P) - 16 : kp_kl(NBIT, FQ, P);
}
__host__ __device__ constexpr bool kp_valid(int NBIT, int FQ) {
  unsigned seen = 0;
  for (int P = 0; P < FQ / 2; ++P) {
    const int kl = kp_kl(NBIT, FQ, P), kh = kp_kh(NBIT, FQ, P);
    if (kl < 0 || kl + NBIT > 10 || kh < 0 || kh + NBIT > 10) return false;
    if (NBIT == 3 && ((kp3_o(FQ, P) % 3) + 3) % 3 == 1) return false;
    seen |= (1u << kp_fl(NBIT, FQ, P)) | (1u << kp_fh(NBIT, FQ, P));
  }
  return seen == (1u << FQ) - 1u;
}
static_assert(kp_valid(3, 16) && kp_valid(3, 8) && kp_valid(4, 16) && kp_valid(4, 8) &&
                  kp_valid(2, 16) && kp_valid(2, 8),
              "key pair tables must cover every field once");

// Sign bits of the fields, flipped so that a field reads c + 2^(b-1):
// 3-bit: bits 3i+2 of a code string after a right shift by o sit at
// positions congruent to (2 - o) mod 3; 4-bit: bit 3 of every nibble;
// 2-bit: bit 1 of every bit pair (the shifts and byte permutes above keep
// nibbles and bit pairs aligned).
constexpr uint32_t kSignRes0 = 0x49249249u;   // positions 0, 3, 6, ...
constexpr uint32_t kSignRes2 = 0x24924924u;   // positions 2, 5, 8, ...
constexpr uint32_t kSign4 = 0x88888888u;
constexpr uint32_t kSign2 = 0xAAAAAAAAu;

// d = (a ^ s) & M in one LOP3 (M an immediate).
template <uint32_t M>
__device__ __forceinline__ uint32_t xor_and(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(d) : "r"(a), "r"(s), "n"(M));
  return d;
}

// Pair P of a key chunk (lo, hi) as a subnormal half2 (c + 2^(b-1)) 2^(k - 24).
// s0 / s2: the sign patterns (3-bit: kSignRes0 / kSignRes2; else both the
// width's pattern) held in registers.
template <int NBIT, int FQ, int P>
__device__ __forceinline__ uint32_t k_pair(uint32_t lo, uint32_t hi, uint32_t s0, uint32_t s2) {
  constexpr int kl = kp_kl(NBIT, FQ, P), kh = kp_kh(NBIT, FQ, P);
  constexpr uint32_t F = (1u << NBIT) - 1u;
  constexpr uint32_t M = (F << kl) | (F << (16 + kh));
  if constexpr (NBIT == 3) {
    constexpr int o = kp3_o(FQ, P);
    uint32_t w;
    if constexpr (o < 0) w = lo << (-o);
    else if constexpr (o == 0) w = lo;
    else w = __funnelshift_r(lo, hi, o);
    return xor_and<M>(w, ((o % 3) + 3) % 3 == 0 ? s2 : s0);
  } else if constexpr (NBIT == 4) {
    const uint32_t w = (P < 4 ? lo : hi) >> ((P % 4) >= 2 ? 8 : 0);
    return xor_and<M>(w, s0);
  } else {
    constexpr uint32_t sel = (P / 4) == 0 ? 0x1100u : 0x3322u;
    return xor_and<M>(__byte_perm(lo, 0u, sel), s0);
  }
}

// Value codes: fields f = 0..F-1 (F = 8 or 4) of two tokens' chunks -> half2
// (token0, token1) of field f, equal to c 2^(voff(f) - 24).
//   3-bit: the byte permute takes bytes g, g+1 of each token's chunk (g = 0,
//     1, 2 for fields 0-2, 3-5, 6-7); the sign bits of that half sit at the
//     positions of kSignVg[g] (both halves).
//   4-bit: byte f/2 of each chunk, field at bit 4 (f % 2).
//   2-bit: byte f/4 of each chunk, field at bit 2 (f % 4).
__host__ __device__ constexpr int v_off(int NBIT, int f) {
  return NBIT == 4 ? 4 * (f % 2)
       : NBIT == 2 ? 2 * (f % 4)
       : (f == 0 ? 0 : f == 1 ? 3 : f == 2 ? 6 : f == 3 ? 1 : f == 4 ? 4 : f == 5 ? 7 : f == 6 ? 2 : 5);
}
constexpr uint32_t kSignVg0 = 0x49244924u, kSignVg1 = 0x92499249u, kSignVg2 = 0x24922492u;

// UNS: unsigned codes (the asymmetric variant): the field is the code itself,
// with no sign flip (s0..s2 are 0) and no offset to remove.
template <int NBIT, int F, bool UNS = false>
__device__ __forceinline__ uint32_t v_field(uint32_t c0, uint32_t c1, uint32_t s0, uint32_t s1, uint32_t s2) {
  constexpr int o = v_off(NBIT, F);
  constexpr uint32_t FM = (1u << NBIT) - 1u;
  constexpr uint32_t M = (FM << o) | (FM << (16 + o));
  constexpr uint32_t OFS = (1u << (NBIT - 1)) * 0x00010001u << o;   // 2^(b-1) in both halves
  if constexpr (UNS) {
    constexpr uint32_t sel = NBIT == 3 ? (F < 3 ? 0x5410u : (F < 6 ? 0x6521u : 0x7632u))
                                       : ((NBIT == 4 ? F / 2 : F / 4) * 0x1111u + 0x4400u);
    return __byte_perm(c0, c1, sel) & M;
  } else if constexpr (NBIT == 3) {
    constexpr uint32_t sel = F < 3 ? 0x5410u : (F < 6 ? 0x6521u : 0x7632u);
    const uint32_t w = __byte_perm(c0, c1, sel);
    return hsub2_bits(xor_and<M>(w, F < 3 ? s0 : (F < 6 ? s1 : s2)), OFS);
  } else {
    constexpr uint32_t g = NBIT == 4 ? F / 2 : F / 4;
    constexpr uint32_t sel = g | (g << 4) | ((4 + g) << 8) | ((4 + g) << 12);
    return hsub2_bits(xor_and<M>(__byte_perm(c0, c1, sel), s0), OFS);
  }
}

// Bits [boff, boff + 64) of a code string (two aligned words, funnel shift).
__device__ __forceinline__ void load_bits(const uint8_t* str, int boff, uint32_t& lo, uint32_t& hi) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(str) + (boff >> 5);
  const int sh = boff & 31;
  const uint32_t w0 = w[0], w1 = w[1];
  lo = __funnelshift_r(w0, w1, sh);
  hi = w1 >> sh;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------------ kernel 1
// Shared-memory loads at 32-bit addresses with immediate offsets.  volatile:
// they must stay after the mbarrier wait that publishes the stage.
template <int OFF>
__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}

// N bytes (1..32, a power of two) at shared address a + OFF as 32-bit words.
template <int N, int OFF>
__device__ __forceinline__ void lds_bytes(uint32_t a, uint32_t (&w)[(N + 3) / 4]) {
  if constexpr (N == 1) w[0] = lds8<OFF>(a);
  else if constexpr (N == 2) w[0] = lds16<OFF>(a);
  else if constexpr (N == 4) w[0] = lds32<OFF>(a);
  else if constexpr (N == 8) {
    const uint2 v = lds64<OFF>(a);
    w[0] = v.x; w[1] = v.y;
  } else if constexpr (N == 16) {
    const uint4 v = lds128<OFF>(a);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint4 v = lds128<OFF>(a), u = lds128<OFF + 16>(a);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    w[4] = u.x; w[5] = u.y; w[6] = u.z; w[7] = u.w;
  }
}

// Decoded scales: NB values of type SCALE from raw words (pairs converted
// together: one half2 -> float2 for fp16, one fp8x2 -> half2 -> float2 for E4M3).
template <int NB, int SCALE>
struct ScaleDec {
  static constexpr int SB = SCALE == KVQ3_SCALE_F32 ? 4
                          : (SCALE == KVQ3_SCALE_F16 || SCALE == KVQ3_SCALE_E4M3_ZP) ? 2 : 1;
  static constexpr int BPT = NB * SB;
  // values i = 0..n-1 starting at value index i0 of w
  template <int N, int I0>
  __device__ static __forceinline__ void decode(const uint32_t* w, float* s) {
    if constexpr (SCALE == KVQ3_SCALE_F32) {
#pragma unroll
      for (int i = 0; i < N; ++i) s[i] = __uint_as_float(w[I0 + i]);
    } else if constexpr (SCALE == KVQ3_SCALE_F16) {
      if constexpr (N == 1) {
        s[0] = __half2float(__ushort_as_half((unsigned short)(w[I0 / 2] >> (16 * (I0 & 1)))));
      } else {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
          const uint32_t v = w[(I0 + i) / 2];
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
          s[i] = f.x;
          s[i + 1] = f.y;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < N; i += 2) {
        const uint32_t v = w[(I0 + i) / 4] >> (8 * ((I0 + i) & 3));
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
        const float2 f = __half22float2(__half2(hr));
        s[i] = f.x;
        if (i + 1 < N) s[i + 1] = f.y;
      }
    }
  }
  template <int OFF>
  __device__ static __forceinline__ void one(uint32_t a, float (&s)[NB]) {
    uint32_t w[(BPT + 3) / 4];
    lds_bytes<BPT, OFF>(a, w);
    decode<NB, 0>(w, s);
  }
  // tokens at a and a + BPT (the pair is aligned to its size)
  template <int OFF>
  __device__ static __forceinline__ void two(uint32_t a, float (&s0)[NB], float (&s1)[NB]) {
    uint32_t w[(2 * BPT + 3) / 4];
    lds_bytes<2 * BPT, OFF>(a, w);
    decode<NB, 0>(w, s0);
    decode<NB, NB>(w, s1);
  }
  // Asymmetric variant: (scale, zero point) E4M3 byte pairs of blocks
  // I0 .. I0+N-1, one fp8x2 conversion per block.
  template <int N, int I0>
  __device__ static __forceinline__ void decode_sz(const uint32_t* w, float* s, float* z) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const uint32_t v = w[(I0 + i) / 2] >> (16 * ((I0 + i) & 1));
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
      const float2 f = __half22float2(__half2(hr));
      s[i] = f.x;
      z[i] = f.y;
    }
  }
  template <int OFF>
  __device__ static __forceinline__ void one_sz(uint32_t a, float (&s)[NB], float (&z)[NB]) {
    uint32_t w[(BPT + 3) / 4];
    lds_bytes<BPT, OFF>(a, w);
    decode_sz<NB, 0>(w, s, z);
  }
  template <int OFF>
  __device__ static __forceinline__ void two_sz(uint32_t a, float (&s0)[NB], float (&s1)[NB], float (&z0)[NB],
                                                float (&z1)[NB]) {
    uint32_t w[(2 * BPT + 3) / 4];
    lds_bytes<2 * BPT, OFF>(a, w);
    decode_sz<NB, 0>(w, s0, z0);
    decode_sz<NB, NB>(w, s1, z1);
  }
};

// Per-step values handed between the parts of a decode step.
template <int NTQ>
struct StepLogits {
  float s0[NTQ], s1[NTQ];   // rows r and r + 8
};
template <int NB, int NTP>
struct StepP {
  uint32_t b[NB][NTP][2];   // P' fragments (B operand of PV)
};

// What the producer thread publishes with each chunk (at the end of its stage).
struct ChunkDesc {
  int32_t unit, b, kvh, n_tok;
  uint32_t page_ok;  // bit i: page i of the chunk has a valid id (else masked)
  int32_t c;         // chunk index within its unit
  int32_t nc;        // chunks of the unit
  int32_t len;       // attended length of the sequence
};

// q1 fragments live in shared memory (one copy per CTA) for the variants
// where they would take 32+ registers; elsewhere in registers.
__host__ __device__ constexpr bool decode_qf_smem(int D, int GPAD) { return D == 256 || GPAD == 16; }

template <int D, int GPAD>
struct DecodeSmem {
  static constexpr int kFullOff = 0;                              // kMaxStages mbarriers
  static constexpr int kEmptyOff = kFullOff + 8 * kMaxStages;     // abort flag (+ spare)
  static constexpr int kMLOff = kEmptyOff + 8 * kMaxStages;       // [kWarps][2][GPAD] floats
  static constexpr int kQOff = (kMLOff + kWarps * 2 * GPAD * 4 + 15) / 16 * 16;  // [GPAD][D]
  static constexpr int kQInvOff = kQOff + GPAD * D * 4;           // [GPAD]
  static constexpr int kKofsOff = kQInvOff + GPAD * 4;            // [D/32][GPAD] logit seeds
  static constexpr int kQfOff = (kKofsOff + (D / 32) * GPAD * 4 + 15) / 16 * 16;  // [D/16][GPAD/4][32] uint2
  static constexpr int kStageOff =
      ((kQfOff + (decode_qf_smem(D, GPAD) ? (D / 16) * (GPAD / 4) * 256 : 0)) + 127) / 128 * 128;
};

// Resident CTAs per SM the register budget is sized for: the accumulators
// (D/16 x 4 per PV n-tile) and the q1 fragments (D/8 per QK n-tile) grow
// with D and the group padding.
__host__ __device__ constexpr int decode_min_blocks(int D, int GPAD) {
  return GPAD == 16 ? (D == 256 ? 1 : 2) : GPAD == 8 ? (D == 256 ? 2 : 3) : (D == 256 ? 3 : 4);
}

// PSPLIT: the probabilities-times-value-scales P' enter PV as hi + lo fp16
// halves (PV n-tile = 4 heads x (hi, lo), like QK) -- needed when the value
// scales are fp32, since p = 1 times an fp32 scale is not an fp16 value;
// otherwise one fp16 value per head (PV n-tile = 8 heads).
template <int D, int BLOCK, int GPAD, int SCALE, int NBIT, bool PSPLIT, bool PF = false>
__global__ void __launch_bounds__(128, decode_min_blocks(D, GPAD))
    decode_split_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ RotParams rp) {
  constexpr int NB = D / BLOCK;
  constexpr int KS = D / 16;          // k-steps of QK^T == M-tiles of PV
  constexpr int KSB = BLOCK / 16;     // per block
  constexpr int NTQ = GPAD / 4;       // QK n-tiles: 4 heads x (hi, lo)
  constexpr int NTP = PSPLIT ? NTQ : (GPAD + 7) / 8;  // PV n-tiles
  constexpr int FQ = BLOCK / 4;       // key fields per lane per block
  constexpr int FV = BLOCK / 8;       // value fields per lane per block
  constexpr int CB = NBIT * D / 8;    // code bytes per token
  // Asymmetric variant: unsigned codes, x_hat = s u + z per (token, block):
  // logits gain z_k * sum_{d in block} q1_d, outputs sum_t p_t z_v
  constexpr bool ASYM = SCALE == KVQ3_SCALE_E4M3_ZP;
  static_assert(!ASYM || PSPLIT, "the asymmetric variant splits P'");
  constexpr int EQ = D >= 128 ? D / 32 : 4;  // query rotation layout
  constexpr int LQ = D / EQ;
  constexpr int GPWQ = 32 / LQ;
  using SM = DecodeSmem<D, GPAD>;
  using SDec = ScaleDec<NB, SCALE>;
  constexpr int BPT = SDec::BPT;

  // Launched as a programmatic dependent of the preceding kernel (the token
  // write, typically): everything up to here overlaps it, and nothing is
  // read before its writes are complete and visible.
  griddep_wait();
  // the combine kernel may launch now: it waits for this grid before reading
  griddep_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int j = lane & 3, r = lane >> 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kFullOff);
  volatile uint32_t* abort_s = reinterpret_cast<volatile uint32_t*>(smem + SM::kEmptyOff);  // a copy never arrived
  float* ml_s = reinterpret_cast<float*>(smem + SM::kMLOff);
  float* qs = reinterpret_cast<float*>(smem + SM::kQOff);
  float* qinv_s = reinterpret_cast<float*>(smem + SM::kQInvOff);
  uint8_t* stg = smem + SM::kStageOff;
  const uint32_t stg_u32 = smem_u32(stg);
  const int S = p.stages;
  const CacheGeom& g = p.g;
  const uint32_t REC = (uint32_t)g.record_bytes, HDR = (uint32_t)g.scale_hdr_bytes;
  const uint32_t desc_off = p.stage_bytes - (uint32_t)sizeof(ChunkDesc);

  const int64_t cta = blockIdx.x;
  const int64_t T = total_chunks(p, cta == 0 && wid == 0);
  // W = min(CTAs, chunks): every CTA below W gets a non-empty range, so the
  // CTAs holding a unit's chunks are consecutive (the combine walks them)
  const int64_t W = T < p.ctas ? T : p.ctas;
  if (cta >= W) return;  // uniform over the CTA
  const int64_t c0 = cta * T / W, c1 = (cta + 1) * T / W;
  const int64_t nch = c1 - c0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    *abort_s = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---- producer: chunk descriptor + bulk copies of its pages, issued by one
  // whole warp (lane i copies page i of the chunk): warp 0 fills the first
  // stages; afterwards the last warp to release a stage refills it
  const uint64_t pol = policy_evict_first();
  auto issue = [&](const Cursor& c, int stage, int64_t len) {   // warp-collective
    uint8_t* dst = stg + (size_t)stage * p.stage_bytes;
    // chunk c.c covers logical pages c.c*ppc .. of sequence c.b (32-bit: a
    // sequence holds fewer than 2^31 tokens)
    const int ppc = p.pages_per_chunk;
    const int tok0 = (int)c.c * p.chunk_tokens;
    const int n_tok = min(p.chunk_tokens, (int)len - tok0);
    const int npg = n_tok == p.chunk_tokens ? ppc : (n_tok + g.page_size - 1) / g.page_size;
    const int lp = (int)c.c * ppc + lane;
    int64_t pg = -1;
    const int64_t row = p.pf_n > 0 ? p.pf_seq : c.b;   // prefill tiles all read one sequence
    if (lane < npg)
      pg = p.page_table ? (int64_t)p.page_table[row * g.max_pages + lp] : row * g.max_pages + lp;
    const bool ok = pg >= 0 && pg < g.num_pages;
    const uint32_t okm = __ballot_sync(kFull, ok);
    if (lane == 0) {
      if (okm != (1u << npg) - 1u) set_status(p.status, KVQ3_DEV_BAD_PAGE);
      ChunkDesc* dsc = reinterpret_cast<ChunkDesc*>(dst + desc_off);
      dsc->unit = c.b * g.hkv + c.kvh;
      dsc->b = c.b;
      dsc->kvh = c.kvh;
      dsc->n_tok = n_tok;
      dsc->page_ok = okm;
      dsc->c = (int32_t)c.c;
      dsc->nc = (int32_t)c.nc;
      dsc->len = (int32_t)len;
      if (okm) mbar_expect_tx(&full[stage], (uint32_t)__popc(okm) * 2u * REC);
      else mbar_arrive(&full[stage]);
    }
    __syncwarp();
    if (ok && KVQ3_CHECK(p.status, in_range(SM::kStageOff + (int64_t)stage * p.stage_bytes + (int64_t)lane * 2 * REC,
                                            2 * REC, p.smem_bytes) &&
                                   in_range(pg * g.page_bytes + (int64_t)(c.kvh * 2) * REC, 2 * REC,
                                            g.num_pages * g.page_bytes)))
      bulk_g2s(dst + (size_t)lane * 2 * REC, p.pool + (int64_t)(c.kvh * 2) * REC + pg * g.page_bytes, 2 * REC,
               &full[stage], pol);
  };
  {
    Cursor cp = cursor_at(p, c0);  // warp-collective
    if (wid == 0) {
      for (int64_t i = 0; i < nch && i < S; ++i) {
        issue(cp, (int)i, seq_len_checked(p, cp.b, false));
        cursor_next(p, cp);
      }
    }
  }

  // per-lane query rotation parameters (dims rq*EQ ..)
  const int rq = lane % LQ, gq = lane / LQ;
  const uint32_t sgn_q = lane_signs<EQ>(rp, rq);

  // lane-constant offsets from a page's K record: this lane's key chunk
  // (token r, fields j*FQ.. of each block), value chunk (token 2j, fields
  // r*FV.. of each block) and their scales.  Block b's chunk lies 3*BLOCK/8
  // bytes after block 0's, at the same bit shift (3*BLOCK is a multiple of 32).
  const uint32_t kshf = (uint32_t)(NBIT * j * FQ) & 31u, vshf = (uint32_t)(NBIT * r * FV) & 31u;
  const uint32_t k_lane = HDR + (uint32_t)(r * CB) + ((uint32_t)(NBIT * j * FQ) >> 5) * 4u;
  const uint32_t v_lane = REC + HDR + (uint32_t)(2 * j * CB) + ((uint32_t)(NBIT * r * FV) >> 5) * 4u;
  const uint32_t ks_lane = (uint32_t)(r * BPT), vs_lane = REC + (uint32_t)(2 * j * BPT);
  static_assert((NBIT * BLOCK) % 32 == 0, "block chunks must start on a word boundary");
  constexpr int KBB = NBIT * BLOCK / 8;   // bytes per block of a code string
  constexpr int KBITS = NBIT * FQ, VBITS = NBIT * FV;   // bits of a lane's key / value chunk

  // sign-bit patterns of the key windows, kept in registers (one LOP3 per pair)
  constexpr uint32_t kSignB = NBIT == 4 ? kSign4 : kSign2;
  // unsigned codes (ASYM) flip no sign bit: (x ^ 0) & M
  const uint32_t sgn0 = ASYM ? 0u : NBIT == 3 ? kSignRes0 : kSignB;
  const uint32_t sgn2 = ASYM ? 0u : NBIT == 3 ? kSignRes2 : kSignB;
  const uint32_t vsg0 = NBIT == 3 ? kSignVg0 : kSignB, vsg1 = kSignVg1, vsg2 = kSignVg2;

  // q1 fragments (B operand of QK^T): in registers for d = 128 with up to 8
  // heads per kv head (they are read by every MMA of the logit chain); in
  // shared memory, one copy per CTA, where they would take 32+ registers of a
  // larger variant: fragment (k-step s, n-tile tq) of lane l at
  // kQfOff + ((s*NTQ + tq)*32 + l)*8
  constexpr bool QF_SMEM = decode_qf_smem(D, GPAD);
  uint32_t qf[QF_SMEM ? 1 : NTQ][QF_SMEM ? 1 : KS][2];
  uint2* qf_s = reinterpret_cast<uint2*>(smem + SM::kQfOff);
  const uint32_t qf_lane = smem_u32(qf_s) + (uint32_t)lane * 8u;
  float qinv[NTQ];
  int64_t lim[PF ? NTQ : 1];   // prefill: causal limit of each logit column
  // logit accumulator seeds (key offset, see setup_unit): registers when few,
  // else shared memory [block][head]
  constexpr bool KOFS_REG = NB * NTQ <= 4;
  float kofs[KOFS_REG ? NB : 1][KOFS_REG ? NTQ : 1];
  float* kofs_s = reinterpret_cast<float*>(smem + SM::kKofsOff);
  float m[NTQ], l[NTQ];
  float acc[KS][NTP][4];
  // ASYM: sum_t p_t z_v[t, block] of this lane's P' column (head 4tp + r/2)
  float zacc[ASYM ? NTP : 1][ASYM ? NB : 1];
  int cur_unit = -1;
  bool cur_first = false, cur_last = false;

  // merge the four warps' states of a unit into workspace slot (cta + unit);
  // the CTA holding the unit's first (last) chunk records itself as such
  auto flush = [&](int unit, bool first, bool last) {
    // checked builds: the slot and the unit range entry lie in the workspace
    // (the merge below still runs, every warp reaching its barriers)
    const bool slot_ok =
        KVQ3_CHECK(p.status, cta + unit < p.slots && unit >= 0 && unit < (int64_t)g.batch * g.hkv);
    if (threadIdx.x == 0 && slot_ok) {
      if (first) p.unit_cta[2 * unit] = (int32_t)cta;
      if (last) p.unit_cta[2 * unit + 1] = (int32_t)cta;
    }
    float* slot = p.ws + (size_t)(cta + unit) * p.slot_floats;
    float* mS = slot + p.G * D;
    float* lS = mS + p.G;
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      float lt = l[tq];
      lt += __shfl_xor_sync(kFull, lt, 4);
      lt += __shfl_xor_sync(kFull, lt, 8);
      lt += __shfl_xor_sync(kFull, lt, 16);
      if (r == 0) {
        ml_s[(wid * 2 + 0) * GPAD + 4 * tq + j] = m[tq];
        ml_s[(wid * 2 + 1) * GPAD + 4 * tq + j] = lt;
      }
    }
    named_barrier(1, 128);
    float cw[NTQ];  // this warp's weight for QK head 4tq + j
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      const int h = 4 * tq + j;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml_s[(w * 2) * GPAD + h]);
      cw[tq] = M == -INFINITY ? 0.0f : ex2(m[tq] - M);
      if (wid == 0 && r == 0 && h < p.G) {
        float L = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = ml_s[(w * 2) * GPAD + h];
          L += (M == -INFINITY ? 0.0f : ex2(mw - M)) * ml_s[(w * 2 + 1) * GPAD + h];
        }
        if (slot_ok) {
          mS[h] = M;
          lS[h] = L;
        }
      }
    }
    // weights for the PV columns this lane holds
    float cpv[NTP][2];
#pragma unroll
    for (int tp = 0; tp < NTP; ++tp) {
      if constexpr (PSPLIT) {
        cpv[tp][0] = cpv[tp][1] = cw[tp];
      } else {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hc = 8 * tp + 2 * j + e;
          float v = 0.0f;
#pragma unroll
          for (int tq = 0; tq < NTQ; ++tq) {
            const float t = __shfl_sync(kFull, cw[tq], hc & 3);
            v = (tq == (hc >> 2)) ? t : v;
          }
          cpv[tp][e] = v;
        }
      }
    }
    // ASYM: the zero-point sums of head 4tp + j: column 2j's lanes 8j..8j+3
    // hold its tokens (the hi column; the lo column holds the same sums)
    float zh[ASYM ? NTP : 1][ASYM ? NB : 1];
    if constexpr (ASYM) {
#pragma unroll
      for (int tp = 0; tp < NTP; ++tp)
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float z = zacc[tp][b];
          z += __shfl_xor_sync(kFull, z, 1);
          z += __shfl_xor_sync(kFull, z, 2);
          zh[tp][b] = __shfl_sync(kFull, z, 8 * j);
        }
    }
    // warp 0 stores its weighted state, then warps 1..3 add theirs
    for (int pass = 0; pass < 2; ++pass) {
      if ((pass == 0) == (wid == 0)) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int b = mt / KSB, mp = mt % KSB;
#pragma unroll
          for (int tp = 0; tp < NTP; ++tp) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {      // row r (e = 0) or r + 8 (e = 1)
              const int f = 2 * mp + e;
              const int dim = b * BLOCK + r * FV + f;
              const float sc = (float)(1 << (24 - v_off(NBIT, f)));   // value halves are c 2^(voff-24)
              if constexpr (PSPLIT) {
                const int h = 4 * tp + j;
                float v = (acc[mt][tp][2 * e] + acc[mt][tp][2 * e + 1]) * sc;
                if constexpr (ASYM) v += zh[tp % (ASYM ? NTP : 1)][b % (ASYM ? NB : 1)];
                v *= cpv[tp][0];
                if (h < p.G && slot_ok) {
                  if (pass == 0) slot[h * D + dim] = v;
                  else atomicAdd(&slot[h * D + dim], v);
                }
              } else {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                  const int h = 8 * tp + 2 * j + c;
                  const float v = acc[mt][tp][2 * e + c] * sc * cpv[tp][c];
                  if (h < p.G && slot_ok) {
                    if (pass == 0) slot[h * D + dim] = v;
                    else atomicAdd(&slot[h * D + dim], v);
                  }
                }
              }
            }
          }
        }
      }
      named_barrier(1, 128);
    }
  };

  // rotate the unit's G query heads once per CTA, then build each warp's
  // B fragments: qs[g][dim] = (U q)[dim] * sm_scale*log2e * 2^e_g
  auto setup_unit = [&](int b, int kvh) {
    if constexpr (PF) {
      // causal limit of this lane's logit columns 4tq + j: position of its
      // query token (columns past the last token keep no limit: their q is 0)
#pragma unroll
      for (int tq = 0; tq < NTQ; ++tq) {
        const int col = 4 * tq + j;
        const int tok = (b / p.pf_hb) * p.pf_qt + col / p.pf_hpb;
        lim[tq] = (col < p.G && tok < p.pf_n) ? p.pf_pos0 + tok : INT64_MAX;
      }
    }
    for (int g0 = wid * GPWQ; g0 < GPAD; g0 += kWarps * GPWQ) {
      const int gg = g0 + gq;
      bool valid = gg < p.G;
      int64_t qrow;   // row of q [..][Hq][D]
      if constexpr (PF) {
        const int tok = (b / p.pf_hb) * p.pf_qt + gg / p.pf_hpb;
        const int hd = (b % p.pf_hb) * p.pf_hpb + gg % p.pf_hpb;   // head within the kv group
        valid = valid && tok < p.pf_n && hd < p.pf_gkv;
        qrow = (int64_t)tok * p.Hq + (int64_t)kvh * p.pf_gkv + hd;
      } else {
        qrow = (int64_t)b * p.Hq + (int64_t)kvh * p.G + gg;
      }
      float x[EQ];
      const __half* src = p.q + (valid ? qrow : 0) * D + rq * EQ;
#pragma unroll
      for (int e = 0; e < EQ; ++e) x[e] = valid ? __half2float(src[e]) : 0.0f;
      {
        // this lane's quaternions, read from the parameter space here rather
        // than held in registers across the kernel
        float4 quat_q[EQ / 4], quat_r[EQ / 4];
        lane_quats<EQ>(rp, rq, quat_q);
        lane_quats_r<EQ>(rp, rq, quat_r);
        rotate_forward<EQ, LQ>(x, rq, sgn_q, quat_q, quat_r, p.inv_sqrt_d, rot_so4(rp), rot_pair(rp));
      }
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < EQ; ++e) {
        x[e] *= p.qk_scale;
        amax = fmaxf(amax, fabsf(x[e]));
      }
#pragma unroll
      for (int o = 1; o < LQ; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      int ex = 0;
      if (amax > 0.0f) frexpf(amax, &ex);           // amax < 2^ex
      ex = max(-100, min(100, 8 - ex));               // scaled max in (2^7, 2^8]
      const float sc = ldexpf(1.0f, ex);
      if (gg < GPAD) {
#pragma unroll
        for (int e = 0; e < EQ; ++e) qs[gg * D + rq * EQ + e] = x[e] * sc;
        if (rq == 0) qinv_s[gg] = ldexpf(1.0f, 24 - ex);   // 2^24: subnormal key halves
      }
    }
    named_barrier(1, 128);
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      const int head = 4 * tq + (r >> 1);
      const int part = r & 1;
      float csum[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) csum[b] = 0.0f;
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int b = s / KSB, sp = s % KSB;
        uint32_t q2[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int P = 2 * sp + hf;
          const int dlo = b * BLOCK + j * FQ + kp_fl(NBIT, FQ, P);
          const int dhi = b * BLOCK + j * FQ + kp_fh(NBIT, FQ, P);
          const float vlo = qs[head * D + dlo] * (1.0f / (float)(1 << kp_kl(NBIT, FQ, P)));
          const float vhi = qs[head * D + dhi] * (1.0f / (float)(1 << kp_kh(NBIT, FQ, P)));
          const __half hlo = __float2half_rn(vlo), hhi = __float2half_rn(vhi);
          const float olo = part == 0 ? __half2float(hlo) : vlo - __half2float(hlo);
          const float ohi = part == 0 ? __half2float(hhi) : vhi - __half2float(hhi);
          q2[hf] = pack_half2(olo, ohi);
          // sum_d 2^k_d q1_d of the fp16 values the MMA sees (this lane's part)
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&q2[hf]));
          csum[b] += f.x * (float)(1 << kp_kl(NBIT, FQ, P)) + f.y * (float)(1 << kp_kh(NBIT, FQ, P));
        }
        if constexpr (QF_SMEM) {
          if (wid == 0) qf_s[(s * NTQ + tq) * 32 + lane] = make_uint2(q2[0], q2[1]);
        } else {
          qf[tq % (QF_SMEM ? 1 : NTQ)][s % (QF_SMEM ? 1 : KS)][0] = q2[0];
          qf[tq % (QF_SMEM ? 1 : NTQ)][s % (QF_SMEM ? 1 : KS)][1] = q2[1];
        }
      }
      // reduce over the lane's quad (fields) and the hi/lo parts: lanes 8h..8h+7
      // then hold head 4tq + h; the logit lanes of head 4tq + j read lane 8j.
      // The key halves are (c + 2^(b-1)) 2^(k-24): seed the accumulators with
      // -2^(b-1) * 2^-24 * sum_d 2^k_d q1_d so they sum c 2^(k-24) q1.  The
      // asymmetric variant seeds nothing and keeps 2^-24 * sum_d q1_d (the
      // same sum) for its zero-point term.
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float t = csum[b];
        t += __shfl_xor_sync(kFull, t, 1);
        t += __shfl_xor_sync(kFull, t, 2);
        t += __shfl_xor_sync(kFull, t, 4);
        // ASYM: no offset; the zero-point term needs 2^-24 sum_d q1_d instead
        const float ko = (ASYM ? 1.0f : -(float)(1 << (NBIT - 1))) * 0x1p-24f * __shfl_sync(kFull, t, 8 * j);
        if constexpr (KOFS_REG) kofs[b][tq] = ko;
        else if (wid == 0 && r == 0) kofs_s[b * GPAD + 4 * tq + j] = ko;
      }
      qinv[tq] = qinv_s[4 * tq + j];
    }
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      m[tq] = -INFINITY;
      l[tq] = 0.0f;
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int tp = 0; tp < NTP; ++tp)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[mt][tp][c] = 0.0f;
#pragma unroll
    for (int tp = 0; tp < (ASYM ? NTP : 1); ++tp)
#pragma unroll
      for (int b = 0; b < (ASYM ? NB : 1); ++b) zacc[tp][b] = 0.0f;
    named_barrier(1, 128);  // qs is rewritten at the next unit
  };

  // A 16-token step at token offset t0 of a page whose K record starts at
  // shared address pg (V record at pg + REC), n_valid tokens of the page,
  // comes in four parts: the logits, the running-max update, P' and PV.
  // FULL: all 16 tokens valid.  tok (prefill): position of token t0.
  // ------------------------------------------------ S = K q1 (per block)
  // sc0 / sc1: logits of tokens t0 + r and t0 + r + 8, column 4tq + j
  using SL = StepLogits<NTQ>;
  using SP = StepP<NB, NTP>;
  auto logits = [&](uint32_t pg, int t0, auto full_c, int n_valid, int64_t tok, SL& sl) {
    constexpr bool FULL = decltype(full_c)::value;
    float* sc0 = sl.s0;
    float* sc1 = sl.s1;
    float accq[NB][NTQ][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int tq = 0; tq < NTQ; ++tq) {
        accq[b][tq][0] = accq[b][tq][2] = 0.0f;
        accq[b][tq][1] = accq[b][tq][3] =
            ASYM ? 0.0f
                 : KOFS_REG ? kofs[b % (KOFS_REG ? NB : 1)][tq % (KOFS_REG ? NTQ : 1)]
                            : kofs_s[b * GPAD + 4 * tq + j];   // lo column
      }
    const uint32_t kt = pg + (uint32_t)(t0 * CB) + k_lane;   // token t0 + r
    static_for<NB>([&](auto bc) {
      constexpr int b = decltype(bc)::value;
      // this lane's key chunks of tokens r and r + 8 as 64-bit windows lo:hi
      uint32_t lo0, hi0 = 0, lo8, hi8 = 0;
      if constexpr (KBITS % 32 == 0) {          // whole words (kshf = 0)
        lo0 = lds32<b * KBB>(kt);
        lo8 = lds32<b * KBB + 8 * CB>(kt);
        if constexpr (KBITS > 32) {
          hi0 = lds32<b * KBB + 4>(kt);
          hi8 = lds32<b * KBB + 8 * CB + 4>(kt);
        }
      } else if constexpr (32 % KBITS == 0) {   // within one word
        lo0 = lds32<b * KBB>(kt) >> kshf;
        lo8 = lds32<b * KBB + 8 * CB>(kt) >> kshf;
      } else {
        const uint32_t x0 = lds32<b * KBB>(kt), x1 = lds32<b * KBB + 4>(kt);
        const uint32_t y0 = lds32<b * KBB + 8 * CB>(kt), y1 = lds32<b * KBB + 8 * CB + 4>(kt);
        lo0 = __funnelshift_r(x0, x1, kshf);
        hi0 = x1 >> kshf;
        lo8 = __funnelshift_r(y0, y1, kshf);
        hi8 = y1 >> kshf;
      }
      static_for<KSB>([&](auto spc) {
        constexpr int sp = decltype(spc)::value;
        uint32_t af[4];
        af[0] = k_pair<NBIT, FQ, 2 * sp>(lo0, hi0, sgn0, sgn2);
        af[1] = k_pair<NBIT, FQ, 2 * sp>(lo8, hi8, sgn0, sgn2);
        af[2] = k_pair<NBIT, FQ, 2 * sp + 1>(lo0, hi0, sgn0, sgn2);
        af[3] = k_pair<NBIT, FQ, 2 * sp + 1>(lo8, hi8, sgn0, sgn2);
        static_for<NTQ>([&](auto tqc) {
          constexpr int tq = decltype(tqc)::value;
          if constexpr (QF_SMEM) {
            const uint2 qv = lds64<((b * KSB + sp) * NTQ + tq) * 256>(qf_lane);
            mma_16816(accq[b][tq], af, qv.x, qv.y);
          } else {
            constexpr int s1 = QF_SMEM ? 0 : b * KSB + sp, t1 = QF_SMEM ? 0 : tq;
            mma_16816(accq[b][tq], af, qf[t1][s1][0], qf[t1][s1][1]);
          }
        });
      });
    });
    float skr[NB], skr8[NB], zkr[NB], zkr8[NB];
    {
      const uint32_t a = pg + (uint32_t)(t0 * BPT) + ks_lane;
      if constexpr (ASYM) {
        SDec::template one_sz<0>(a, skr, zkr);
        SDec::template one_sz<8 * BPT>(a, skr8, zkr8);
      } else {
        SDec::template one<0>(a, skr);
        SDec::template one<8 * BPT>(a, skr8);
      }
    }
    const bool vr = FULL || t0 + r < n_valid, vr8 = FULL || t0 + r + 8 < n_valid;
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if constexpr (ASYM) {   // + z_k * 2^-24 sum_{d in block} q1_d
          const float qz = KOFS_REG ? kofs[b % (KOFS_REG ? NB : 1)][tq % (KOFS_REG ? NTQ : 1)]
                                    : kofs_s[b * GPAD + 4 * tq + j];
          s0 = fmaf(zkr[b], qz, s0);
          s1 = fmaf(zkr8[b], qz, s1);
        }
        s0 = fmaf(skr[b], accq[b][tq][0] + accq[b][tq][1], s0);
        s1 = fmaf(skr8[b], accq[b][tq][2] + accq[b][tq][3], s1);
      }
      sc0[tq] = vr ? s0 * qinv[tq] : -INFINITY;
      sc1[tq] = vr8 ? s1 * qinv[tq] : -INFINITY;
      if constexpr (PF) {   // causal mask: rows are tokens t0 + r and t0 + r + 8
        const int64_t t = tok + r;
        if (t > lim[tq % (PF ? NTQ : 1)]) sc0[tq] = -INFINITY;
        if (t + 8 > lim[tq % (PF ? NTQ : 1)]) sc1[tq] = -INFINITY;
      }
    }
  };

  // ------------------------------------------------ online softmax
  // The running max m of a head moves only when a score exceeds it: one vote
  // finds that, and only then are the exact max (quad-column reduction) and
  // the rescale of l and of the accumulators computed; otherwise
  // p = 2^(s - m) <= 1 as before.
  auto update = [&](const SL& sl) {
    const float* sc0 = sl.s0;
    const float* sc1 = sl.s1;
    bool over = false;
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) over |= sc0[tq] > m[tq] || sc1[tq] > m[tq];
    if (__any_sync(kFull, over)) {
      float alpha[NTQ];
#pragma unroll
      for (int tq = 0; tq < NTQ; ++tq) {
        float mx = fmaxf(sc0[tq], sc1[tq]);
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float mn = fmaxf(m[tq], mx);   // decode: finite, every step has a valid token
        // prefill: a column may have seen no token yet (all masked): keep 1
        alpha[tq] = (PF && mn == -INFINITY) ? 1.0f : ex2(m[tq] - mn);
        l[tq] *= alpha[tq];
        m[tq] = mn;
      }
      if constexpr (PSPLIT) {
        // this lane's PV columns belong to its own QK head 4tp + j
#pragma unroll
        for (int tp = 0; tp < NTP; ++tp)
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][tp][c] *= alpha[tp];
        if constexpr (ASYM) {   // zacc belongs to head 4tp + r/2: lane r/2 holds its alpha
#pragma unroll
          for (int tp = 0; tp < NTP; ++tp) {
            const float az = __shfl_sync(kFull, alpha[tp], r >> 1);
#pragma unroll
            for (int b = 0; b < NB; ++b) zacc[tp % (ASYM ? NTP : 1)][b % (ASYM ? NB : 1)] *= az;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float av[NTQ];
#pragma unroll
          for (int tq = 0; tq < NTQ; ++tq) av[tq] = __shfl_sync(kFull, alpha[tq], (2 * j + e) & 3);
#pragma unroll
          for (int tp = 0; tp < NTP; ++tp) {
            const int tsel = (8 * tp + 2 * j + e) >> 2;
            float a = 1.0f;
#pragma unroll
            for (int tq = 0; tq < NTQ; ++tq) a = (tq == tsel) ? av[tq] : a;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              acc[mt][tp][e] *= a;
              acc[mt][tp][2 + e] *= a;
            }
          }
        }
      }
    }
  };

  // ------------------------------------------------ P' = p * s_v (B of PV)
  // p = 2^(s - m) of the step's logits; l += p
  auto pprime = [&](uint32_t pg, int t0, auto full_c, int n_valid, const SL& sl, SP& sp) {
    constexpr bool FULL = decltype(full_c)::value;
    const float* sc0 = sl.s0;
    const float* sc1 = sl.s1;
    auto& pb = sp.b;
    float pr[NTQ], pr8[NTQ];
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      const float mref = (PF && m[tq] == -INFINITY) ? 0.0f : m[tq];   // all masked: p = 0
      pr[tq] = ex2(sc0[tq] - mref);
      pr8[tq] = ex2(sc1[tq] - mref);
      l[tq] += pr[tq] + pr8[tq];
    }
    const int T0 = t0 + 2 * j;
    float x0[NTQ], x1[NTQ], x2[NTQ], x3[NTQ];
    {
      // B element (token T, column r) comes from QK lane 4*(T%8) + head%4
      const int hl = PSPLIT ? (r >> 1) : (r & 3);
      const int srcA = 8 * j + hl, srcB = 8 * j + 4 + hl;
#pragma unroll
      for (int tq = 0; tq < NTQ; ++tq) {
        x0[tq] = __shfl_sync(kFull, pr[tq], srcA);
        x1[tq] = __shfl_sync(kFull, pr[tq], srcB);
        x2[tq] = __shfl_sync(kFull, pr8[tq], srcA);
        x3[tq] = __shfl_sync(kFull, pr8[tq], srcB);
      }
    }
    const bool v0 = FULL || T0 < n_valid, v1 = FULL || T0 + 1 < n_valid,
               v2 = FULL || T0 + 8 < n_valid, v3 = FULL || T0 + 9 < n_valid;
    // Columns of padded heads (>= G) carry finite values (their q1 is zero)
    // and are never stored, so only invalid tokens are masked (their scale
    // bytes are stale stage contents).
    if constexpr (PSPLIT) {
      float sv0[NB], sv1[NB], sv2[NB], sv3[NB];
      {
        const uint32_t a = pg + (uint32_t)(t0 * BPT) + vs_lane;
        if constexpr (ASYM) {
          float zv0[NB], zv1[NB], zv2[NB], zv3[NB];
          SDec::template two_sz<0>(a, sv0, sv1, zv0, zv1);
          SDec::template two_sz<8 * BPT>(a, sv2, sv3, zv2, zv3);
          // sum_t p_t z_v[t, block] for this lane's column (invalid tokens: 0,
          // their scale bytes are stale stage contents)
#pragma unroll
          for (int tp = 0; tp < NTP; ++tp)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              float zs = v0 ? x0[tp] * zv0[b] : 0.0f;
              zs = v1 ? fmaf(x1[tp], zv1[b], zs) : zs;
              zs = v2 ? fmaf(x2[tp], zv2[b], zs) : zs;
              zs = v3 ? fmaf(x3[tp], zv3[b], zs) : zs;
              zacc[tp % (ASYM ? NTP : 1)][b % (ASYM ? NB : 1)] += zs;
            }
        } else {
          SDec::template two<0>(a, sv0, sv1);
          SDec::template two<8 * BPT>(a, sv2, sv3);
        }
      }
      // hi column (r even): fp16(y); lo column (r odd): fp16(y - fp16(y)),
      // the difference exact in fp32 -- one rounding of y - m * fp16(y)
      const float m_lo = (r & 1) ? 1.0f : 0.0f;
#pragma unroll
      for (int tp = 0; tp < NTP; ++tp) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const float y0 = v0 ? x0[tp] * sv0[b] : 0.0f;
          const float y1 = v1 ? x1[tp] * sv1[b] : 0.0f;
          const float y2 = v2 ? x2[tp] * sv2[b] : 0.0f;
          const float y3 = v3 ? x3[tp] * sv3[b] : 0.0f;
          const float2 f01 = __half22float2(__floats2half2_rn(y0, y1));
          const float2 f23 = __half22float2(__floats2half2_rn(y2, y3));
          pb[b][tp][0] = pack_half2(fmaf(-m_lo, f01.x, y0), fmaf(-m_lo, f01.y, y1));
          pb[b][tp][1] = pack_half2(fmaf(-m_lo, f23.x, y2), fmaf(-m_lo, f23.y, y3));
        }
      }
    } else {
      // P' = fp16(p * s_v): one rounding of the fp32 product
      float sv0[NB], sv1[NB], sv2[NB], sv3[NB];
      {
        const uint32_t a = pg + (uint32_t)(t0 * BPT) + vs_lane;
        SDec::template two<0>(a, sv0, sv1);
        SDec::template two<8 * BPT>(a, sv2, sv3);
      }
#pragma unroll
      for (int tp = 0; tp < NTP; ++tp) {
        float y0 = x0[0], y1 = x1[0], y2 = x2[0], y3 = x3[0];
        if constexpr (NTQ > 1) {
          const int tsel = (8 * tp + r) >> 2;   // < NTQ
#pragma unroll
          for (int tq = 1; tq < NTQ; ++tq) {
            const bool sel = tq == tsel;
            y0 = sel ? x0[tq] : y0;
            y1 = sel ? x1[tq] : y1;
            y2 = sel ? x2[tq] : y2;
            y3 = sel ? x3[tq] : y3;
          }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if constexpr (FULL) {
            pb[b][tp][0] = pack_half2(y0 * sv0[b], y1 * sv1[b]);
            pb[b][tp][1] = pack_half2(y2 * sv2[b], y3 * sv3[b]);
          } else {
            pb[b][tp][0] = pack_half2(v0 ? y0 * sv0[b] : 0.0f, v1 ? y1 * sv1[b] : 0.0f);
            pb[b][tp][1] = pack_half2(v2 ? y2 * sv2[b] : 0.0f, v3 ? y3 * sv3[b] : 0.0f);
          }
        }
      }
    }
  };

  // ------------------------------------------------ o1^T += V^T P'^T
  auto pv = [&](uint32_t pg, int t0, const SP& sp) {
    const auto& pb = sp.b;
    const uint32_t vt = pg + (uint32_t)(t0 * CB) + v_lane;   // token t0 + 2j
    static_for<NB>([&](auto bc) {
      constexpr int b = decltype(bc)::value;
      constexpr int O = b * KBB;
      // this lane's value chunks of tokens T0, T0+1, T0+8, T0+9 (at bit 0)
      uint32_t c0v, c1v, c2v, c3v;
      if constexpr (32 % VBITS == 0) {   // a chunk never crosses a word
        c0v = lds32<O>(vt) >> vshf;
        c1v = lds32<O + CB>(vt) >> vshf;
        c2v = lds32<O + 8 * CB>(vt) >> vshf;
        c3v = lds32<O + 9 * CB>(vt) >> vshf;
      } else {
        c0v = __funnelshift_r(lds32<O>(vt), lds32<O + 4>(vt), vshf);
        c1v = __funnelshift_r(lds32<O + CB>(vt), lds32<O + CB + 4>(vt), vshf);
        c2v = __funnelshift_r(lds32<O + 8 * CB>(vt), lds32<O + 8 * CB + 4>(vt), vshf);
        c3v = __funnelshift_r(lds32<O + 9 * CB>(vt), lds32<O + 9 * CB + 4>(vt), vshf);
      }
      static_for<KSB>([&](auto mpc) {
        constexpr int mp = decltype(mpc)::value;
        uint32_t af[4];
        af[0] = v_field<NBIT, 2 * mp, ASYM>(c0v, c1v, vsg0, vsg1, vsg2);
        af[1] = v_field<NBIT, 2 * mp + 1, ASYM>(c0v, c1v, vsg0, vsg1, vsg2);
        af[2] = v_field<NBIT, 2 * mp, ASYM>(c2v, c3v, vsg0, vsg1, vsg2);
        af[3] = v_field<NBIT, 2 * mp + 1, ASYM>(c2v, c3v, vsg0, vsg1, vsg2);
#pragma unroll
        for (int tp = 0; tp < NTP; ++tp) mma_16816(acc[b * KSB + mp][tp], af, pb[b][tp][0], pb[b][tp][1]);
      });
    });
  };

  const int P = g.page_size;
  int stage = 0;          // i mod S
  uint32_t parity = 0;    // (i / S) mod 2
  int prev = S - 1;       // (i - 1) mod S
  for (int64_t i = 0; i < nch; ++i) {
    if (!mbar_wait(&full[stage], parity, p.wait_limit) && lane == 0) *abort_s = 1;
    // One barrier per chunk: the four warps have finished chunk i - 1 and
    // waited for chunk i.  They decide together whether to go on (every
    // barrier below is then reached by all of them), and the stage of chunk
    // i - 1 is free: warp (i - 1) mod 4 refills it with chunk i - 1 + S.
    // Keeping the warps within one chunk of each other gives every warp the
    // ring's lookahead (a fast warp would otherwise wait on a refill that
    // only the slowest warp can trigger).
    named_barrier(2, 32 * kWarps);
    if (*abort_s) {
      // A copy did not arrive within the bound: flag it, wait for every copy
      // this CTA still has in flight so that no asynchronous write outlives
      // it, and stop.  In flight: chunk i itself (the one that ran out) up to
      // the last chunk issued, S - 1 from the prologue at i = 0, else i + S - 2
      // (the refill of iteration i - 1).  The drain has its own bound,
      // independent of the caller's wait limit.
      if (threadIdx.x == 0) set_status(p.status, KVQ3_DEV_TIMEOUT);
      const int64_t last = i == 0 ? (int64_t)S - 1 : i + S - 2;
      for (int64_t k = i; k < nch && k <= last; ++k)
        mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), kDrainPolls);
      return;
    }
    if (i > 0 && (((int)i - 1) & (kWarps - 1)) == wid && i - 1 + S < nch) {
      // chunk i - 1 + S; within the same sequence no global read is needed
      // (the descriptor carries nc and the length)
      const uint32_t sp = stg_u32 + (uint32_t)prev * p.stage_bytes;
      const uint4 pv = lds128<0>(sp + desc_off);      // unit, b, kvh, n_tok
      const uint4 px = lds128<16>(sp + desc_off);     // page_ok, c, nc, len
      Cursor c{(int)pv.y, (int)pv.z, (int64_t)px.y, (int64_t)px.z};
      const int b_now = c.b;
      for (int k = 0; k < S; ++k) cursor_next(p, c);
      const int64_t len = c.b == b_now ? (int64_t)px.w : seq_len_checked(p, c.b, false);
      fence_proxy_async();
      issue(c, prev, len);
    }
    const uint32_t st = stg_u32 + (uint32_t)stage * p.stage_bytes;
    const uint4 dv = lds128<0>(st + desc_off);            // unit, b, kvh, n_tok
    const uint2 dw = lds64<16>(st + desc_off);            // page_ok, c
    const int unit = (int)dv.x, n_tok = (int)dv.w;
    const uint32_t page_ok = dw.x;
    if (unit != cur_unit) {
      if (cur_unit >= 0) flush(cur_unit, cur_first, cur_last);
      setup_unit((int)dv.y, (int)dv.z);
      cur_unit = unit;
      cur_first = dw.y == 0;
    }
    cur_last = (int)dw.y == (int)lds32<24>(st + desc_off) - 1;   // c == nc - 1
    if (!PF && n_tok == p.chunk_tokens && page_ok == (1u << p.pages_per_chunk) - 1u &&
        p.chunk_tokens % (16 * kWarps) == 0 &&
        KVQ3_CHECK(p.status, in_range(SM::kStageOff + (int64_t)stage * p.stage_bytes,
                                      (int64_t)p.pages_per_chunk * 2 * REC + 16, p.smem_bytes))) {
      // A whole chunk: the warp's steps t = 16 wid + 64 k, software-pipelined
      // so that P' and PV of step k and the logits of step k + 1 form one
      // branch-free stretch (the running-max update follows PV of step k).
      const int nsw = p.chunk_tokens / (16 * kWarps);
      int pi = 0, tin = wid * 16;                       // page of the chunk, offset in it
      while (tin >= P) {
        tin -= P;
        ++pi;
      }
      uint32_t pg = st + (uint32_t)pi * 2 * REC;
      int t0 = tin;
      SL sa;
      logits(pg, t0, std::true_type{}, P, 0, sa);
      update(sa);
      for (int k = 1; k < nsw; ++k) {
        tin += 16 * kWarps;
        while (tin >= P) {
          tin -= P;
          ++pi;
        }
        const uint32_t pgn = st + (uint32_t)pi * 2 * REC;
        SP pb;
        pprime(pg, t0, std::true_type{}, P, sa, pb);
        SL sb;
        logits(pgn, tin, std::true_type{}, P, 0, sb);
        pv(pg, t0, pb);
        update(sb);
        pg = pgn;
        t0 = tin;
        sa = sb;
      }
      SP pb;
      pprime(pg, t0, std::true_type{}, P, sa, pb);
      pv(pg, t0, pb);
    } else {
      for (int t = wid * 16; t < n_tok; t += kWarps * 16) {
        int pi = 0, tin = t;                            // page of the chunk, offset in it
        while (tin >= P) {
          tin -= P;
          ++pi;
        }
        if (((page_ok >> pi) & 1u) &&
            KVQ3_CHECK(p.status, pi < p.pages_per_chunk && tin + 16 <= P &&
                                     in_range(SM::kStageOff + (int64_t)stage * p.stage_bytes + (int64_t)(pi + 1) * 2 * REC,
                                              0, p.smem_bytes))) {
          const uint32_t pg = st + (uint32_t)pi * 2 * REC;
          const int nv = min(P, n_tok - pi * P);        // valid tokens of this page
          const int64_t tok = (int64_t)dw.y * p.chunk_tokens + t;
          SL sc;
          SP pb;
          if (nv - tin >= 16) {
            logits(pg, tin, std::true_type{}, nv, tok, sc);
            update(sc);
            pprime(pg, tin, std::true_type{}, nv, sc, pb);
          } else {
            logits(pg, tin, std::false_type{}, nv, tok, sc);
            update(sc);
            pprime(pg, tin, std::false_type{}, nv, sc, pb);
          }
          pv(pg, tin, pb);
        }
      }
    }
    prev = stage;
    if (++stage == S) {
      stage = 0;
      parity ^= 1u;
    }
  }
  if (cur_unit >= 0) flush(cur_unit, cur_first, cur_last);
}

// ------------------------------------------------------------------ kernel 2
// Merge the partials of each (sequence, query head) and rotate back by U^T.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const __grid_constant__ DecodeParams p,
                                                             const __grid_constant__ RotParams rp,
                                                             float* __restrict__ out) {
  constexpr int E = D >= 128 ? D / 32 : 4;
  constexpr int L = D / E;
  const int lane = threadIdx.x & 31;
  const int rr = lane % L, grp = lane / L;
  const uint32_t sgn = lane_signs<E>(rp, rr);
  float4 qt[E / 4], qtr[E / 4];
  lane_quats<E>(rp, rr, qt);
  lane_quats_r<E>(rp, rr, qtr);
  const bool so4 = rot_so4(rp), pair = rot_pair(rp);
  // launched as a programmatic dependent of the split kernel: everything above
  // overlaps its tail; its partials are complete and visible after this
  griddep_wait();
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
  // output row it = (sequence or query token) * Hq + query head
  const int items = (p.pf_n > 0 ? p.pf_n : p.g.batch) * p.Hq;
  for (int it = warp; it < items; it += nwarps) {
    int b, h, kvh, gh;   // unit sequence (prefill: query tile), head, kv head, column
    if (p.pf_n > 0) {
      const int i = it / p.Hq;
      h = it - i * p.Hq;
      kvh = h / p.pf_gkv;
      const int hd = h - kvh * p.pf_gkv, hb = hd / p.pf_hpb;
      const int tb = i / p.pf_qt;
      b = tb * p.pf_hb + hb;
      gh = (i - tb * p.pf_qt) * p.pf_hpb + (hd - hb * p.pf_hpb);
    } else {
      b = it / p.Hq;
      h = it - b * p.Hq;
      kvh = h / p.G;
      gh = h - kvh * p.G;
    }
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.0f;
    if (seq_len_checked(p, b, false) > 0) {
      const int unit = b * p.g.hkv + kvh;
      // the consecutive CTAs that hold the unit's chunks (clamped: a CTA that
      // gave up on a copy may not have recorded itself; the status says so)
      const int last_cta = p.ctas - 1;
      const int wlo = min(max(p.unit_cta[2 * unit], 0), last_cta);
      int whi = min(max(p.unit_cta[2 * unit + 1], 0), last_cta);
      float M = -INFINITY;
      if (!KVQ3_CHECK(p.status, whi + unit < p.slots)) whi = wlo - 1;   // checked builds: no slot past the end
      for (int w = wlo; w <= whi; ++w) {
        const float* slot = p.ws + (size_t)(w + unit) * p.slot_floats;
        M = fmaxf(M, slot[p.G * D + gh]);
      }
      if (M != -INFINITY) {
        float lsum = 0.0f;
        for (int w = wlo; w <= whi; ++w) {
          const float* slot = p.ws + (size_t)(w + unit) * p.slot_floats;
          const float c = ex2(slot[p.G * D + gh] - M);
          lsum += c * slot[p.G * D + p.G + gh];
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] += c * slot[gh * D + rr * E + e];
        }
        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] *= inv;
      }
    }
    rotate_inverse<E, L>(o, rr, sgn, qt, qtr, p.inv_sqrt_d, so4, pair);
    if (grp == 0) {
#pragma unroll
      for (int e = 0; e < E; ++e) out[(int64_t)it * D + rr * E + e] = o[e];
    }
  }
}

// ------------------------------------------------------------------ host
struct DecodePlan {
  int gpad;
  int ctas;
  int stages;
  int chunk_tokens, pages_per_chunk;
  uint32_t stage_bytes, smem;
  size_t ws_bytes;
};

template <int D, int BLOCK, int GPAD, int SCALE, int NBIT, bool PSPLIT, bool PF = false>
kvq3_status decode_plan_t(const CacheGeom& g, int G, DecodePlan* plan) {
  using SM = DecodeSmem<D, GPAD>;
  const void* k = reinterpret_cast<const void*>(&decode_split_kernel<D, BLOCK, GPAD, SCALE, NBIT, PSPLIT, PF>);
  plan->gpad = GPAD;
  // the SM's 228 KB of shared memory split over the CTAs that the register
  // budget lets reside (1 KB of it reserved per CTA)
  const int mb = decode_min_blocks(D, GPAD);
  const size_t per_cta = 228 * 1024 / mb - 1024 < 227 * 1024 ? 228 * 1024 / mb - 1024 : 227 * 1024;
  // + 16: word reads past the last code string; + descriptor at the end
  auto stage_of = [&](int ppc) {
    return (uint32_t)(((size_t)ppc * 2 * g.record_bytes + 16 + sizeof(ChunkDesc) + 127) / 128 * 128);
  };
  // Chunk: the pages of kChunk tokens, fewer where two stages of them would
  // not fit in a CTA's share (one CTA fewer per SM costs more than a shorter
  // chunk), preferring a whole number of 64-token rounds (4 warps x 16
  // tokens) so that no warp idles at the chunk barrier.
  {
    const int most = (kChunk + g.page_size - 1) / g.page_size;
    int fit = 0, even = 0;
    for (int n = most; n >= 1 && even == 0; --n) {
      if (SM::kStageOff + 2 * (size_t)stage_of(n) > per_cta) continue;
      if (fit == 0) fit = n;
      if ((n * g.page_size) % (16 * kWarps) == 0) even = n;
    }
    plan->pages_per_chunk = even ? even : (fit ? fit : 1);
  }
  plan->chunk_tokens = plan->pages_per_chunk * g.page_size;
  plan->stage_bytes = stage_of(plan->pages_per_chunk);
  // stages: as many as fit in the CTA's share; at least 2
  int stages = per_cta > SM::kStageOff ? (int)((per_cta - SM::kStageOff) / plan->stage_bytes) : 0;
  stages = stages < 2 ? 2 : (stages > kMaxStages ? kMaxStages : stages);
  const size_t smem = SM::kStageOff + (size_t)stages * plan->stage_bytes;
  if (smem > 227 * 1024) return KVQ3_ERR_UNSUPPORTED;  // pages too large for a two-stage ring
  plan->stages = stages;
  plan->smem = (uint32_t)smem;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return KVQ3_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 32 * kWarps, smem) != cudaSuccess)
    return KVQ3_ERR_CUDA;
  if (per_sm < 1) return KVQ3_ERR_UNSUPPORTED;
  plan->ctas = sm_count() * per_sm;
  const size_t slots = (size_t)plan->ctas + (size_t)g.batch * g.hkv;
  // partial slots, then [units][2] int32 first/last CTA of each unit
  plan->ws_bytes = slots * (size_t)G * (D + 2) * sizeof(float) + (size_t)g.batch * g.hkv * 2 * sizeof(int32_t);
  return KVQ3_OK;
}

template <int D, int BLOCK, int GPAD, int SCALE, int NBIT, bool PSPLIT, bool PF = false>
kvq3_status decode_run_t(const DecodePlan& plan, DecodeParams prm, const RotParams& rp, float* out,
                         cudaStream_t st) {
  prm.stages = plan.stages;
  prm.stage_bytes = plan.stage_bytes;
  prm.chunk_tokens = plan.chunk_tokens;
  prm.pages_per_chunk = plan.pages_per_chunk;
  prm.ctas = plan.ctas;
  prm.smem_bytes = plan.smem;
  prm.slots = (int64_t)plan.ctas + (int64_t)prm.g.batch * prm.g.hkv;
  // Both kernels are programmatic dependents of what precedes them on the
  // stream: the split kernel's launch overlaps the preceding kernel (the
  // token write) and the combine's the split kernel's last CTAs; each waits
  // on the preceding grid before its first read.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.ctas);
  cfg.blockDim = dim3(32 * kWarps);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_split_kernel<D, BLOCK, GPAD, SCALE, NBIT, PSPLIT, PF>, prm, rp) !=
      cudaSuccess)
    return KVQ3_ERR_CUDA;
  const int64_t items = (int64_t)(prm.pf_n > 0 ? prm.pf_n : prm.g.batch) * prm.Hq;
  int64_t blocks = (items + 7) / 8;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap > 0 ? cap : 1;
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  if (cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, prm, rp, out) != cudaSuccess) return KVQ3_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ3_OK : KVQ3_ERR_CUDA;
}

// Per-(head dim, scale type, code width) entry points, one translation unit each.
#define KVQ3_DECODE_DECL1(D, SN, NB)                                                          \
  kvq3_status decode_plan_d##D##_##SN##_b##NB(const CacheGeom& g, int G, DecodePlan* plan);  \
  kvq3_status decode_run_d##D##_##SN##_b##NB(const DecodePlan&, const DecodeParams&,          \
                                             const RotParams&, float*, cudaStream_t);         \
  kvq3_status prefill_plan_d##D##_##SN##_b##NB(const CacheGeom& g, int G, DecodePlan* plan); \
  kvq3_status prefill_run_d##D##_##SN##_b##NB(const DecodePlan&, const DecodeParams&,         \
                                              const RotParams&, float*, cudaStream_t);
#define KVQ3_DECODE_DECL(D, SN) KVQ3_DECODE_DECL1(D, SN, 2) KVQ3_DECODE_DECL1(D, SN, 3) KVQ3_DECODE_DECL1(D, SN, 4)
KVQ3_DECODE_DECL(64, f32) KVQ3_DECODE_DECL(64, f16) KVQ3_DECODE_DECL(64, e4m3)
KVQ3_DECODE_DECL(128, f32) KVQ3_DECODE_DECL(128, f16) KVQ3_DECODE_DECL(128, e4m3)
KVQ3_DECODE_DECL(256, f32) KVQ3_DECODE_DECL(256, f16) KVQ3_DECODE_DECL(256, e4m3)
KVQ3_DECODE_DECL1(64, e4m3zp, 3) KVQ3_DECODE_DECL1(128, e4m3zp, 3) KVQ3_DECODE_DECL1(256, e4m3zp, 3)

// P' split into hi + lo halves for fp32 value scales (p times an fp32 scale is
// not an fp16 value) and for up to 4 heads per kv head, where the split
// columns fit the same 8-column PV tile (no extra MMAs) and remove the fp16
// rounding of P' from the error.
#define KVQ3_DECODE_PICK(D, BLK, SC, NB, FN, ...)                                             \
  {                                                                                           \
    constexpr bool SPLIT = (SC) == KVQ3_SCALE_F32 || (SC) == KVQ3_SCALE_E4M3_ZP;              \
    if (gp == 4) return FN<D, BLK, 4, SC, NB, true>(__VA_ARGS__);                             \
    if (gp == 8) return FN<D, BLK, 8, SC, NB, SPLIT>(__VA_ARGS__);                            \
    return FN<D, BLK, 16, SC, NB, SPLIT>(__VA_ARGS__);                                        \
  }

#define KVQ3_DECODE_INSTANCES(D, SN, SC, NB)                                                  \
  kvq3_status decode_plan_d##D##_##SN##_b##NB(const CacheGeom& g, int G, DecodePlan* plan) { \
    const int gp = G <= 4 ? 4 : (G <= 8 ? 8 : 16);                                            \
    if (g.block == 32) KVQ3_DECODE_PICK(D, 32, SC, NB, decode_plan_t, g, G, plan)             \
    KVQ3_DECODE_PICK(D, 64, SC, NB, decode_plan_t, g, G, plan)                                \
  }                                                                                           \
  kvq3_status decode_run_d##D##_##SN##_b##NB(const DecodePlan& plan, const DecodeParams& prm, \
                                             const RotParams& rp, float* out, cudaStream_t st) { \
    const int gp = plan.gpad;                                                                 \
    if (prm.g.block == 32) KVQ3_DECODE_PICK(D, 32, SC, NB, decode_run_t, plan, prm, rp, out, st) \
    KVQ3_DECODE_PICK(D, 64, SC, NB, decode_run_t, plan, prm, rp, out, st)                     \
  }                                                                                           \
  /* chunked prefill: 8 logit columns = query tokens x a block of query heads of a kv head, \
     with P' split into hi + lo halves (the many outputs of a prefill chunk leave the  \
     single fp16 rounding of P' too close to the tolerance) */                         \
  kvq3_status prefill_plan_d##D##_##SN##_b##NB(const CacheGeom& g, int G, DecodePlan* plan) { \
    if (g.block == 32) return decode_plan_t<D, 32, 8, SC, NB, true, true>(g, G, plan);        \
    return decode_plan_t<D, 64, 8, SC, NB, true, true>(g, G, plan);                           \
  }                                                                                           \
  kvq3_status prefill_run_d##D##_##SN##_b##NB(const DecodePlan& plan, const DecodeParams& prm, \
                                              const RotParams& rp, float* out, cudaStream_t st) { \
    if (prm.g.block == 32) return decode_run_t<D, 32, 8, SC, NB, true, true>(plan, prm, rp, out, st); \
    return decode_run_t<D, 64, 8, SC, NB, true, true>(plan, prm, rp, out, st);                \
  }

}  // namespace kvq3
