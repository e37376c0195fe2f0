// Chunked-prefill attention over the packed cache on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory): head dimension 128, 3-bit
// symmetric codes, quantisation blocks of 64.
//
// "Orthogonally mixed 3-bit KV cache", Implementation notes (read path) and
// Key formulas, with the causal mask of a prefill chunk: query token i sits at
// position pos0 + i and attends to positions [0, pos0 + i] of its sequence.
// "Orthogonal Invariance in Activation Space", sections 4.1 and 4.3: the cache
// is read with dequantisation fused into the attention products.
//
// One CTA = 128 query rows of one kv head (a row is a (query token, query
// head) pair: 128 / G tokens x G heads), one row per TMEM lane.  It walks the
// sequence in 64-key tiles up to its last row's position.
//
// Arithmetic.  q1 = U q is scaled by sm_scale * log2(e) and a per-row power
// of two and kept as hi + lo fp16 halves.  Key codes enter the products as
// exact small fp16 integers, one accumulator per 64-dimension scale block:
//   S_b = (q1_hi + q1_lo)[block b] . c_k[block b]       (two MMAs per k-step)
// and the key scales are applied in fp32 afterwards: s = S_0 k_0 + S_1 k_1.
// The online softmax (base 2, lazy rescaling: the running maximum moves only
// when a row's maximum grows by more than 2^8) gives p <= 2^8, kept as hi + lo
// fp16 halves.  A value's scale is split as s_v = s_hi + s_lo with s_hi its
// top 9 significant bits, so that c * s_hi and c * s_lo (|c| <= 4) are exact
// fp16 numbers and
//   O += p_hi . (c s_hi) + p_lo . (c s_hi) + p_hi . (c s_lo)
// over full 128-dimension rows (the dropped p_lo . (c s_lo) is below 2^-20 of
// the product; E4M3 scales have s_lo = 0 and skip the third MMA).  Dequantised
// values must lie in the fp16 range, as for every kernel of this library.
//
// Roles (9 warps):
//  * warps 0-3, softmax: thread = row.  tcgen05.ld of S, scales, mask, online
//    softmax, p_hi / p_lo written back over S with tcgen05.st (the A operand
//    of PV), rare rescales of O in place;
//  * warps 4-7, dequantisation: thread = (key, half of the dimensions).  Thread
//    0 issues the bulk copies of packed codes and scales into a ring of raw
//    stages; all unpack a tile into the MMA layouts in shared memory: integer
//    key codes K-major, values c*s_hi and c*s_lo MN-major;
//  * warp 8, lane 0: issues QK^T of tile t, then PV of tile t - 1.
// TMEM: q1 hi / lo (128 columns), two S/P buffers (128 each), O (128).
// Every hand-off is an mbarrier; every wait is bounded (a time-out sets
// KVQ3_DEV_TIMEOUT and the CTA winds down: MMAs and copies in flight are
// drained and TMEM freed before it exits).
#include <string.h>

#include "kvq3_internal.h"
#include "kvq3_tc.cuh"

using namespace kvq3;

namespace {

constexpr int kRows = 128;            // query rows per CTA = TMEM lanes
constexpr int kKeys = 64;             // keys per tile
constexpr int kD = 128;               // head dimension
constexpr int kCB = 3 * kD / 8;       // code bytes per vector (48)
constexpr int kStages = 4;            // raw stages in flight
constexpr int kThreads = 9 * 32;
constexpr int kMmaThread = 8 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColSP = 128, kColO = 384;   // TMEM column map
constexpr float kRescale = 8.0f;      // log2 of the largest p between rescales

// shared memory (bytes)
constexpr int kTile = kKeys * kD * 2;                          // one fp16 tile (16 KB)
constexpr int kOffK = 0;                                       // [2] key codes, K-major
constexpr int kOffV = kOffK + 2 * kTile;                       // [2][hi, lo] values, MN-major
constexpr int kRawK = 0, kRawV = kKeys * kCB;                  // raw stage: codes K, V
constexpr int kRawKs = 2 * kKeys * kCB, kRawVs = kRawKs + kKeys * 2 * 4;   // scales K, V (<= 8 B a key)
constexpr int kRawBytes = kRawVs + kKeys * 2 * 4;              // 7168
constexpr int kOffRaw = kOffV + 4 * kTile;
constexpr int kOffKs = kOffRaw + kStages * kRawBytes;          // [2][2 blocks][64] fp32 key scales
constexpr int kPitch = kD + 1;                                 // row staging pitch (floats)
constexpr int kOffRows = kOffKs + 2 * 2 * kKeys * 4;           // [128][129] fp32 rows
constexpr int kOffQinv = kOffRows + kRows * kPitch * 4;        // [128] fp32
constexpr int kNumBars = 2 * kStages + 11;
constexpr int kOffBars = kOffQinv + kRows * 4;
constexpr int kOffMisc = kOffBars + kNumBars * 8;              // TMEM base, abort flag, masks
constexpr int kSmem = kOffMisc + 16 + (kStages + 2) * 8;
static_assert(kOffRaw % 16 == 0 && kRawBytes % 16 == 0 && kOffBars % 8 == 0, "alignment");
static_assert(kSmem <= 227 * 1024, "shared memory");

struct TcParams {
  CacheGeom g;
  const uint8_t* pool;
  const int32_t* page_table;
  const __half* q;      // [n][Hq][128]
  float* out;           // [n][Hq][128]
  int32_t* status;
  int32_t seq, n, Hq, G, qb;   // qb: query tokens per CTA (128 / G)
  int64_t pos0;
  float qk_scale;       // sm_scale * log2(e)
  float inv_sqrt_d;
  uint32_t wait_limit;
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// 1-D bulk copy global -> shared counted on an mbarrier (default L2 policy:
// every kv head's tiles are read by all the query blocks of that head).
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// two 3-bit two's-complement fields (bits 0-2 and 3-5 of w6) -> half2 of the
// exact integers: (0x6400 | (c + 4)) - 1028
__device__ __forceinline__ __half2 codes2(uint32_t w6) {
  const uint32_t h = (((w6 & 63u) * 0x2001u) & 0x00070007u) ^ 0x64046404u;
  return __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6404), __ushort_as_half(0x6404)));
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

template <int SCALE>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p,
                                                                  const __grid_constant__ RotParams rp) {
  constexpr int SB = SCALE == KVQ3_SCALE_F32 ? 4 : SCALE == KVQ3_SCALE_F16 ? 2 : 1;
  constexpr bool kLo = SCALE != KVQ3_SCALE_E4M3;   // values carry a low part of the scale
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* raw_full = bars;                   // [kStages] bulk copies landed
  uint64_t* raw_empty = bars + kStages;        // [kStages] dequantisation done with a stage
  uint64_t* k_full = bars + 2 * kStages;       // [2] key tile and key scales ready
  uint64_t* v_full = k_full + 2;               // [2] value tiles ready
  uint64_t* s_full = v_full + 2;               // [2] S of the tile in TMEM
  uint64_t* p_full = s_full + 2;               // [2] P of the tile in TMEM (and O rescaled)
  uint64_t* pv_done = p_full + 2;              // [2] PV of the tile complete
  uint64_t* drain = pv_done + 2;               // every MMA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint64_t* stage_mask = reinterpret_cast<uint64_t*>(smem + kOffMisc + 16);   // [kStages] valid keys
  uint64_t* key_mask = stage_mask + kStages;                                  // [2]
  float* rows = reinterpret_cast<float*>(smem + kOffRows);
  float* qinv_s = reinterpret_cast<float*>(smem + kOffQinv);
  float* ks_s = reinterpret_cast<float*>(smem + kOffKs);

  const CacheGeom& g = p.g;
  const int kvh = blockIdx.y;
  const int qblk = (int)gridDim.x - 1 - (int)blockIdx.x;   // longest query blocks first
  const int t0 = qblk * p.qb;
  const int ntok = min(p.qb, p.n - t0);
  const int nrows = ntok * p.G;
  const int64_t kmax = p.pos0 + t0 + ntok - 1;             // last position any row attends to
  const int T = (int)(kmax / kKeys) + 1;                   // key tiles

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&k_full[b], 128);
      mbar_init(&v_full[b], 128);
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 128);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 8) tc::alloc(tmem_slot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  // bounded wait; a time-out (or another thread's) winds the CTA down
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    for (uint32_t it = 0; it < p.wait_limit; ++it) {
      if (mbar_try(bar, parity)) return true;
      if ((it & 31u) == 31u && *abort_flag) return false;
    }
    *abort_flag = 1u;
    set_status(p.status, KVQ3_DEV_TIMEOUT);
    return false;
  };

  // bulk copies of tile t (16-key groups; a page holds whole groups since P
  // is a multiple of 16) into its raw stage; called by dequant thread 0 only
  const int64_t pool_bytes = g.num_pages * g.page_bytes;
  (void)pool_bytes;   // read by the checked build only
  auto issue = [&](int t) {
    const int s = t % kStages;
    uint8_t* st = smem + kOffRaw + s * kRawBytes;
    const int64_t k0 = (int64_t)t * kKeys;
    int64_t gpage[4];
    uint64_t mask = 0;
    uint32_t bytes = 0;
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      const int64_t pos = k0 + 16 * gi;
      gpage[gi] = -1;
      if (pos > kmax) continue;
      const int64_t pg = page_of(g, p.page_table, p.seq, pos / g.page_size);
      if (pg < 0) {
        set_status(p.status, KVQ3_DEV_BAD_PAGE);
        continue;
      }
      gpage[gi] = pg;
      mask |= 0xFFFFull << (16 * gi);
      bytes += 16u * (2u * kCB + 2u * 2u * SB);
    }
    if (kmax - k0 < kKeys - 1) mask &= (1ull << (kmax - k0 + 1)) - 1ull;   // keys past the last row
    stage_mask[s] = mask;
    mbar_expect_tx(&raw_full[s], bytes);
    for (int gi = 0; gi < 4; ++gi) {
      if (gpage[gi] < 0) continue;
      int gj = gi;
      while (gj + 1 < 4 && gpage[gj + 1] == gpage[gi]) ++gj;   // consecutive groups of one page
      const uint32_t nk = 16u * (uint32_t)(gj - gi + 1);
      const int64_t slot = (k0 + 16 * gi) % g.page_size;
      const int64_t rk = record_offset(g, gpage[gi], kvh, 0), rv = record_offset(g, gpage[gi], kvh, 1);
      const int64_t ck = rk + g.scale_hdr_bytes + slot * kCB, cv = rv + g.scale_hdr_bytes + slot * kCB;
      const int64_t sk = rk + slot * 2 * SB, sv = rv + slot * 2 * SB;
      if (KVQ3_CHECK(p.status, in_range(ck, nk * kCB, pool_bytes) && in_range(cv, nk * kCB, pool_bytes) &&
                                   in_range(sk, nk * 2 * SB, pool_bytes) && in_range(sv, nk * 2 * SB, pool_bytes))) {
        bulk_copy(st + kRawK + 16 * gi * kCB, p.pool + ck, nk * kCB, &raw_full[s]);
        bulk_copy(st + kRawV + 16 * gi * kCB, p.pool + cv, nk * kCB, &raw_full[s]);
        bulk_copy(st + kRawKs + 16 * gi * 2 * SB, p.pool + sk, nk * 2 * SB, &raw_full[s]);
        bulk_copy(st + kRawVs + 16 * gi * 2 * SB, p.pool + sv, nk * 2 * SB, &raw_full[s]);
      } else {
        // checked build: the copies are skipped; complete the expected bytes
        // so that the stage still lands (its keys read as garbage, flagged)
        asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&raw_full[s])),
                     "r"(nk * (2u * kCB + 2u * 2u * SB))
                     : "memory");
      }
      gi = gj;
    }
  };
  int issued = 0;   // tiles whose copies dequant thread 0 has issued
  if (tid == 128)
    for (; issued < min(kStages - 1, T); ++issued) issue(issued);

  // ---- q1 = U q of the rows, scaled by qk_scale and a per-row power of two
  {
    const uint32_t sgn = lane_signs<4>(rp, lane);
    float4 qt[1], qtr[1];
    lane_quats<4>(rp, lane, qt);
    lane_quats_r<4>(rp, lane, qtr);
    const bool so4 = rot_so4(rp), pair = rot_pair(rp);
    for (int row = warp; row < kRows; row += kThreads / 32) {
      float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (row < nrows) {
        const int tok = t0 + row / p.G, h = kvh * p.G + row % p.G;
        const uint2 raw = *reinterpret_cast<const uint2*>(p.q + ((int64_t)tok * p.Hq + h) * kD + lane * 4);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        x[0] = a.x;
        x[1] = a.y;
        x[2] = b.x;
        x[3] = b.y;
      }
      rotate_forward<4, 32>(x, lane, sgn, qt, qtr, p.inv_sqrt_d, so4, pair);
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] *= p.qk_scale;
        amax = fmaxf(amax, fabsf(x[e]));
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      int ex = 0;
      if (amax > 0.0f) frexpf(amax, &ex);
      ex = max(-100, min(100, 8 - ex));                    // row maximum into (2^7, 2^8]
      const float sc = ldexpf(1.0f, ex);
#pragma unroll
      for (int e = 0; e < 4; ++e) rows[row * kPitch + lane * 4 + e] = x[e] * sc;
      if (lane == 0) qinv_s[row] = ldexpf(1.0f, -ex);
    }
  }
  __syncthreads();
  if (warp < 4) {   // row = thread: hi and lo halves into TMEM (q1_hi cols 0-63, q1_lo 64-127)
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t hv[32], lv[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float a = rows[tid * kPitch + 64 * hf + 2 * c], b = rows[tid * kPitch + 64 * hf + 2 * c + 1];
        const __half2 hi = __floats2half2_rn(a, b);
        const float2 f = __half22float2(hi);
        hv[c] = h2u(hi);
        lv[c] = h2u(__floats2half2_rn(a - f.x, b - f.y));
      }
      tc::st32(tmem + lanes + kColQ + 32 * hf, hv);
      tc::st32(tmem + lanes + kColQ + 64 + 32 * hf, lv);
    }
    tc::wait_st();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  if (warp < 4) {
    // ================================================================ softmax
    const int row = tid;
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
    const float qinv = qinv_s[row];
    const int64_t lim = row < nrows ? p.pos0 + t0 + row / p.G : -1;
    float m_used = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int b = t & 1;
      const uint32_t ph = (uint32_t)(t >> 1) & 1u;
      ok = __all_sync(kFull, wait(&s_full[b], ph) && wait(&k_full[b], ph));
      if (!ok) break;
      tc::fence_after();
      const uint32_t tS = tmem + lanes + kColSP + 128u * b;
      const uint64_t km = key_mask[b];
      const int64_t k0 = (int64_t)t * kKeys;
      const bool full = km == ~0ull && k0 + kKeys - 1 <= lim;
      float sv[kKeys];
#pragma unroll
      for (int h = 0; h < 2; ++h) {   // keys 32h .. 32h + 31
        uint32_t a[32], c[32];
        tc::ld32(tS + 32 * h, a);         // block 0
        tc::ld32(tS + 64 + 32 * h, c);    // block 1
        tc::wait_ld();
        tc::reg_fence(a);
        tc::reg_fence(c);
        const float2* k0s = reinterpret_cast<const float2*>(ks_s + (b * 2 + 0) * kKeys + 32 * h);
        const float2* k1s = reinterpret_cast<const float2*>(ks_s + (b * 2 + 1) * kKeys + 32 * h);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x0 = k0s[i], x1 = k1s[i];
          sv[32 * h + 2 * i] = fmaf(__uint_as_float(c[2 * i]), x1.x, __uint_as_float(a[2 * i]) * x0.x);
          sv[32 * h + 2 * i + 1] = fmaf(__uint_as_float(c[2 * i + 1]), x1.y, __uint_as_float(a[2 * i + 1]) * x0.y);
        }
      }
      if (!full) {
#pragma unroll
        for (int k = 0; k < kKeys; ++k)
          if (!((km >> k) & 1ull) || k0 + k > lim) sv[k] = -INFINITY;
      }
      float mx = sv[0];
#pragma unroll
      for (int k = 1; k < kKeys; ++k) mx = fmaxf(mx, sv[k]);
      const float xm = mx * qinv;
      const bool need = xm > m_used + kRescale;
      if (__any_sync(kFull, need)) {
        const float m_new = need ? xm : m_used;
        const float alpha = need ? (m_used == -INFINITY ? 0.0f : ex2(m_used - m_new)) : 1.0f;
        l *= alpha;
        if (t > 0) {   // O holds PV up to tile t - 1: wait for it, then scale it in place
          ok = __all_sync(kFull, wait(&pv_done[(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u));
          if (!ok) break;
          tc::fence_after();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t o[32];
            tc::ld32(tmem + lanes + kColO + 32 * c4, o);
            tc::wait_ld();
            tc::reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc::st32(tmem + lanes + kColO + 32 * c4, o);
          }
        }
        m_used = m_new;
      }
      const float moff = m_used == -INFINITY ? 0.0f : m_used;
      uint32_t hv[32], lv[32];
      float lsum = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ex2(fmaf(sv[2 * i], qinv, -moff)), p1 = ex2(fmaf(sv[2 * i + 1], qinv, -moff));
        lsum += p0 + p1;
        const __half2 hi = __floats2half2_rn(p0, p1);
        const float2 f = __half22float2(hi);
        hv[i] = h2u(hi);
        lv[i] = h2u(__floats2half2_rn(p0 - f.x, p1 - f.y));
      }
      l += lsum;
      tc::st32(tS, hv);        // P hi over the first S columns (already read)
      tc::st32(tS + 32, lv);   // P lo
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(&p_full[b]);
    }
    if (ok) ok = __all_sync(kFull, wait(&pv_done[(T - 1) & 1], (uint32_t)((T - 1) >> 1) & 1u));
    tc::fence_after();
    const float inv = (ok && l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t o[32];
      if (ok) {
        tc::ld32(tmem + lanes + kColO + 32 * c4, o);
        tc::wait_ld();
        tc::reg_fence(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) rows[row * kPitch + 32 * c4 + i] = __uint_as_float(o[i]) * inv;
    }
  } else if (warp < 8) {
    // ================================================================ dequantisation
    const int dt = tid - 128, key = dt >> 1, half = dt & 1;
    int waited = 0;   // thread 0: tiles whose copies it has seen land
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int s = t % kStages, b = t & 1;
      if (dt == 0 && issued < T) {   // refill the stage tile t - 1 used
        if (t >= 1) ok = wait(&raw_empty[issued % kStages], (uint32_t)((issued / kStages) - 1) & 1u);
        if (ok) issue(issued++);
      }
      ok = ok && wait(&raw_full[s], (uint32_t)(t / kStages) & 1u);
      if (dt == 0 && ok) waited = t + 1;
      const uint8_t* st = smem + kOffRaw + s * kRawBytes;
      const uint64_t vm = ok ? stage_mask[s] : 0ull;
      const bool kv = (vm >> key) & 1ull;
      // ---- keys: exact integer codes, K-major: (key, d) at (key/8)*2048 + (d/8)*128 + (key%8)*16 + (d%8)*2
      if (t >= 2) ok = ok && wait(&p_full[b], (uint32_t)((t - 2) >> 1) & 1u);
      if (ok) {
        const uint2* src = reinterpret_cast<const uint2*>(st + kRawK + key * kCB + half * 24);
        uint32_t w[7];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const uint2 u = src[i];
          w[2 * i] = u.x;
          w[2 * i + 1] = u.y;
        }
        w[6] = 0u;
        uint8_t* kt = smem + kOffK + b * kTile + (key >> 3) * 2048 + (key & 7) * 16;
#pragma unroll
        for (int gq = 0; gq < 8; ++gq) {
          const int bit = 24 * gq;
          const uint32_t w24 = __funnelshift_r(w[bit >> 5], w[(bit >> 5) + 1], bit & 31);
          uint4 o;
          o.x = h2u(codes2(w24));
          o.y = h2u(codes2(w24 >> 6));
          o.z = h2u(codes2(w24 >> 12));
          o.w = h2u(codes2(w24 >> 18));
          *reinterpret_cast<uint4*>(kt + (8 * half + gq) * 128) = o;
        }
        uint32_t bits;
        const uint8_t* sp = st + kRawKs + (key * 2 + half) * SB;
        if (SB == 4) bits = *reinterpret_cast<const uint32_t*>(sp);
        else if (SB == 2) bits = *reinterpret_cast<const uint16_t*>(sp);
        else bits = *sp;
        ks_s[(b * 2 + half) * kKeys + key] = kv ? decode_scale(bits, SCALE) : 0.0f;
        if (dt == 0) key_mask[b] = vm;
      }
      fence_proxy_async();
      mbar_arrive(&k_full[b]);
      // ---- values c * s_hi, c * s_lo, MN-major: (key, d) at (d/8)*1024 + (key/8)*128 + (key%8)*16 + (d%8)*2
      if (t >= 2) ok = ok && wait(&pv_done[b], (uint32_t)((t - 2) >> 1) & 1u);
      if (ok) {
        const uint2* src = reinterpret_cast<const uint2*>(st + kRawV + key * kCB + half * 24);
        uint32_t w[7];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const uint2 u = src[i];
          w[2 * i] = u.x;
          w[2 * i + 1] = u.y;
        }
        w[6] = 0u;
        uint32_t bits;
        const uint8_t* sp = st + kRawVs + (key * 2 + half) * SB;
        if (SB == 4) bits = *reinterpret_cast<const uint32_t*>(sp);
        else if (SB == 2) bits = *reinterpret_cast<const uint16_t*>(sp);
        else bits = *sp;
        const float sv = kv ? decode_scale(bits, SCALE) : 0.0f;
        const float s_hi = __uint_as_float(__float_as_uint(sv) & 0xFFFF8000u);   // top 9 significant bits
        const __half2 hs = __float2half2_rn(s_hi), ls = __float2half2_rn(sv - s_hi);
        uint8_t* vt = smem + kOffV + b * 2 * kTile + (key >> 3) * 128 + (key & 7) * 16;
#pragma unroll
        for (int gq = 0; gq < 8; ++gq) {
          const int bit = 24 * gq;
          const uint32_t w24 = __funnelshift_r(w[bit >> 5], w[(bit >> 5) + 1], bit & 31);
          const __half2 c0 = codes2(w24), c1 = codes2(w24 >> 6), c2 = codes2(w24 >> 12), c3 = codes2(w24 >> 18);
          uint4 o;
          o.x = h2u(__hmul2(c0, hs));
          o.y = h2u(__hmul2(c1, hs));
          o.z = h2u(__hmul2(c2, hs));
          o.w = h2u(__hmul2(c3, hs));
          *reinterpret_cast<uint4*>(vt + (8 * half + gq) * 1024) = o;
          if (kLo) {
            o.x = h2u(__hmul2(c0, ls));
            o.y = h2u(__hmul2(c1, ls));
            o.z = h2u(__hmul2(c2, ls));
            o.w = h2u(__hmul2(c3, ls));
            *reinterpret_cast<uint4*>(vt + kTile + (8 * half + gq) * 1024) = o;
          }
        }
      }
      fence_proxy_async();
      mbar_arrive(&v_full[b]);
      mbar_arrive(&raw_empty[s]);
    }
    if (dt == 0) {   // no bulk copy may still target this CTA's shared memory at exit
      for (int t = waited; t < issued; ++t)
        mbar_wait(&raw_full[t % kStages], (uint32_t)(t / kStages) & 1u, kDrainPolls);
    }
  } else if (tid == kMmaThread) {
    // ================================================================ MMA issue
    constexpr uint32_t kIdQK = tc::idesc_f16(128, kKeys, false);
    constexpr uint32_t kIdPV = tc::idesc_f16(128, kD, true);
    bool ok = true;
    for (int t = 0; t <= T && ok; ++t) {
      if (t < T) {   // S_b(t) = q1[block b] . c_k[block b], hi and lo halves of q1
        const int b = t & 1;
        ok = wait(&k_full[b], (uint32_t)(t >> 1) & 1u);
        if (ok && t >= 2) ok = wait(&pv_done[b], (uint32_t)((t - 2) >> 1) & 1u);   // P(t-2) consumed
        if (!ok) break;
        tc::fence_after();
        const uint32_t kb = smem_u32(smem + kOffK + b * kTile);
        const uint32_t dS = tmem + kColSP + 128u * b;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_ts(dS + 64u * blk, tmem + kColQ + 64u * part + 32u * blk + 8u * ks,
                         tc::sdesc(kb + (uint32_t)(blk * 8 + ks * 2) * 128u, 128u, 2048u), kIdQK,
                         (part | ks) != 0);
        tc::commit(&s_full[b]);
      }
      if (t >= 1) {   // O += P(t-1) V(t-1)
        const int tp = t - 1, b = tp & 1;
        ok = wait(&p_full[b], (uint32_t)(tp >> 1) & 1u) && wait(&v_full[b], (uint32_t)(tp >> 1) & 1u);
        if (!ok) break;
        tc::fence_after();
        const uint32_t vb = smem_u32(smem + kOffV + b * 2 * kTile);
        const uint32_t aP = tmem + kColSP + 128u * b;
#pragma unroll
        for (int pr = 0; pr < (kLo ? 3 : 2); ++pr)   // (p_hi, v_hi), (p_lo, v_hi), (p_hi, v_lo)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_ts(tmem + kColO, aP + (pr == 1 ? 32u : 0u) + 8u * ks,
                       tc::sdesc(vb + (pr == 2 ? (uint32_t)kTile : 0u) + (uint32_t)ks * 256u, 128u, 1024u), kIdPV,
                       !(tp == 0 && pr == 0 && ks == 0));
        tc::commit(&pv_done[b]);
      }
    }
    tc::commit(drain);   // whatever was issued completes before TMEM is freed
    mbar_wait(drain, 0u, kDrainPolls);
  }
  __syncthreads();

  // ---- outputs: rotate back with U^T (warp per row) and store
  {
    const uint32_t sgn = lane_signs<4>(rp, lane);
    float4 qt[1], qtr[1];
    lane_quats<4>(rp, lane, qt);
    lane_quats_r<4>(rp, lane, qtr);
    const bool so4 = rot_so4(rp), pair = rot_pair(rp);
    for (int row = warp; row < nrows; row += kThreads / 32) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = rows[row * kPitch + lane * 4 + e];
      rotate_inverse<4, 32>(x, lane, sgn, qt, qtr, p.inv_sqrt_d, so4, pair);
      const int tok = t0 + row / p.G, h = kvh * p.G + row % p.G;
      float4* dst = reinterpret_cast<float4*>(p.out + ((int64_t)tok * p.Hq + h) * kD + lane * 4);
      *dst = make_float4(x[0], x[1], x[2], x[3]);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 8) tc::dealloc(tmem, kTmemCols);
}

template <int SCALE>
kvq3_status launch_tc(const TcParams& p, const RotParams& rp, cudaStream_t st) {
  auto k = prefill_tc_kernel<SCALE>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return KVQ3_ERR_CUDA;
  const dim3 grid((unsigned)((p.n + p.qb - 1) / p.qb), (unsigned)p.g.hkv);
  k<<<grid, kThreads, kSmem, st>>>(p, rp);
  return cudaGetLastError() == cudaSuccess ? KVQ3_OK : KVQ3_ERR_CUDA;
}

}  // namespace

namespace kvq3 {

bool prefill_tc_supported(const CacheGeom& g, int32_t hq) {
  return g.d == kD && g.bits == 3 && g.block == 64 && g.scale_type != KVQ3_SCALE_E4M3_ZP && hq / g.hkv <= kRows;
}

// tcgen05 path of kvq3_prefill_attn; arguments already checked.
kvq3_status prefill_tc(const CacheGeom& g, const kvq3_cache* cache, int32_t seq, int64_t pos0, int64_t n_q,
                       const void* q, int32_t hq, float qk_scale, float* out, int32_t* dev_status,
                       const RotParams& rp, uint32_t wait_limit, cudaStream_t st) {
  if (!prefill_tc_supported(g, hq)) return KVQ3_ERR_UNSUPPORTED;
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.g = g;
  p.pool = static_cast<const uint8_t*>(cache->pool);
  p.page_table = cache->page_table;
  p.q = static_cast<const __half*>(q);
  p.out = out;
  p.status = dev_status;
  p.seq = seq;
  p.n = (int32_t)n_q;
  p.Hq = hq;
  p.G = hq / g.hkv;
  p.qb = kRows / p.G;
  p.pos0 = pos0;
  p.qk_scale = qk_scale;
  p.inv_sqrt_d = inv_sqrt(g.d);
  p.wait_limit = wait_limit;
  if (g.scale_type == KVQ3_SCALE_F32) return launch_tc<KVQ3_SCALE_F32>(p, rp, st);
  if (g.scale_type == KVQ3_SCALE_F16) return launch_tc<KVQ3_SCALE_F16>(p, rp, st);
  return launch_tc<KVQ3_SCALE_E4M3>(p, rp, st);
}

}  // namespace kvq3
