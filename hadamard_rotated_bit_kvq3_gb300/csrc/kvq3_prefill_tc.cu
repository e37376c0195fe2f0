// Chunked-prefill attention over the packed cache on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory): head dimension 128,
// quantisation blocks of 64, symmetric codes of b = 2, 3 or 4 bits or the
// asymmetric 3-bit codes (E4M3 scale and zero point).
//
// "Orthogonally mixed 3-bit KV cache", Implementation notes (read path) and
// Key formulas, with the causal mask of a prefill chunk: query token i sits at
// position pos0 + i and attends to positions [0, pos0 + i] of its sequence.
// "Orthogonal Invariance in Activation Space", sections 4.1 and 4.3: the cache
// is read with dequantisation fused into the attention products.
//
// A unit = 128 query rows of one kv head (a row is a (query token, query
// head) pair: 128 / G tokens x G heads), one row per TMEM lane.  Its keys are
// walked in 64-key tiles up to its last row's position: by one CTA, or, for a
// unit of at least kMinSplit tiles, by np CTAs over equal shares of the tiles
// (two, or one per kChain tiles, at most kMaxParts), each leaving O
// (unnormalised), its reference maximum and its row sum in the workspace; the
// last to finish (a per-unit counter) merges them by log-sum-exp.  Bounding a
// CTA's share also bounds how many tiles of products the accumulator in tensor
// memory sums, and the error of that sum grows with the count (about linearly:
// 3.8e-4 of rms(out) at 48-64 tiles, 1.8e-3 at 240, on 4-bit parity cases).
//
// Arithmetic.  q1 = U q is scaled by sm_scale * log2(e) and a per-row power
// of two and kept as hi + lo fp16 halves.  Key codes enter the products as
// exact small fp16 integers, one accumulator per 64-dimension scale block:
//   S_b = (q1_hi + q1_lo)[block b] . c_k[block b]       (two MMAs per k-step)
// and the key scales are applied in fp32 afterwards: s = S_0 k_0 + S_1 k_1
// (asymmetric codes: unsigned u, and s gains z_k(b) * sum_{d in b} q1_d).
// The online softmax (base 2, lazy rescaling: the running maximum moves only
// when a row's maximum grows by more than 2^8) gives p <= 2^8, kept as hi + lo
// fp16 halves.  A value's scale is split as s_v = s_hi + s_lo with s_hi its
// top 9 significant bits (8 at b = 4), so that c * s_hi and c * s_lo
// (|c| <= 2^(b-1)) are exact fp16 numbers and
//   O += p_hi . (c s_hi) + p_lo . (c s_hi) + p_hi . (c s_lo)
// over full 128-dimension rows (the dropped p_lo . (c s_lo) is below 2^-20 of
// the product; E4M3 scales have s_lo = 0 and skip the third MMA; asymmetric
// codes enter centred, as (u - 2^(b-1)) s, and each softmax thread adds
// sum_k p_k (z_v(k, b) + 2^(b-1) s_v(k, b)) to its row's block b: the
// accumulator in tensor memory, which adds each tile's products to the sum of
// the tiles before it, then holds sums of the size of the result rather than
// of u s >= 0).  Dequantised values must lie in the fp16 range, as for every
// kernel of this library.
//
// Roles (15 warps):
//  * warps 6-13, softmax: warps w and w + 4 share the 32 rows of TMEM lane
//    quarter w % 4 (thread = row), each taking 32 of a tile's 64 keys; they trade
//    row maxima through shared memory at a 64-thread named barrier that also
//    carries their decision to go on.  tcgen05.ld of S, key scales, mask,
//    online softmax, p_hi / p_lo written back over S with tcgen05.st (the A
//    operand of PV), rare rescales of O in place;
//  * warps 2-5, dequantisation: thread = (key, half of the dimensions); a tile
//    is unpacked into the MMA layouts in shared memory: integer key codes
//    K-major, values c*s_hi and c*s_lo MN-major;
//  * warp 0, lane 0: issues QK^T; warp 14, lane 0: issues PV -- two streams,
//    so that a wait of one never holds up the other's MMAs;
//  * warp 1, lane 0: issues the bulk copies of packed codes and scales into a
//    ring of raw stages, up to kStages tiles ahead.
// TMEM: three S/P buffers (128 columns each) and O (128); q1 hi / lo live in
// shared memory as the A operand of QK^T.
// Every hand-off is an mbarrier; every wait is bounded (a time-out sets
// KVQ3_DEV_TIMEOUT and the CTA winds down: MMAs and copies in flight are
// drained and TMEM freed before it exits).
#include <string.h>

#include <algorithm>

#include "kvq3_internal.h"
#include "kvq3_tc.cuh"

using namespace kvq3;

namespace {

constexpr int kRows = 128;            // query rows per CTA = TMEM lanes
constexpr int kKeys = 64;             // keys per tile
constexpr int kD = 128;               // head dimension
constexpr int kStages = 4;            // raw stages in flight
constexpr int kThreads = 15 * 32;
constexpr int kMmaWarp = 0;           // QK^T issue (lane 0) and the TMEM allocation
constexpr int kMmaThread = 0;
constexpr int kProducer = 32;         // warp 1, lane 0
constexpr int kDequant0 = 2 * 32;     // warps 2-5
constexpr int kSoftmax0 = 6;          // warps 6-13
constexpr int kPvThread = 14 * 32;    // warp 14, lane 0: PV issue
constexpr uint32_t kTmemCols = 512;
constexpr int kSP = 3;                // S/P buffers in TMEM
constexpr uint32_t kColSP = 0, kColO = 384;   // TMEM: S/P buffer j at 128 j, O
constexpr float kRescale = 8.0f;      // log2 of the largest p between rescales
constexpr int kMinSplit = 8;          // a unit of at least this many key tiles runs as several CTAs
constexpr int kChain = 128;           // ... each over at most this many key tiles (while kMaxParts allow)
constexpr int kMaxParts = 16;         // CTAs a unit can run as
constexpr int kPartStride = 132;      // floats a row of a partial takes: O (128), m, l, padding

// shared memory (bytes)
constexpr int kTile = kKeys * kD * 2;                          // one fp16 tile (16 KB)
constexpr int kOffK = 0;                                       // [2] key codes, K-major
constexpr int kOffV = kOffK + 2 * kTile;                       // [2][hi, lo] values, MN-major
constexpr int kMaxCB = 4 * kD / 8;                             // code bytes per vector at b = 4
constexpr int kRawK = 0, kRawV = kKeys * kMaxCB;               // raw stage: codes K, V
constexpr int kRawKs = 2 * kKeys * kMaxCB, kRawVs = kRawKs + kKeys * 2 * 4;   // scales K, V (<= 8 B a key)
constexpr int kRawBytes = kRawVs + kKeys * 2 * 4;              // 9216
constexpr int kOffQ = kOffV + 4 * kTile;                       // q1 hi, lo: K-major A of QK^T
constexpr int kOffRaw = kOffQ + 4 * kTile;
constexpr int kOffKs = kOffRaw + kStages * kRawBytes;          // [kStages][64 keys][2 blocks] fp32 key scales
constexpr int kOffZk = kOffKs + kStages * kKeys * 2 * 4;       // [kStages][64][2] key zero points (asymmetric codes)
constexpr int kOffZv = kOffZk + kStages * kKeys * 2 * 4;       // [kStages][64][2] value zero points
constexpr int kOffRsum = kOffZv + kStages * kKeys * 2 * 4;     // [128][2] per-row block sums of q1 (asymmetric codes)
constexpr int kOffZred = kOffRsum + kRows * 2 * 4;             // [2][2][128] value zero-point sums traded
constexpr int kOffRed = kOffZred + 2 * 2 * kRows * 4;          // [2][2][128] fp32 row maxima / sums traded
constexpr int kPitch = kD + 1;                                 // row staging pitch (floats)
constexpr int kOffRows = kOffK;                                // [128][129] fp32 outputs over the K/V tiles
constexpr int kOffQinv = kOffRed + 2 * 2 * kRows * 4;          // [128] fp32
constexpr int kNumBars = 3 * kStages + 4 + 3 * kSP + 2;
static_assert(kRows * kPitch * 4 <= kOffQ - kOffK, "output staging fits over the K/V tiles");
constexpr int kOffBars = kOffQinv + kRows * 4;
constexpr int kOffMisc = kOffBars + kNumBars * 8;              // TMEM base, abort flag, masks
constexpr int kSmem = kOffMisc + 16 + 2 * kStages * 8;
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
  int32_t parts;        // CTAs in the grid per unit (2 .. kMaxParts)
  int32_t* counters;    // [units] parts of a split unit done (zeroed before the launch)
  float* partial;       // [units][parts][128 rows][kPartStride]: O (unnormalised), m, l of each part
  int64_t ws_floats;    // floats of the partial area (bounds of the checked build)
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

// two b-bit unsigned fields -> half2 of the exact integers u: (0x6400 | u) - 1024
template <int B>
__device__ __forceinline__ __half2 ucodes2(uint32_t w) {
  constexpr uint32_t f = (1u << B) - 1u;
  const uint32_t h = (((w & ((1u << (2 * B)) - 1u)) * (1u + (1u << (16 - B)))) & (f | (f << 16))) ^ 0x64006400u;
  return __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
}
// two unsigned b-bit fields -> half2 of the centred integers u - 2^(b-1)
template <int B>
__device__ __forceinline__ __half2 ccodes2(uint32_t w) {
  constexpr uint32_t f = (1u << B) - 1u;
  const uint32_t h = (((w & ((1u << (2 * B)) - 1u)) * (1u + (1u << (16 - B)))) & (f | (f << 16))) ^ 0x64006400u;
  const __half off = __ushort_as_half((unsigned short)(0x6400u | (1u << (B - 1))));
  return __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(off, off));
}
// two b-bit two's-complement fields (bits 0..b-1 and b..2b-1 of w) -> half2
// of the exact integers: times 1 + 2^(16-b) puts the second field at bit
// 16; flipping the sign bit gives c + 2^(b-1), and (0x6400 | (c + 2^(b-1)))
// - (1024 + 2^(b-1)) = c
template <int B>
__device__ __forceinline__ __half2 codes2(uint32_t w) {
  constexpr uint32_t f = (1u << B) - 1u, sgn = 1u << (B - 1);
  const uint32_t h = (((w & ((1u << (2 * B)) - 1u)) * (1u + (1u << (16 - B)))) & (f | (f << 16))) ^
                     ((0x6400u | sgn) * 0x10001u);
  const __half off = __ushort_as_half((unsigned short)(0x6400u | sgn));
  return __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(off, off));
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Named barrier `id` of two warps (64 threads) that also returns the AND of
// their flags; it orders their shared-memory accesses like bar.sync.
__device__ __forceinline__ bool pair_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.and.pred po, %2, 64, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

template <int SCALE, int BITS>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p,
                                                                  const __grid_constant__ RotParams rp) {
  constexpr bool kAsym = SCALE == KVQ3_SCALE_E4M3_ZP;   // E4M3 scale and zero point, unsigned codes
  constexpr int SB = SCALE == KVQ3_SCALE_F32 ? 4 : (SCALE == KVQ3_SCALE_F16 || kAsym) ? 2 : 1;
  constexpr int kCB = BITS * kD / 8;   // code bytes per vector
  constexpr bool kLo = SCALE != KVQ3_SCALE_E4M3 && !kAsym;   // values carry a low part of the scale
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* raw_full = bars;                   // [kStages] bulk copies landed
  uint64_t* raw_empty = bars + kStages;        // [kStages] dequantisation and softmax done with a stage
  uint64_t* ks_full = bars + 2 * kStages;      // [kStages] key scales and valid-key mask of a stage ready
  uint64_t* k_full = bars + 3 * kStages;       // [2] key tile ready
  uint64_t* v_full = k_full + 2;               // [2] value tiles ready
  uint64_t* s_full = v_full + 2;               // [kSP] S of the tile in TMEM
  uint64_t* p_full = s_full + kSP;             // [kSP] P of the tile in TMEM (and O rescaled)
  uint64_t* pv_done = p_full + kSP;            // [kSP] PV of the tile complete
  uint64_t* drain = pv_done + kSP;             // [2] every MMA of an issuer complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint64_t* stage_mask = reinterpret_cast<uint64_t*>(smem + kOffMisc + 16);   // [kStages] valid keys
  uint64_t* key_mask = stage_mask + kStages;                                  // [kStages]
  float* rows = reinterpret_cast<float*>(smem + kOffRows);
  float* qinv_s = reinterpret_cast<float*>(smem + kOffQinv);
  float* ks_s = reinterpret_cast<float*>(smem + kOffKs);
  float* red_s = reinterpret_cast<float*>(smem + kOffRed);
  float* zk_s = reinterpret_cast<float*>(smem + kOffZk);
  float* zv_s = reinterpret_cast<float*>(smem + kOffZv);
  float* rsum_s = reinterpret_cast<float*>(smem + kOffRsum);
  float* zred_s = reinterpret_cast<float*>(smem + kOffZred);

  const CacheGeom& g = p.g;
  const int kvh = blockIdx.y;
  const int nqb = (int)gridDim.x / p.parts;
  const int qblk = nqb - 1 - (int)blockIdx.x / p.parts;    // longest query blocks first
  const int part = (int)blockIdx.x % p.parts;              // which part of the unit's keys
  const int unit = kvh * nqb + qblk;
  const int t0 = qblk * p.qb;
  const int ntok = min(p.qb, p.n - t0);
  const int nrows = ntok * p.G;
  const int64_t kmax = p.pos0 + t0 + ntok - 1;             // last position any row attends to
  const int T = (int)(kmax / kKeys) + 1;                   // key tiles of the unit
  // a long unit runs as np CTAs over equal shares of its key tiles, at most
  // kChain each (so that no accumulation in tensor memory runs longer), each
  // leaving its partial in the workspace, merged by the last to finish; a
  // short one as one CTA (the unit's other CTAs return at once)
  const int np = T < kMinSplit ? 1 : min(p.parts, max(2, (T + kChain - 1) / kChain));
  const bool split = np > 1;
  if (part >= np) return;
  const int tlo = (int)((int64_t)T * part / np);
  const int nt = (int)((int64_t)T * (part + 1) / np) - tlo;   // key tiles of this CTA

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 128 + 256);
      mbar_init(&ks_full[s], 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&k_full[b], 128);
      mbar_init(&v_full[b], 128);
    }
    for (int j = 0; j < kSP; ++j) {
      mbar_init(&s_full[j], 1);
      mbar_init(&p_full[j], 256);
      mbar_init(&pv_done[j], 1);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tc::alloc(tmem_slot, kTmemCols);
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
  // is a multiple of 16) into its raw stage; producer thread only.  Key 64 t
  // sits at slot slot0 of logical page lp0 (tracked by the caller from tile
  // to tile: no division); positions are below 2^31 (checked on the host).
  const int64_t pool_bytes = g.num_pages * g.page_bytes;
  (void)pool_bytes;   // read by the checked build only
  auto issue = [&](int u, int t, uint32_t lp0, uint32_t slot0) {   // u: this CTA's tile count, t: the key tile
    const int s = u % kStages;
    uint8_t* st = smem + kOffRaw + s * kRawBytes;
    const uint32_t k0 = (uint32_t)t * kKeys, P = (uint32_t)g.page_size, last = (uint32_t)kmax;
    int64_t pg[4];
    uint32_t slot[4];
    uint64_t mask = 0;
    uint32_t bytes = 0;
    uint32_t lp = lp0, sl = slot0;
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      if (gi > 0 && (sl += 16u) == P) {   // the next 16-key group starts a page
        sl = 0u;
        ++lp;
      }
      const uint32_t pos = k0 + 16u * gi;
      pg[gi] = -1;
      slot[gi] = sl;
      if (pos > last) continue;
      pg[gi] = page_of(g, p.page_table, p.seq, lp);
      if (pg[gi] < 0) {
        set_status(p.status, KVQ3_DEV_BAD_PAGE);
        continue;
      }
      mask |= 0xFFFFull << (16 * gi);
      bytes += 16u * (2u * kCB + 2u * 2u * SB);
    }
    if (last - k0 < (uint32_t)kKeys - 1u) mask &= (1ull << (last - k0 + 1u)) - 1ull;   // keys past the last row
    stage_mask[s] = mask;
    mbar_expect_tx(&raw_full[s], bytes);
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      if (pg[gi] < 0 || (gi > 0 && pg[gi - 1] == pg[gi])) continue;   // not the first group of a run
      uint32_t nk = 16u;                                                // consecutive groups of one page
#pragma unroll
      for (int gj = gi + 1; gj < 4; ++gj)
        if (pg[gj] == pg[gi] && nk == 16u * (uint32_t)(gj - gi)) nk += 16u;
      const int64_t rk = record_offset(g, pg[gi], kvh, 0), rv = record_offset(g, pg[gi], kvh, 1);
      const int64_t ck = rk + g.scale_hdr_bytes + (int64_t)slot[gi] * kCB;
      const int64_t cv = rv + g.scale_hdr_bytes + (int64_t)slot[gi] * kCB;
      const int64_t sk = rk + (int64_t)slot[gi] * 2 * SB, sv = rv + (int64_t)slot[gi] * 2 * SB;
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
    }
  };

  // ---- the unit's fp16 query rows (row = token * G + head) staged in the
  // key/value tile area, idle until the roles start: every thread's 16-byte
  // loads in flight at once, rather than one row's latency after another
  uint8_t* qrows = smem + kOffK;   // [128 rows][256 B]
  static_assert(kRows * kD * 2 <= kOffQ - kOffK, "query staging fits the key/value tiles");
  {
    constexpr int kPieces = kRows * kD * 2 / 16, kPer = (kPieces + kThreads - 1) / kThreads;
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + k * kThreads, row = i >> 4;
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if (i < kPieces && row < nrows) {
        const int tok = t0 + row / p.G, h = kvh * p.G + row % p.G;
        v[k] = *reinterpret_cast<const uint4*>(p.q + ((int64_t)tok * p.Hq + h) * kD + (i & 15) * 8);
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + k * kThreads;
      if (i < kPieces) *reinterpret_cast<uint4*>(qrows + i * 16) = v[k];
    }
  }
  __syncthreads();

  // ---- q1 = U q of the rows, scaled by qk_scale and a per-row power of two,
  // as hi + lo fp16 halves in the K-major A layout of QK^T: (row, d) at
  // (row/8)*2048 + (d/8)*128 + (row%8)*16 + (d%8)*2, the lo halves 32 KB on
  {
    const uint32_t sgn = lane_signs<4>(rp, lane);
    float4 qt[1], qtr[1];
    lane_quats<4>(rp, lane, qt);
    lane_quats_r<4>(rp, lane, qtr);
    const bool so4 = rot_so4(rp), pair = rot_pair(rp);
    for (int row = warp; row < kRows; row += kThreads / 32) {
      float x[4];
      {   // zeros for the rows past the unit's (staged as zeros)
        const uint2 raw = *reinterpret_cast<const uint2*>(qrows + row * 256 + lane * 8);
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
      const float2 y0 = make_float2(x[0] * sc, x[1] * sc), y1 = make_float2(x[2] * sc, x[3] * sc);
      const __half2 h0 = __floats2half2_rn(y0.x, y0.y), h1 = __floats2half2_rn(y1.x, y1.y);
      const float2 r0 = f2sub(y0, __half22float2(h0)), r1 = f2sub(y1, __half22float2(h1));
      uint8_t* qa = smem + kOffQ + (row >> 3) * 2048 + (lane >> 1) * 128 + (row & 7) * 16 + (lane & 1) * 8;
      *reinterpret_cast<uint2*>(qa) = make_uint2(h2u(h0), h2u(h1));
      *reinterpret_cast<uint2*>(qa + 2 * kTile) =
          make_uint2(h2u(__floats2half2_rn(r0.x, r0.y)), h2u(__floats2half2_rn(r1.x, r1.y)));
      if (lane == 0) qinv_s[row] = ldexpf(1.0f, -ex);
      if constexpr (kAsym) {   // sum of the q1 the MMAs see over each block (lanes 16b .. 16b + 15)
        const float2 fh0 = __half22float2(h0), fh1 = __half22float2(h1);
        const float2 fl0 = __half22float2(__floats2half2_rn(r0.x, r0.y));
        const float2 fl1 = __half22float2(__floats2half2_rn(r1.x, r1.y));
        float bs = ((fh0.x + fl0.x) + (fh0.y + fl0.y)) + ((fh1.x + fl1.x) + (fh1.y + fl1.y));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) bs += __shfl_xor_sync(kFull, bs, o);
        if ((lane & 15) == 0) rsum_s[row * 2 + (lane >> 4)] = bs;
      }
    }
  }
  fence_proxy_async();   // generic stores read by the tensor cores
  __syncthreads();

  if (warp >= kSoftmax0 && warp < kSoftmax0 + 8) {
    // ================================================================ softmax
    const int wq = warp & 3, kh = (warp - kSoftmax0) >> 2;   // lane quarter; key half (keys 32kh .. 32kh + 31)
    const int row = 32 * wq + lane;
    const uint32_t lanes = (uint32_t)(32 * wq) << 16;
    const float qinv = qinv_s[row];
    const float2 qinv2 = make_float2(qinv, qinv);
    const int64_t lim = row < nrows ? p.pos0 + t0 + row / p.G : -1;
    float m_used = -INFINITY;
    float2 l2 = make_float2(0.0f, 0.0f);
    // asymmetric codes: per-row block sums of q1 (the keys' zero-point term)
    // and this warp's share of sum_k p_k z_v(k, block) for blocks 0 and 1
    const float2 rs0 = kAsym ? make_float2(rsum_s[row * 2], rsum_s[row * 2]) : make_float2(0.0f, 0.0f);
    const float2 rs1 = kAsym ? make_float2(rsum_s[row * 2 + 1], rsum_s[row * 2 + 1]) : make_float2(0.0f, 0.0f);
    float2 za0 = make_float2(0.0f, 0.0f), za1 = make_float2(0.0f, 0.0f);
    bool okw = true;   // this warp's waits all succeeded (warp-uniform)
    for (int t = 0; t < nt; ++t) {   // t counts this CTA's tiles; key tile tlo + t
      const int b = t & 1, s = t % kStages, j = t % kSP;
      okw = okw && __all_sync(kFull, wait(&s_full[j], (uint32_t)(t / kSP) & 1u) &&
                                         wait(&ks_full[s], (uint32_t)(t / kStages) & 1u));
      const uint32_t tS = tmem + lanes + kColSP + 128u * j;
      float2 sv[16];
      float pmax = -INFINITY;
      if (okw) {
        tc::fence_after();
        uint32_t a[32], c[32];
        tc::ld32(tS + 32 * kh, a);          // S, block 0, this half's keys
        tc::ld32(tS + 64 + 32 * kh, c);     // S, block 1
        const float4* ksr = reinterpret_cast<const float4*>(ks_s + (s * kKeys + 32 * kh) * 2);
        const uint32_t km = (uint32_t)(key_mask[s] >> (32 * kh));
        float4 kk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) kk[i] = ksr[i];   // (k0, k1) of keys 2i, 2i + 1
        if (!kAsym) mbar_arrive(&raw_empty[s]);       // done with the stage's scales and mask
        tc::wait_ld();
        tc::reg_fence(a);
        tc::reg_fence(c);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          sv[i] = f2fma(make_float2(__uint_as_float(c[2 * i]), __uint_as_float(c[2 * i + 1])),
                        make_float2(kk[i].y, kk[i].w),
                        f2mul(make_float2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1])),
                              make_float2(kk[i].x, kk[i].z)));
        if constexpr (kAsym) {   // + z_k(block) * sum_{d in block} q1_d
          const float4* zkr = reinterpret_cast<const float4*>(zk_s + (s * kKeys + 32 * kh) * 2);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 z = zkr[i];
            sv[i] = f2fma(make_float2(z.y, z.w), rs1, f2fma(make_float2(z.x, z.z), rs0, sv[i]));
          }
        }
        const int64_t k0 = (int64_t)(tlo + t) * kKeys + 32 * kh;
        if (!(km == 0xFFFFFFFFu && k0 + 31 <= lim)) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (!((km >> (2 * i)) & 1u) || k0 + 2 * i > lim) sv[i].x = -INFINITY;
            if (!((km >> (2 * i + 1)) & 1u) || k0 + 2 * i + 1 > lim) sv[i].y = -INFINITY;
          }
        }
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmaxf(fmaxf(sv[2 * i].x, sv[2 * i].y), fmaxf(sv[2 * i + 1].x, sv[2 * i + 1].y));
#pragma unroll
        for (int i = 0; i < 4; ++i) m8[i] = fmaxf(m8[i], m8[i + 4]);
        pmax = fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3]));
        red_s[(b * 2 + kh) * kRows + row] = pmax;
      }
      if (!pair_and(1 + wq, okw)) break;                 // both warps of the rows go on, or neither
      const float mx = fmaxf(pmax, red_s[(b * 2 + (kh ^ 1)) * kRows + row]);
      const float xm = mx * qinv;
      const bool need = xm > m_used + kRescale;
      if (__any_sync(kFull, need)) {
        const float m_new = need ? xm : m_used;
        const float alpha = need ? (m_used == -INFINITY ? 0.0f : ex2(m_used - m_new)) : 1.0f;
        l2.x *= alpha;
        l2.y *= alpha;
        if constexpr (kAsym) {
          za0 = f2mul(za0, make_float2(alpha, alpha));
          za1 = f2mul(za1, make_float2(alpha, alpha));
        }
        if (t > 0) {   // O holds PV up to tile t - 1: wait for it, then scale this warp's half in place
          okw = __all_sync(kFull, wait(&pv_done[(t - 1) % kSP], (uint32_t)((t - 1) / kSP) & 1u));
          if (okw) {
            tc::fence_after();
#pragma unroll
            for (int c4 = 0; c4 < 2; ++c4) {
              uint32_t o[32];
              const uint32_t ta = tmem + lanes + kColO + 64u * kh + 32u * c4;
              tc::ld32(ta, o);
              tc::wait_ld();
              tc::reg_fence(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tc::st32(ta, o);
            }
          }
        }
        m_used = m_new;
      }
      if (!okw) continue;   // the partner learns of it at the next exchange
      const float moff = m_used == -INFINITY ? 0.0f : m_used;
      const float2 moff2 = make_float2(-moff, -moff);
      uint32_t hv[16], lv[16];
      const float4* zvr = reinterpret_cast<const float4*>(zv_s + (s * kKeys + 32 * kh) * 2);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 x = f2fma(sv[i], qinv2, moff2);
        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
        l2 = f2add(l2, pp);
        if constexpr (kAsym) {
          const float4 z = zvr[i];
          za0 = f2fma(pp, make_float2(z.x, z.z), za0);
          za1 = f2fma(pp, make_float2(z.y, z.w), za1);
        }
        const __half2 hi = __floats2half2_rn(pp.x, pp.y);
        const float2 lo = f2sub(pp, __half22float2(hi));
        hv[i] = h2u(hi);
        lv[i] = h2u(__floats2half2_rn(lo.x, lo.y));
      }
      if (kAsym) mbar_arrive(&raw_empty[s]);   // done with the stage's zero points too
      tc::st16(tS + 16 * kh, hv);        // P hi (keys 32kh..) over S columns both warps have read
      tc::st16(tS + 32 + 16 * kh, lv);   // P lo
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(&p_full[j]);
    }
    // row sums of the two halves (in the slots of parity nt & 1, which no one
    // reads after the last tile's exchange); O of this warp's 64 columns
    const int e = (nt & 1) * 2;
    red_s[(e + kh) * kRows + row] = l2.x + l2.y;
    if constexpr (kAsym) {
      zred_s[(kh * 2 + 0) * kRows + row] = za0.x + za0.y;
      zred_s[(kh * 2 + 1) * kRows + row] = za1.x + za1.y;
    }
    bool ok = pair_and(1 + wq, okw);
    const float l = red_s[(e + kh) * kRows + row] + red_s[(e + (kh ^ 1)) * kRows + row];
    // the zero-point share of O for this warp's columns (block kh)
    const float zo = kAsym ? zred_s[(0 * 2 + kh) * kRows + row] + zred_s[(1 * 2 + kh) * kRows + row] : 0.0f;
    if (ok) ok = __all_sync(kFull, wait(&pv_done[(nt - 1) % kSP], (uint32_t)((nt - 1) / kSP) & 1u));
    tc::fence_after();
    // a whole unit: normalised rows into the staging; part of a split unit:
    // O (unnormalised, relative to 2^m_used), m_used and l to its partial
    const float inv = split ? 1.0f : (ok && l > 0.0f) ? 1.0f / l : 0.0f;
    float* prow = p.partial + ((int64_t)(unit * p.parts + part) * kRows + row) * kPartStride;
    const bool pw = split && KVQ3_CHECK(p.status, in_range((prow - p.partial), kPartStride, p.ws_floats));
#pragma unroll
    for (int c4 = 0; c4 < 2; ++c4) {
      uint32_t o[32];
      if (ok) {
        tc::ld32(tmem + lanes + kColO + 64u * kh + 32u * c4, o);
        tc::wait_ld();
        tc::reg_fence(o);
        if constexpr (kAsym) {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) + zo);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (split) {
        if (pw) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(prow + 64 * kh + 32 * c4 + i) =
                make_float4(__uint_as_float(o[i]), __uint_as_float(o[i + 1]), __uint_as_float(o[i + 2]),
                            __uint_as_float(o[i + 3]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) rows[row * kPitch + 64 * kh + 32 * c4 + i] = __uint_as_float(o[i]) * inv;
      }
    }
    if (pw && kh == 0) {
      prow[kD] = ok ? m_used : -INFINITY;
      prow[kD + 1] = ok ? l : 0.0f;
    }
  } else if (tid >= kDequant0 && tid < kDequant0 + 128) {
    // ================================================================ dequantisation
    // lane -> (key, half): 8 consecutive lanes hold 8 consecutive keys, so a
    // 16-byte store of 8 lanes covers the 32 banks once
    const int dt = tid - kDequant0, key = (dt >> 5) * 16 + (dt & 15), hd = (dt >> 4) & 1;   // key; half of the dimensions
    for (int t = 0; t < nt; ++t) {   // this CTA's tiles
      const int s = t % kStages, b = t & 1;
      // a failed wait leaves at once, arriving nowhere: a stage is released
      // (raw_empty) only once its copies have landed
      if (!wait(&raw_full[s], (uint32_t)(t / kStages) & 1u)) break;
      const uint8_t* st = smem + kOffRaw + s * kRawBytes;
      const uint64_t vm = stage_mask[s];
      const bool kv = (vm >> key) & 1ull;
      // ---- keys: exact integer codes, K-major: (key, d) at (key/8)*2048 + (d/8)*128 + (key%8)*16 + (d%8)*2
      if (t >= 2 && !wait(&s_full[(t - 2) % kSP], (uint32_t)((t - 2) / kSP) & 1u)) break;   // QK(t - 2) read the buffer
      {
        // the lane's 64 codes as two runs of 96 bits (32 codes, 4 groups of 8);
        // the run loop is not unrolled, to keep the roles' code small
        uint8_t* kt = smem + kOffK + b * kTile + (key >> 3) * 2048 + (key & 7) * 16 + 8 * hd * 128;
#pragma unroll 1
        for (int r = 0; r < 2; ++r) {   // 32 codes: BITS words
          const uint32_t* src = reinterpret_cast<const uint32_t*>(st + kRawK + key * kCB + hd * (kCB / 2) + r * (kCB / 4));
          uint32_t w[BITS + 1];
#pragma unroll
          for (int i = 0; i < BITS; ++i) w[i] = src[i];
          w[BITS] = 0u;
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {   // 8 codes at bit 8 BITS gq
            const int bit = 8 * BITS * gq;
            const uint32_t wg = (bit & 31) ? __funnelshift_r(w[bit >> 5], w[(bit >> 5) + 1], bit & 31) : w[bit >> 5];
            uint4 o;
            if constexpr (kAsym) {
              o.x = h2u(ucodes2<BITS>(wg));
              o.y = h2u(ucodes2<BITS>(wg >> (2 * BITS)));
              o.z = h2u(ucodes2<BITS>(wg >> (4 * BITS)));
              o.w = h2u(ucodes2<BITS>(wg >> (6 * BITS)));
            } else {
              o.x = h2u(codes2<BITS>(wg));
              o.y = h2u(codes2<BITS>(wg >> (2 * BITS)));
              o.z = h2u(codes2<BITS>(wg >> (4 * BITS)));
              o.w = h2u(codes2<BITS>(wg >> (6 * BITS)));
            }
            *reinterpret_cast<uint4*>(kt + (4 * r + gq) * 128) = o;
          }
        }
        uint32_t bits;
        const uint8_t* sp = st + kRawKs + (key * 2 + hd) * SB;
        if (SB == 4) bits = *reinterpret_cast<const uint32_t*>(sp);
        else if (SB == 2) bits = *reinterpret_cast<const uint16_t*>(sp);
        else bits = *sp;
        if constexpr (kAsym) {   // scale byte, then zero-point byte; the value's zero point as well
          const uint32_t vbits = *reinterpret_cast<const uint16_t*>(st + kRawVs + (key * 2 + hd) * SB);
          ks_s[(s * kKeys + key) * 2 + hd] = kv ? decode_scale(bits & 0xFFu, KVQ3_SCALE_E4M3) : 0.0f;
          zk_s[(s * kKeys + key) * 2 + hd] = kv ? decode_scale(bits >> 8, KVQ3_SCALE_E4M3) : 0.0f;
          // values enter the MMAs centred, (u - 2^(b-1)) s: their zero point
          // gains 2^(b-1) s, so that the accumulator in tensor memory holds
          // sums of the size of the result, not of u s >= 0
          zv_s[(s * kKeys + key) * 2 + hd] =
              kv ? decode_scale(vbits >> 8, KVQ3_SCALE_E4M3) +
                       (float)(1 << (BITS - 1)) * decode_scale(vbits & 0xFFu, KVQ3_SCALE_E4M3)
                 : 0.0f;
        } else {
          ks_s[(s * kKeys + key) * 2 + hd] = kv ? decode_scale(bits, SCALE) : 0.0f;
        }
        if (dt == 0) key_mask[s] = vm;
      }
      fence_proxy_async();
      mbar_arrive(&k_full[b]);
      mbar_arrive(&ks_full[s]);
      // ---- values c * s_hi, c * s_lo, MN-major: (key, d) at (d/8)*1024 + (key/8)*128 + (key%8)*16 + (d%8)*2
      if (t >= 2 && !wait(&pv_done[(t - 2) % kSP], (uint32_t)((t - 2) / kSP) & 1u)) break;
      {
        uint32_t bits;
        const uint8_t* sp = st + kRawVs + (key * 2 + hd) * SB;
        if (SB == 4) bits = *reinterpret_cast<const uint32_t*>(sp);
        else if (SB == 2) bits = *reinterpret_cast<const uint16_t*>(sp);
        else bits = *sp;
        const float sv = kv ? decode_scale(kAsym ? (bits & 0xFFu) : bits, kAsym ? KVQ3_SCALE_E4M3 : SCALE) : 0.0f;
        // top 9 significant bits (8 at b = 4): c s_hi stays within fp16's 11
        const float s_hi = __uint_as_float(__float_as_uint(sv) & (BITS == 4 ? 0xFFFF0000u : 0xFFFF8000u));
        const __half2 hs = __float2half2_rn(s_hi), ls = __float2half2_rn(sv - s_hi);
        uint8_t* vt = smem + kOffV + b * 2 * kTile + (key >> 3) * 128 + (key & 7) * 16 + 8 * hd * 1024;
#pragma unroll 1
        for (int r = 0; r < 2; ++r) {
          const uint32_t* src = reinterpret_cast<const uint32_t*>(st + kRawV + key * kCB + hd * (kCB / 2) + r * (kCB / 4));
          uint32_t w[BITS + 1];
#pragma unroll
          for (int i = 0; i < BITS; ++i) w[i] = src[i];
          w[BITS] = 0u;
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const int bit = 8 * BITS * gq;
            const uint32_t wg = (bit & 31) ? __funnelshift_r(w[bit >> 5], w[(bit >> 5) + 1], bit & 31) : w[bit >> 5];
            __half2 c0, c1, c2, c3;
            if constexpr (kAsym) {   // (u - 2^(b-1)) s: the zero point's share is summed by the softmax
              c0 = ccodes2<BITS>(wg), c1 = ccodes2<BITS>(wg >> (2 * BITS));
              c2 = ccodes2<BITS>(wg >> (4 * BITS)), c3 = ccodes2<BITS>(wg >> (6 * BITS));
            } else {
              c0 = codes2<BITS>(wg), c1 = codes2<BITS>(wg >> (2 * BITS));
              c2 = codes2<BITS>(wg >> (4 * BITS)), c3 = codes2<BITS>(wg >> (6 * BITS));
            }
            uint4 o;
            o.x = h2u(__hmul2(c0, hs));
            o.y = h2u(__hmul2(c1, hs));
            o.z = h2u(__hmul2(c2, hs));
            o.w = h2u(__hmul2(c3, hs));
            *reinterpret_cast<uint4*>(vt + (4 * r + gq) * 1024) = o;
            if (kLo) {
              o.x = h2u(__hmul2(c0, ls));
              o.y = h2u(__hmul2(c1, ls));
              o.z = h2u(__hmul2(c2, ls));
              o.w = h2u(__hmul2(c3, ls));
              *reinterpret_cast<uint4*>(vt + kTile + (4 * r + gq) * 1024) = o;
            }
          }
        }
      }
      fence_proxy_async();
      mbar_arrive(&v_full[b]);
      mbar_arrive(&raw_empty[s]);
    }
  } else if (tid == kProducer) {
    // ================================================================ bulk copies
    int issued = 0;
    bool ok = true;
    uint32_t lp = (uint32_t)(tlo * kKeys) / (uint32_t)g.page_size;   // key 64 (tlo + t) = lp * P + slot
    uint32_t slot = (uint32_t)(tlo * kKeys) - lp * (uint32_t)g.page_size;
    for (int t = 0; t < nt && ok; ++t) {
      if (t >= kStages) ok = wait(&raw_empty[t % kStages], (uint32_t)(t / kStages - 1) & 1u);   // tile t - kStages consumed
      if (ok && *abort_flag) ok = false;
      if (ok) issue(t, tlo + t, lp, slot), issued = t + 1;
      for (slot += kKeys; slot >= (uint32_t)g.page_size; slot -= (uint32_t)g.page_size) ++lp;
    }
    // no bulk copy may still target this CTA's shared memory at exit: the
    // last kStages tiles issued are the only ones that can be in flight
    for (int t = max(0, issued - kStages); t < issued; ++t)
      mbar_wait(&raw_full[t % kStages], (uint32_t)(t / kStages) & 1u, kDrainPolls);
  } else if (tid == kMmaThread) {
    // ================================================================ QK^T issue
    constexpr uint32_t kIdQK = tc::idesc_f16(128, kKeys, false);
    // descriptors (start addresses in 16-byte units in the low half)
    const uint64_t dq = tc::sdesc(smem_u32(smem + kOffQ), 128u, 2048u);
    const uint64_t dk = tc::sdesc(smem_u32(smem + kOffK), 128u, 2048u);
    const uint32_t dq_lo = (uint32_t)dq, dq_hi = (uint32_t)(dq >> 32);
    const uint32_t dk_lo = (uint32_t)dk, dk_hi = (uint32_t)(dk >> 32);
    for (int t = 0; t < nt; ++t) {   // S_b(t) = q1[block b] . c_k[block b], hi and lo halves of q1
      const int b = t & 1, j = t % kSP;
      if (!wait(&k_full[b], (uint32_t)(t >> 1) & 1u)) break;
      if (t >= kSP && !wait(&pv_done[j], (uint32_t)(t / kSP - 1) & 1u)) break;   // P(t - kSP) consumed
      tc::fence_after();
      const uint32_t kb = dk_lo + (uint32_t)b * (kTile >> 4);
      const uint32_t dS = tmem + kColSP + 128u * j;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk)
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t al = dq_lo + (uint32_t)((part * 2 * kTile + (blk * 8 + ks * 2) * 128) / 16);
            const uint32_t bl = kb + (uint32_t)((blk * 8 + ks * 2) * 128 / 16);
            if (part == 0 && ks == 0) tc::mma_ss_c<false>(dS + 64u * blk, al, dq_hi, bl, dk_hi, kIdQK);
            else tc::mma_ss_c<true>(dS + 64u * blk, al, dq_hi, bl, dk_hi, kIdQK);
          }
      tc::commit(&s_full[j]);
    }
    tc::commit(&drain[0]);   // whatever was issued completes before TMEM is freed
    mbar_wait(&drain[0], 0u, kDrainPolls);
  } else if (tid == kPvThread) {
    // ================================================================ PV issue
    constexpr uint32_t kIdPV = tc::idesc_f16(128, kD, true);
    const uint64_t dv = tc::sdesc(smem_u32(smem + kOffV), 128u, 1024u);
    const uint32_t dv_lo = (uint32_t)dv, dv_hi = (uint32_t)(dv >> 32);
    for (int t = 0; t < nt; ++t) {   // O += P(t) V(t)
      const int b = t & 1, j = t % kSP;
      if (!wait(&p_full[j], (uint32_t)(t / kSP) & 1u) || !wait(&v_full[b], (uint32_t)(t >> 1) & 1u)) break;
      tc::fence_after();
      const uint32_t vb = dv_lo + (uint32_t)b * (2 * kTile >> 4);
      const uint32_t aP = tmem + kColSP + 128u * j;
#pragma unroll
      for (int pr = 0; pr < (kLo ? 3 : 2); ++pr)   // (p_hi, v_hi), (p_lo, v_hi), (p_hi, v_lo)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t a = aP + (pr == 1 ? 32u : 0u) + 8u * ks;
          const uint32_t bl = vb + (uint32_t)(((pr == 2 ? kTile : 0) + ks * 256) / 16);
          if (t == 0 && pr == 0 && ks == 0) tc::mma_ts_c<false>(tmem + kColO, a, bl, dv_hi, kIdPV);
          else tc::mma_ts_c<true>(tmem + kColO, a, bl, dv_hi, kIdPV);
        }
      tc::commit(&pv_done[j]);
    }
    tc::commit(&drain[1]);
    mbar_wait(&drain[1], 0u, kDrainPolls);
  }
  __syncthreads();

  // ---- a split unit: the last part to finish merges the partials
  volatile int32_t* order = reinterpret_cast<volatile int32_t*>(tmem_slot + 2);
  if (split) {
    __threadfence();   // this part's partial before its count
    __syncthreads();
    if (tid == 0) *order = atomicAdd(p.counters + unit, 1);
    __syncthreads();
    if (*order == np - 1 && tid < 2 * kRows) {
      __threadfence();
      const int row = tid & (kRows - 1), ch = tid >> 7;   // 64 columns each
      const float* p0 = p.partial + ((int64_t)(unit * p.parts) * kRows + row) * kPartStride;
      const int64_t ps = (int64_t)kRows * kPartStride;    // between parts
      float m = -INFINITY;
      for (int k = 0; k < np; ++k) m = fmaxf(m, __ldcg(p0 + k * ps + kD));
      float* r = rows + row * kPitch + 64 * ch;
#pragma unroll 4
      for (int c = 0; c < 64; ++c) r[c] = 0.0f;
      float lt = 0.0f;
      for (int k = 0; k < np; ++k) {
        const float* pk = p0 + k * ps;
        const float mk = __ldcg(pk + kD), fk = mk == -INFINITY ? 0.0f : ex2(mk - m);
        lt = fmaf(__ldcg(pk + kD + 1), fk, lt);
#pragma unroll 4
        for (int c = 0; c < 64; c += 4) {
          const float4 a = __ldcg(reinterpret_cast<const float4*>(pk + 64 * ch + c));
          r[c] = fmaf(a.x, fk, r[c]);
          r[c + 1] = fmaf(a.y, fk, r[c + 1]);
          r[c + 2] = fmaf(a.z, fk, r[c + 2]);
          r[c + 3] = fmaf(a.w, fk, r[c + 3]);
        }
      }
      const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
#pragma unroll 4
      for (int c = 0; c < 64; ++c) r[c] *= inv;
    }
    __syncthreads();
  }
  const bool write_out = !split || *order == np - 1;

  // ---- outputs: rotate back with U^T (warp per row) and store
  {
    const uint32_t sgn = lane_signs<4>(rp, lane);
    float4 qt[1], qtr[1];
    lane_quats<4>(rp, lane, qt);
    lane_quats_r<4>(rp, lane, qtr);
    const bool so4 = rot_so4(rp), pair = rot_pair(rp);
    for (int row = warp; write_out && row < nrows; row += kThreads / 32) {
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
  if (warp == kMmaWarp) tc::dealloc(tmem, kTmemCols);
}

template <int SCALE, int BITS>
kvq3_status launch_tc(const TcParams& p, const RotParams& rp, cudaStream_t st) {
  auto k = prefill_tc_kernel<SCALE, BITS>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return KVQ3_ERR_CUDA;
  const dim3 grid((unsigned)(p.parts * ((p.n + p.qb - 1) / p.qb)), (unsigned)p.g.hkv);
  k<<<grid, kThreads, kSmem, st>>>(p, rp);
  return cudaGetLastError() == cudaSuccess ? KVQ3_OK : KVQ3_ERR_CUDA;
}

template <int BITS>
kvq3_status launch_bits(const CacheGeom& g, const TcParams& p, const RotParams& rp, cudaStream_t st) {
  if constexpr (BITS == 3)
    if (g.scale_type == KVQ3_SCALE_E4M3_ZP) return launch_tc<KVQ3_SCALE_E4M3_ZP, 3>(p, rp, st);
  if (g.scale_type == KVQ3_SCALE_F32) return launch_tc<KVQ3_SCALE_F32, BITS>(p, rp, st);
  if (g.scale_type == KVQ3_SCALE_F16) return launch_tc<KVQ3_SCALE_F16, BITS>(p, rp, st);
  return launch_tc<KVQ3_SCALE_E4M3, BITS>(p, rp, st);
}

}  // namespace

namespace kvq3 {

bool prefill_tc_supported(const CacheGeom& g, int32_t hq) {
  return g.d == kD && g.bits >= 2 && g.bits <= 4 && g.block == 64 &&
         (g.scale_type != KVQ3_SCALE_E4M3_ZP || g.bits == 3) && hq / g.hkv <= kRows;
}

// Workspace of the tcgen05 path: one counter per unit (128 query rows of a kv
// head), then per unit one partial of 128 rows x kPartStride floats per CTA
// the unit can run as (parts_for the longest context the cache holds).
// CTAs per unit for units of up to `tiles` key tiles: enough for kChain
// tiles each, at least 2, at most kMaxParts
static int parts_for(int64_t tiles) {
  return (int)std::min<int64_t>(kMaxParts, std::max<int64_t>(2, (tiles + kChain - 1) / kChain));
}

size_t prefill_tc_workspace(const CacheGeom& g, int32_t hq, int64_t n_q) {
  const int64_t units = (n_q + kRows / (hq / g.hkv) - 1) / (kRows / (hq / g.hkv)) * g.hkv;
  const int parts = parts_for(((int64_t)g.max_pages * g.page_size + kKeys - 1) / kKeys);   // the longest context the cache holds
  return (size_t)((units * 4 + 255) / 256 * 256) + (size_t)units * parts * kRows * kPartStride * sizeof(float);
}

// tcgen05 path of kvq3_prefill_attn; arguments already checked.
kvq3_status prefill_tc(const CacheGeom& g, const kvq3_cache* cache, int32_t seq, int64_t pos0, int64_t n_q,
                       const void* q, int32_t hq, float qk_scale, float* out, void* workspace, size_t ws_bytes,
                       int32_t* dev_status, const RotParams& rp, uint32_t wait_limit, cudaStream_t st) {
  if (!prefill_tc_supported(g, hq)) return KVQ3_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < prefill_tc_workspace(g, hq, n_q)) return KVQ3_ERR_WORKSPACE;
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
  const int64_t units = (n_q + p.qb - 1) / p.qb * g.hkv;
  const size_t cbytes = (size_t)((units * 4 + 255) / 256 * 256);
  // the longest unit (the last query block) attends to pos0 + n_q keys; the
  // workspace holds parts_for() of the cache's capacity, which is not less
  p.parts = std::min(parts_for((pos0 + n_q + kKeys - 1) / kKeys),
                     parts_for(((int64_t)g.max_pages * g.page_size + kKeys - 1) / kKeys));
  p.counters = static_cast<int32_t*>(workspace);
  p.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + cbytes);
  p.ws_floats = (int64_t)((ws_bytes - cbytes) / sizeof(float));
  if (cudaMemsetAsync(workspace, 0, (size_t)units * 4, st) != cudaSuccess) return KVQ3_ERR_CUDA;
  return g.bits == 2 ? launch_bits<2>(g, p, rp, st) : g.bits == 4 ? launch_bits<4>(g, p, rp, st)
                      : launch_bits<3>(g, p, rp, st);
}

}  // namespace kvq3
