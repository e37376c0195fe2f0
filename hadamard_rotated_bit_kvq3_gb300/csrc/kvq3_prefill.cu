// Chunked-prefill attention over the packed cache with shared dequantised
// tiles (head dimension 128).
//
// "Orthogonally mixed 3-bit KV cache", Implementation notes (read path) and
// Key formulas, with the causal mask of a prefill chunk: query token i sits at
// position pos0 + i and attends to positions [0, pos0 + i] of its sequence.
//
// Design (FlashAttention-style, one GPU):
//  * one CTA per (kv head, block of 64 query rows); a row is (query token,
//    query head of the kv head), 64 / G tokens x G heads; 4 warps x 16 rows;
//  * the CTA walks 64-key tiles of the sequence up to its last row's
//    position: packed K and V code strings are staged with cp.async (double
//    buffered), scales are read and widened to fp32, and every tile is
//    dequantised ONCE into shared memory, as exact fp16 small integers laid
//    out in mma.sync fragment order, then read by all 64 rows;
//  * QK^T: q1 = U q (scaled by sm_scale*log2e and a per-row power of two) as
//    hi + lo fp16 halves against the integer codes, one accumulator per scale
//    block, times the per-(key, block) key scale in fp32;
//  * online softmax per row (base 2), causal mask on the tiles that cross a
//    row's position; the probability fragments are reused as the A operand of
//    PV (the QK^T accumulator layout is the PV operand layout), times the
//    per-(key, block) value scale and split into hi + lo fp16 halves;
//  * the rows' outputs are rotated back with U^T through shared memory.
#include <string.h>

#include "kvq3_internal.h"

using namespace kvq3;

namespace {

constexpr int kWarpsP = 4;
constexpr int kRowsP = 16 * kWarpsP;   // query rows per CTA
constexpr int kKeysP = 64;             // keys per tile
constexpr int kThreadsP = 32 * kWarpsP;
constexpr int kD = 128;                // head dimension of this kernel
constexpr int kCB = 3 * kD / 8;        // code bytes per vector (48)

struct PrefillParams {
  CacheGeom g;
  const uint8_t* pool;
  const int32_t* page_table;
  const __half* q;      // [n][Hq][D]
  float* out;           // [n][Hq][D]
  int32_t* status;
  int32_t seq, n, Hq, G, qb;   // qb: query tokens per CTA (kRowsP / G)
  int64_t pos0;
  float qk_scale;       // sm_scale * log2(e)
  float inv_sqrt_d;
};

// Shared memory (bytes)
constexpr int kOffKc = 0;                                  // [2][64][48] packed K codes
constexpr int kOffVc = kOffKc + 2 * kKeysP * kCB;          // [2][64][48] packed V codes
constexpr int kOffKs = kOffVc + 2 * kKeysP * kCB;          // [2][64][4] K scales (fp32)
constexpr int kOffVs = kOffKs + 2 * kKeysP * 4 * 4;        // [2][64][4] V scales (fp32)
constexpr int kOffQinv = kOffVs + 2 * kKeysP * 4 * 4;      // [64] per-row inverse q scale
constexpr int kOffKf = (kOffQinv + kRowsP * 4 + 127) / 128 * 128;   // [8 ks][8 nt][32] uint2
constexpr int kOffVf = kOffKf + 8 * 8 * 32 * 8;            // [4 ks][16 nt][32] uint2
constexpr int kSmemP = kOffVf + 4 * 16 * 32 * 8;
static_assert(kRowsP * kD * 4 <= 8 * 8 * 32 * 8 + 4 * 16 * 32 * 8, "row staging aliases Kf+Vf");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;   // zero-fill when invalid
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

// two 3-bit two's-complement fields (bits 0-2 and 3-5 of w6) -> half2 of the
// exact integers (c0, c1): (0x6400 | (c + 4)) - 1028
__device__ __forceinline__ uint32_t codes2_to_half2(uint32_t w6) {
  const uint32_t x = (w6 & 63u) * 0x2001u;                  // field 1 to bits 16-18
  const uint32_t h = (x & 0x00070007u) ^ 0x64046404u;       // 1024 + (c + 4)
  __half2 v = *reinterpret_cast<const __half2*>(&h);
  v = __hsub2(v, __halves2half2(__ushort_as_half(0x6404), __ushort_as_half(0x6404)));
  return *reinterpret_cast<uint32_t*>(&v);
}
// one field (bits 0-2 of w) and another (bits 0-2 of u) -> half2 (c_w, c_u)
__device__ __forceinline__ uint32_t code_pair_to_half2(uint32_t w, uint32_t u) {
  const uint32_t x = (w & 7u) | ((u & 7u) << 16);
  const uint32_t h = x ^ 0x64046404u;
  __half2 v = *reinterpret_cast<const __half2*>(&h);
  v = __hsub2(v, __halves2half2(__ushort_as_half(0x6404), __ushort_as_half(0x6404)));
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int BLOCK, int SCALE>
__global__ void __launch_bounds__(kThreadsP, 2) prefill_tile_kernel(const __grid_constant__ PrefillParams p,
                                                                    const __grid_constant__ RotParams rp) {
  constexpr int NB = kD / BLOCK;
  constexpr int SB = SCALE == KVQ3_SCALE_F32 ? 4 : SCALE == KVQ3_SCALE_F16 ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int j = lane & 3, r = lane >> 2;
  const uint32_t sbase = smem_u32(smem);
  float* ks_s = reinterpret_cast<float*>(smem + kOffKs);
  float* vs_s = reinterpret_cast<float*>(smem + kOffVs);
  float* qinv_s = reinterpret_cast<float*>(smem + kOffQinv);
  uint2* kf = reinterpret_cast<uint2*>(smem + kOffKf);
  uint2* vf = reinterpret_cast<uint2*>(smem + kOffVf);
  float* rows_s = reinterpret_cast<float*>(smem + kOffKf);   // [64][128] q1 / outputs (aliases Kf+Vf)
  const CacheGeom& g = p.g;
  const int kvh = blockIdx.y;
  const int t0 = blockIdx.x * p.qb;                          // first query token of the block
  const int ntok = min(p.qb, p.n - t0);
  const int nrows = ntok * p.G;
  const int64_t kmax = p.pos0 + t0 + ntok - 1;               // last position any row attends to
  const int ntiles = (int)(kmax / kKeysP) + 1;
  const uint32_t REC = (uint32_t)g.record_bytes, HDR = (uint32_t)g.scale_hdr_bytes;

  // ---- q1 = U q of this CTA's rows into shared memory (warp per row)
  {
    const uint32_t sgn = lane_signs<4>(rp, lane);
    float4 qt[1], qtr[1];
    lane_quats<4>(rp, lane, qt);
    lane_quats_r<4>(rp, lane, qtr);
    const bool so4 = rot_so4(rp), pair = rot_pair(rp);
    for (int row = wid; row < kRowsP; row += kWarpsP) {
      float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (row < nrows) {
        const int tok = t0 + row / p.G, h = kvh * p.G + row % p.G;
        const __half* src = p.q + ((int64_t)tok * p.Hq + h) * kD + lane * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = __half2float(src[e]);
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
      ex = max(-100, min(100, 8 - ex));                     // row max scaled into (2^7, 2^8]
      const float sc = ldexpf(1.0f, ex);
#pragma unroll
      for (int e = 0; e < 4; ++e) rows_s[row * kD + lane * 4 + e] = x[e] * sc;
      if (lane == 0) qinv_s[row] = ldexpf(1.0f, -ex);
    }
  }
  __syncthreads();
  // A fragments of this warp's 16 rows: [k-step][4 regs], hi and lo halves
  uint32_t qa_hi[8][4], qa_lo[8][4];
  {
    const int row0 = wid * 16 + r, row1 = row0 + 8;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int row = (q4 & 1) ? row1 : row0;
        const int col = 16 * s + 2 * j + ((q4 & 2) ? 8 : 0);
        const float a = rows_s[row * kD + col], b = rows_s[row * kD + col + 1];
        const __half2 hi = __floats2half2_rn(a, b);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(a - hf.x, b - hf.y);
        qa_hi[s][q4] = *reinterpret_cast<const uint32_t*>(&hi);
        qa_lo[s][q4] = *reinterpret_cast<const uint32_t*>(&lo);
      }
    }
  }
  const float qinv0 = qinv_s[wid * 16 + r], qinv1 = qinv_s[wid * 16 + r + 8];
  // causal limits of this lane's two rows (rows past the chunk: no keys)
  const int rowA = wid * 16 + r, rowB = rowA + 8;
  const int64_t limA = rowA < nrows ? p.pos0 + t0 + rowA / p.G : -1;
  const int64_t limB = rowB < nrows ? p.pos0 + t0 + rowB / p.G : -1;
  __syncthreads();   // rows_s (aliasing Kf/Vf) is rewritten by the first tile

  // ---- staging of a tile's packed codes (cp.async) and scales (loads)
  auto stage = [&](int tile, int buf) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int pi = tid + kThreadsP * k;      // 384 pieces: [K|V][64 keys][3 x 16 B]
      const int which = pi / 192, rem = pi % 192, key = rem / 3, part = rem % 3;
      const int64_t pos = (int64_t)tile * kKeysP + key;
      int64_t page = -1;
      if (pos <= kmax) page = page_of(g, p.page_table, p.seq, pos / g.page_size);
      const bool ok = page >= 0;
      const int slot = ok ? (int)(pos % g.page_size) : 0;
      const uint8_t* src = p.pool + (ok ? page * g.page_bytes + (int64_t)(kvh * 2 + which) * REC + HDR +
                                              (int64_t)slot * kCB + part * 16
                                        : 0);
      const uint32_t dst = sbase + (which ? kOffVc : kOffKc) + (uint32_t)(buf * kKeysP * kCB + key * kCB + part * 16);
      cp_async16(dst, ok ? (const void*)src : (const void*)p.pool, ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto stage_scales = [&](int tile, int buf) {
    const int which = tid >> 6, key = tid & 63;
    const int64_t pos = (int64_t)tile * kKeysP + key;
    int64_t page = -1;
    if (pos <= kmax) {
      page = page_of(g, p.page_table, p.seq, pos / g.page_size);
      if (page < 0 && which == 0) set_status(p.status, KVQ3_DEV_BAD_PAGE);
    }
    float* dst = (which ? vs_s : ks_s) + (buf * kKeysP + key) * 4;
    if (page >= 0) {
      const uint8_t* sp = p.pool + page * g.page_bytes + (int64_t)(kvh * 2 + which) * REC +
                          (int64_t)(pos % g.page_size) * NB * SB;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        uint32_t bits;
        if (SB == 4) bits = reinterpret_cast<const uint32_t*>(sp)[b];
        else if (SB == 2) bits = reinterpret_cast<const uint16_t*>(sp)[b];
        else bits = sp[b];
        dst[b] = decode_scale(bits, SCALE);
      }
    } else {
#pragma unroll
      for (int b = 0; b < NB; ++b) dst[b] = 0.0f;
    }
  };

  // ---- dequantise a staged tile into fragment order (all 128 threads)
  auto dequant = [&](int buf) {
    {   // K: thread = (key, half of the dims); B operand of QK: [k-step][n-tile][lane] (b0, b1)
      const int key = tid >> 1, hdim = tid & 1;
      const uint32_t* w = reinterpret_cast<const uint32_t*>(smem + kOffKc + buf * kKeysP * kCB + key * kCB + hdim * 24);
      uint32_t wd[7];
#pragma unroll
      for (int i = 0; i < 6; ++i) wd[i] = w[i];
      wd[6] = 0;
      const int nt = key >> 3, rr = key & 7;
#pragma unroll
      for (int i = 0; i < 32; ++i) {            // dims 64*hdim + 2i, +1
        const int bit = 6 * i;
        const uint32_t w6 = __funnelshift_r(wd[bit >> 5], wd[(bit >> 5) + 1], bit & 31);
        const int d = 64 * hdim + 2 * i;
        const int s = d >> 4, kk = d & 15, jj = (kk & 7) >> 1, reg = kk >> 3;
        reinterpret_cast<uint32_t*>(&kf[(s * 8 + nt) * 32 + rr * 4 + jj])[reg] = codes2_to_half2(w6);
      }
    }
    {   // V: thread = (key pair, quarter of the dims); B operand of PV: [k-step][n-tile][lane]
      const int kp = tid >> 2, dq = tid & 3;      // keys 2kp, 2kp+1; dims 32dq ..
      const uint32_t* w0 = reinterpret_cast<const uint32_t*>(smem + kOffVc + buf * kKeysP * kCB + (2 * kp) * kCB + dq * 12);
      const uint32_t* w1 = w0 + kCB / 4;
      uint32_t a[4], b[4];
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        a[i] = w0[i];
        b[i] = w1[i];
      }
      a[3] = b[3] = 0;
      const int key = 2 * kp, ks = key >> 4, kk = key & 15, jj = (kk & 7) >> 1, reg = kk >> 3;
#pragma unroll
      for (int f = 0; f < 32; ++f) {            // dim 32dq + f
        const int bit = 3 * f;
        const uint32_t u0 = __funnelshift_r(a[bit >> 5], a[(bit >> 5) + 1], bit & 31);
        const uint32_t u1 = __funnelshift_r(b[bit >> 5], b[(bit >> 5) + 1], bit & 31);
        const int d = 32 * dq + f, nt = d >> 3, rr = d & 7;
        reinterpret_cast<uint32_t*>(&vf[(ks * 16 + nt) * 32 + rr * 4 + jj])[reg] = code_pair_to_half2(u0, u1);
      }
    }
  };

  // ---- state of this lane's rows: running max, partial sums, output accumulators
  float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nt][c] = 0.0f;

  stage(0, 0);
  stage_scales(0, 0);
  for (int tile = 0; tile < ntiles; ++tile) {
    const int buf = tile & 1;
    if (tile + 1 < ntiles) {
      stage(tile + 1, buf ^ 1);
      stage_scales(tile + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();          // codes and scales of this tile visible; Kf/Vf free
    dequant(buf);
    __syncthreads();          // fragments ready
    const float* ksb = ks_s + buf * kKeysP * 4;
    const float* vsb = vs_s + buf * kKeysP * 4;

    // ---- S = (q1 . c_k) per block, times the key scale, summed over blocks
    float sacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) sacc[nt][c] = 0.0f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float tb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int s = b * BLOCK / 16; s < (b + 1) * BLOCK / 16; ++s) {
          const uint2 kb = kf[(s * 8 + nt) * 32 + lane];
          mma_16816(tb, qa_hi[s], kb.x, kb.y);
          mma_16816(tb, qa_lo[s], kb.x, kb.y);
        }
        const int key0 = nt * 8 + 2 * j;
        const float sk0 = ksb[key0 * 4 + b], sk1 = ksb[(key0 + 1) * 4 + b];
        sacc[nt][0] = fmaf(tb[0], sk0, sacc[nt][0]);
        sacc[nt][1] = fmaf(tb[1], sk1, sacc[nt][1]);
        sacc[nt][2] = fmaf(tb[2], sk0, sacc[nt][2]);
        sacc[nt][3] = fmaf(tb[3], sk1, sacc[nt][3]);
      }
    }
    // ---- causal mask, online softmax (base 2)
    const int64_t kbase = (int64_t)tile * kKeysP;
    float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int64_t k0 = kbase + nt * 8 + 2 * j;
      sacc[nt][0] = k0 <= limA ? sacc[nt][0] * qinv0 : -INFINITY;
      sacc[nt][1] = k0 + 1 <= limA ? sacc[nt][1] * qinv0 : -INFINITY;
      sacc[nt][2] = k0 <= limB ? sacc[nt][2] * qinv1 : -INFINITY;
      sacc[nt][3] = k0 + 1 <= limB ? sacc[nt][3] * qinv1 : -INFINITY;
      mxA = fmaxf(mxA, fmaxf(sacc[nt][0], sacc[nt][1]));
      mxB = fmaxf(mxB, fmaxf(sacc[nt][2], sacc[nt][3]));
    }
    mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 1));
    mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 2));
    mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 1));
    mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 2));
    const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
    const float aA = nA == -INFINITY ? 1.0f : ex2(mA - nA);   // rows with no key yet keep 1
    const float aB = nB == -INFINITY ? 1.0f : ex2(mB - nB);
    mA = nA;
    mB = nB;
    const float rA = mA == -INFINITY ? 0.0f : mA, rB = mB == -INFINITY ? 0.0f : mB;
    lA *= aA;
    lB *= aB;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= aA;
      o[nt][1] *= aA;
      o[nt][2] *= aB;
      o[nt][3] *= aB;
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      sacc[nt][0] = ex2(sacc[nt][0] - rA);
      sacc[nt][1] = ex2(sacc[nt][1] - rA);
      sacc[nt][2] = ex2(sacc[nt][2] - rB);
      sacc[nt][3] = ex2(sacc[nt][3] - rB);
      lA += sacc[nt][0] + sacc[nt][1];
      lB += sacc[nt][2] + sacc[nt][3];
    }
    // ---- O += P' V: the S fragments of n-tiles 2ks, 2ks+1 are the A operand of
    // k-step ks; P' = p * s_v[key][block], split into hi + lo halves
#pragma unroll
    for (int ksp = 0; ksp < 4; ++ksp) {
      const int key0 = ksp * 16 + 2 * j, key8 = key0 + 8;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float v0 = vsb[key0 * 4 + b], v1 = vsb[(key0 + 1) * 4 + b];
        const float v8 = vsb[key8 * 4 + b], v9 = vsb[(key8 + 1) * 4 + b];
        const float y[8] = {sacc[2 * ksp][0] * v0,     sacc[2 * ksp][1] * v1,
                            sacc[2 * ksp][2] * v0,     sacc[2 * ksp][3] * v1,
                            sacc[2 * ksp + 1][0] * v8, sacc[2 * ksp + 1][1] * v9,
                            sacc[2 * ksp + 1][2] * v8, sacc[2 * ksp + 1][3] * v9};
        uint32_t ahi[4], alo[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const __half2 hi = __floats2half2_rn(y[2 * q4], y[2 * q4 + 1]);
          const float2 hf = __half22float2(hi);
          const __half2 lo = __floats2half2_rn(y[2 * q4] - hf.x, y[2 * q4 + 1] - hf.y);
          ahi[q4] = *reinterpret_cast<const uint32_t*>(&hi);
          alo[q4] = *reinterpret_cast<const uint32_t*>(&lo);
        }
        // A layout: a0 = rows r (keys 2j..), a1 = rows r+8, a2 = rows r (keys 2j+8..), a3 = rows r+8
        const uint32_t Ahi[4] = {ahi[0], ahi[1], ahi[2], ahi[3]};
        const uint32_t Alo[4] = {alo[0], alo[1], alo[2], alo[3]};
#pragma unroll
        for (int nt = b * BLOCK / 8; nt < (b + 1) * BLOCK / 8; ++nt) {
          const uint2 vb = vf[(ksp * 16 + nt) * 32 + lane];
          mma_16816(o[nt], Ahi, vb.x, vb.y);
          mma_16816(o[nt], Alo, vb.x, vb.y);
        }
      }
    }
    __syncthreads();          // every warp is done with Kf/Vf and this tile's buffers
  }

  // ---- normalise, stage the rows, rotate back with U^T, store
  lA += __shfl_xor_sync(kFull, lA, 1);
  lA += __shfl_xor_sync(kFull, lA, 2);
  lB += __shfl_xor_sync(kFull, lB, 1);
  lB += __shfl_xor_sync(kFull, lB, 2);
  const float iA = lA > 0.0f ? 1.0f / lA : 0.0f, iB = lB > 0.0f ? 1.0f / lB : 0.0f;
  __syncthreads();
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int d = nt * 8 + 2 * j;
    rows_s[rowA * kD + d] = o[nt][0] * iA;
    rows_s[rowA * kD + d + 1] = o[nt][1] * iA;
    rows_s[rowB * kD + d] = o[nt][2] * iB;
    rows_s[rowB * kD + d + 1] = o[nt][3] * iB;
  }
  __syncthreads();
  {
    const uint32_t sgn = lane_signs<4>(rp, lane);
    float4 qt[1], qtr[1];
    lane_quats<4>(rp, lane, qt);
    lane_quats_r<4>(rp, lane, qtr);
    const bool so4 = rot_so4(rp), pair = rot_pair(rp);
    for (int row = wid; row < nrows; row += kWarpsP) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = rows_s[row * kD + lane * 4 + e];
      rotate_inverse<4, 32>(x, lane, sgn, qt, qtr, p.inv_sqrt_d, so4, pair);
      const int tok = t0 + row / p.G, h = kvh * p.G + row % p.G;
      float4* dst = reinterpret_cast<float4*>(p.out + ((int64_t)tok * p.Hq + h) * kD + lane * 4);
      *dst = make_float4(x[0], x[1], x[2], x[3]);
    }
  }
}

template <int BLOCK, int SCALE>
kvq3_status launch_prefill_tiles(const PrefillParams& p, const RotParams& rp, cudaStream_t st) {
  auto k = prefill_tile_kernel<BLOCK, SCALE>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP) != cudaSuccess)
    return KVQ3_ERR_CUDA;
  const dim3 grid((unsigned)((p.n + p.qb - 1) / p.qb), (unsigned)p.g.hkv);
  k<<<grid, kThreadsP, kSmemP, st>>>(p, rp);
  return cudaGetLastError() == cudaSuccess ? KVQ3_OK : KVQ3_ERR_CUDA;
}

}  // namespace

namespace kvq3 {

// Tile-kernel path of kvq3_prefill_attn (d = 128); arguments already checked.
kvq3_status prefill_tiles(const CacheGeom& g, const kvq3_cache* cache, int32_t seq, int64_t pos0,
                          int64_t n_q, const void* q, int32_t hq, float qk_scale, float* out,
                          int32_t* dev_status, const RotParams& rp, cudaStream_t st) {
  if (g.d != kD) return KVQ3_ERR_UNSUPPORTED;
  PrefillParams p;
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
  p.qb = kRowsP / p.G;
  p.pos0 = pos0;
  p.qk_scale = qk_scale;
  p.inv_sqrt_d = inv_sqrt(g.d);
  const int sc = g.scale_type;
  if (g.block == 32) {
    if (sc == KVQ3_SCALE_F32) return launch_prefill_tiles<32, KVQ3_SCALE_F32>(p, rp, st);
    if (sc == KVQ3_SCALE_F16) return launch_prefill_tiles<32, KVQ3_SCALE_F16>(p, rp, st);
    return launch_prefill_tiles<32, KVQ3_SCALE_E4M3>(p, rp, st);
  }
  if (sc == KVQ3_SCALE_F32) return launch_prefill_tiles<64, KVQ3_SCALE_F32>(p, rp, st);
  if (sc == KVQ3_SCALE_F16) return launch_prefill_tiles<64, KVQ3_SCALE_F16>(p, rp, st);
  return launch_prefill_tiles<64, KVQ3_SCALE_E4M3>(p, rp, st);
}

}  // namespace kvq3
