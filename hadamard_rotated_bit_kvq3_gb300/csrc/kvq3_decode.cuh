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
//  * Work = the flattened list of (sequence, kv head, page) triples.  A
//    persistent grid of warps splits it into equal contiguous ranges; a warp
//    keeps an online-softmax state per (sequence, kv head) segment and writes
//    one fp32 partial (o1[G][d] unnormalised, max, sum) per segment to the
//    workspace, at slot (warp + unit), which is unique because ranges and
//    units are both ordered.  A second kernel merges the partials of each
//    (sequence, query head) with the log-sum-exp rule and applies U^T.
//  * Each page's K and V records of one kv head are contiguous; one lane
//    streams them with cp.async.bulk into a per-warp ring of shared-memory
//    stages (mbarrier completion, L2 evict-first), several pages ahead.
//  * QK^T and PV run on tensor cores (mma.sync m16n8k16, fp16 in, fp32
//    accumulate).  Codes in -3..3 become exact fp16 values by a mask/xor into
//    the 0x6400 exponent pattern and one half2 subtraction; the field's bit
//    offset inside the half leaves a power-of-two factor that is folded into
//    q1 (keys) or into the output (values).  q1 is split into hi + lo fp16
//    halves (two columns per head) so the logits keep ~fp32 accuracy;
//    per-(token, block) scales multiply the per-block partial dot products
//    (keys) or the probabilities (values).
#pragma once

#include <float.h>

#include "kvq3_internal.h"

namespace kvq3 {

struct DecodeParams {
  CacheGeom g;
  const uint8_t* pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const __half* q;        // [B][Hq][D]
  float* ws;              // partial slots
  int32_t* status;
  int32_t G;              // query heads per kv head
  int32_t Hq;
  float qk_scale;         // sm_scale * log2(e)
  float inv_sqrt_d;
  int32_t stages;         // ring depth per warp
  uint32_t stage_bytes;   // bytes per stage (copy_bytes + padding)
  uint32_t copy_bytes;    // K record + V record of one kv head
  int32_t total_warps;
  int32_t warps_per_cta;
  uint32_t slot_floats;   // floats per partial slot: G*(D+2)
  uint32_t warp_smem;     // dynamic shared memory per warp
  uint32_t wait_limit;    // bound on mbarrier polls
};

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ int64_t seq_pages(const DecodeParams& p, int b, bool flag) {
  const int64_t len = p.seq_lens[b];
  const int64_t cap = (int64_t)p.g.max_pages * p.g.page_size;
  if (len < 0 || len > cap) {
    if (flag) set_status(p.status, KVQ3_DEV_BAD_LEN);
    return 0;
  }
  return (len + p.g.page_size - 1) / p.g.page_size;
}

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Total pages over all (sequence, kv head) units.
__device__ __forceinline__ int64_t total_pages(const DecodeParams& p, bool flag) {
  const int lane = threadIdx.x & 31;
  int64_t acc = 0;
  for (int b0 = 0; b0 < p.g.batch; b0 += 32) {
    const int b = b0 + lane;
    acc += warp_sum64(b < p.g.batch ? seq_pages(p, b, flag) : 0);
  }
  return acc * p.g.hkv;
}

// Hkv * (pages of sequences 0..b-1).
__device__ __forceinline__ int64_t pages_before(const DecodeParams& p, int b) {
  const int lane = threadIdx.x & 31;
  int64_t acc = 0;
  for (int b0 = 0; b0 < b; b0 += 32) {
    const int bb = b0 + lane;
    acc += warp_sum64(bb < b ? seq_pages(p, bb, false) : 0);
  }
  return acc * p.g.hkv;
}

// Position in the flattened page list: sequence b, kv head, logical page.
struct Cursor {
  int b, kvh;
  int64_t lp, np;
};

__device__ __forceinline__ Cursor cursor_at(const DecodeParams& p, int64_t pidx) {
  const int lane = threadIdx.x & 31;
  int64_t acc = 0;
  Cursor c{p.g.batch, 0, 0, 0};
  for (int b0 = 0; b0 < p.g.batch; b0 += 32) {
    const int b = b0 + lane;
    const int64_t np = b < p.g.batch ? seq_pages(p, b, false) * p.g.hkv : 0;
    int64_t incl = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t excl = incl - np;
    const unsigned hit = __ballot_sync(kFull, np > 0 && acc + excl <= pidx && pidx < acc + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const int64_t base = acc + __shfl_sync(kFull, excl, src);
      const int64_t npb = __shfl_sync(kFull, np, src) / p.g.hkv;
      const int64_t within = pidx - base;
      c.b = b0 + src;
      c.np = npb;
      c.kvh = (int)(within / npb);
      c.lp = within % npb;
      return c;
    }
    acc += __shfl_sync(kFull, incl, 31);
  }
  return c;
}

__device__ __forceinline__ void cursor_next(const DecodeParams& p, Cursor& c) {
  if (++c.lp < c.np) return;
  c.lp = 0;
  if (++c.kvh < p.g.hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
    c.np = c.b < p.g.batch ? seq_pages(p, c.b, false) : 0;
  } while (c.b < p.g.batch && c.np == 0);
}

// Scales of one token's record: NB values of the runtime scale type.
template <int NB>
__device__ __forceinline__ void load_scales(const uint8_t* hdr, int tok, int type, float (&s)[NB]) {
  if (type == KVQ3_SCALE_F32) {
    const float* f = reinterpret_cast<const float*>(hdr) + tok * NB;
#pragma unroll
    for (int i = 0; i < NB; ++i) s[i] = f[i];
  } else if (type == KVQ3_SCALE_F16) {
    const __half* h = reinterpret_cast<const __half*>(hdr) + tok * NB;
#pragma unroll
    for (int i = 0; i < NB; ++i) s[i] = __half2float(h[i]);
  } else {
    const uint8_t* b = hdr + tok * NB;
#pragma unroll
    for (int i = 0; i < NB; ++i) s[i] = decode_scale(b[i], KVQ3_SCALE_E4M3);
  }
}

// half2 subtraction on raw bits
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a);
  const __half2 y = *reinterpret_cast<const __half2*>(&b);
  x = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&x);
}

// Key codes: a lane's F consecutive fields (F = 16 or 8) in (lo, hi) ->
// F/2 half2 values.  Pair k holds field lf(k) = 8(k/4) + k%4 in its low half
// scaled by 2^(4 or 7) and field lf(k)+4 in its high half scaled by 2^(0 or 3)
// (odd k take the larger offsets).
__host__ __device__ constexpr int kq_lo_field(int k) { return 8 * (k / 4) + (k % 4); }
__host__ __device__ constexpr int kq_lo_off(int k) { return (k & 1) ? 7 : 4; }
__host__ __device__ constexpr int kq_hi_off(int k) { return (k & 1) ? 3 : 0; }

template <int F>
__device__ __forceinline__ void k_codes_to_half2(uint32_t lo, uint32_t hi, uint32_t (&h)[F / 2]) {
#pragma unroll
  for (int k = 0; k < F / 2; ++k) {
    const int i = 8 * (k / 4) + (k & 2);  // first field of the window
    const int o = 3 * i - 4;              // window start bit: field i lands at bit 4
    const uint32_t w = o < 0 ? (lo << (-o)) : __funnelshift_r(lo, hi, o);
    if (k & 1) h[k] = hsub2_bits((w & 0x00380380u) ^ 0x64206600u, 0x64206600u);
    else h[k] = hsub2_bits((w & 0x00070070u) ^ 0x64046440u, 0x64046440u);
  }
}

// Value codes: fields f = 0..F-1 (F = 8 or 4) of two tokens' 3F-bit chunks
// c0, c1 -> half2 (token0, token1) of field f scaled by 2^voff(f).
__host__ __device__ constexpr int v_off(int f) {
  return f == 0 ? 0 : f == 1 ? 3 : f == 2 ? 6 : f == 3 ? 1 : f == 4 ? 4 : f == 5 ? 7 : f == 6 ? 2 : 5;
}

template <int F>
__device__ __forceinline__ void v_codes_to_half2(uint32_t c0, uint32_t c1, uint32_t (&h)[F]) {
  const uint32_t wa = __byte_perm(c0, c1, 0x5410);
  const uint32_t wb = __byte_perm(c0, c1, 0x6521);
  const uint32_t wc = __byte_perm(c0, c1, 0x7632);
#pragma unroll
  for (int f = 0; f < F; ++f) {
    const uint32_t w = f < 3 ? wa : (f < 6 ? wb : wc);
    const int o = v_off(f);
    const uint32_t x = 0x64006400u | (0x00040004u << o);
    h[f] = hsub2_bits((w & (0x00070007u << o)) ^ x, x);
  }
}

// 3*F bits of a code string starting at bit `boff` (two aligned words).
__device__ __forceinline__ void load_bits(const uint8_t* str, int boff, uint32_t& lo, uint32_t& hi) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(str) + (boff >> 5);
  const int sh = boff & 31;
  const uint32_t w0 = w[0], w1 = w[1];
  lo = __funnelshift_r(w0, w1, sh);
  hi = w1 >> sh;
}

// ------------------------------------------------------------------ kernel 1
template <int D, int GPAD>
struct DecodeSmem {
  static constexpr int kBarBytes = 64;  // up to 8 mbarriers
  static constexpr int kQOff = kBarBytes;
  static constexpr int kQInvOff = kQOff + GPAD * D * 4;
  static constexpr int kStageOff = ((kQInvOff + GPAD * 4) + 127) / 128 * 128;
};

// PSPLIT: the probabilities-times-value-scales P' enter PV as hi + lo fp16
// halves too (PV n-tile = 4 heads x (hi, lo), like QK); otherwise one fp16
// value per head (PV n-tile = 8 heads).  The split is needed when the value
// scales are fp32 (p = 1 times an fp32 scale is not an fp16 value) and free
// when G <= 4 (the 8-column tile has room).
template <int D, int BLOCK, int GPAD, bool PSPLIT>
__global__ void __launch_bounds__(128) decode_split_kernel(const __grid_constant__ DecodeParams p,
                                                           const __grid_constant__ RotParams rp) {
  constexpr int NB = D / BLOCK;
  constexpr int KS = D / 16;          // k-steps of QK^T == M-tiles of PV
  constexpr int KSB = BLOCK / 16;     // per block
  constexpr int NTQ = GPAD / 4;       // QK n-tiles: 4 heads x (hi, lo)
  constexpr int NTP = PSPLIT ? NTQ : (GPAD + 7) / 8;  // PV n-tiles
  constexpr int FQ = BLOCK / 4;       // key fields per lane per block
  constexpr int FV = BLOCK / 8;       // value fields per lane per block
  constexpr int CB = 3 * D / 8;
  constexpr int EQ = D >= 128 ? D / 32 : 4;  // query rotation layout
  constexpr int LQ = D / EQ;
  constexpr int GPWQ = 32 / LQ;
  using SM = DecodeSmem<D, GPAD>;

  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int j = lane & 3, r = lane >> 2;
  uint8_t* my = smem + (size_t)wid * p.warp_smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(my);
  float* qs = reinterpret_cast<float*>(my + SM::kQOff);
  float* qinv_s = reinterpret_cast<float*>(my + SM::kQInvOff);
  uint8_t* stg = my + SM::kStageOff;
  const int S = p.stages;

  const int64_t gw = (int64_t)blockIdx.x * p.warps_per_cta + wid;
  const int64_t T = total_pages(p, gw == 0);
  const int64_t W = p.total_warps;
  const int64_t p0 = gw * T / W, p1 = (gw + 1) * T / W;
  if (p0 >= p1) return;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t pol = policy_evict_first();
  const int64_t npg = p1 - p0;
  Cursor cp = cursor_at(p, p0);
  Cursor cc = cp;

  auto issue = [&](const Cursor& c, int stage) {
    if (lane == 0) {
      const int64_t page = page_of(p.g, p.page_table, c.b, c.lp);
      uint8_t* dst = stg + (size_t)stage * p.stage_bytes;
      if (page >= 0) {
        mbar_expect_tx(&bars[stage], p.copy_bytes);
        bulk_g2s(dst, p.pool + record_offset(p.g, page, c.kvh, 0), p.copy_bytes, &bars[stage], pol);
      } else {
        set_status(p.status, KVQ3_DEV_BAD_PAGE);
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[stage]))
                     : "memory");
      }
    }
  };
  for (int64_t i = 0; i < npg && i < S; ++i) {
    issue(cp, (int)i);
    cursor_next(p, cp);
  }

  // per-lane query rotation parameters (dims rq*EQ ..)
  const int rq = lane % LQ, gq = lane / LQ;
  const uint32_t sgn_q = lane_signs<EQ>(rp, rq);
  float4 quat_q[EQ / 4];
  lane_quats<EQ>(rp, rq, quat_q);
  const bool so4 = (rp.flags & KVQ3_ROT_SO4) != 0;

  uint32_t qf[NTQ][KS][2];
  float qinv[NTQ];
  float m[NTQ], l[NTQ];
  float acc[KS][NTP][4];
  int cur_unit = -1;

  auto flush = [&](int unit) {
    float* slot = p.ws + (size_t)(gw + unit) * p.slot_floats;
    float* mS = slot + p.G * D;
    float* lS = mS + p.G;
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      float lt = l[tq];
      lt += __shfl_xor_sync(kFull, lt, 4);
      lt += __shfl_xor_sync(kFull, lt, 8);
      lt += __shfl_xor_sync(kFull, lt, 16);
      const int h = 4 * tq + j;
      if (r == 0 && h < p.G) {
        mS[h] = m[tq];
        lS[h] = lt;
      }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int b = mt / KSB, mp = mt % KSB;
#pragma unroll
      for (int tp = 0; tp < NTP; ++tp) {
        if constexpr (PSPLIT) {
          // columns 2j, 2j+1: head 4tp+j, hi and lo parts
          const int h = 4 * tp + j;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int f = 2 * mp + e;
            const int dim = b * BLOCK + r * FV + f;
            if (h < p.G)
              slot[h * D + dim] = (acc[mt][tp][2 * e] + acc[mt][tp][2 * e + 1]) *
                                  (1.0f / (float)(1 << v_off(f)));
          }
        } else {
#pragma unroll
          for (int reg = 0; reg < 4; ++reg) {
            const int f = 2 * mp + (reg >> 1);
            const int dim = b * BLOCK + r * FV + f;
            const int h = 8 * tp + 2 * j + (reg & 1);
            if (h < p.G) slot[h * D + dim] = acc[mt][tp][reg] * (1.0f / (float)(1 << v_off(f)));
          }
        }
      }
    }
  };

  auto setup_unit = [&](int b, int kvh) {
    // rotate the G query heads: qs[g][dim] = (U q)[dim] * sm_scale*log2e * 2^e_g
    for (int g0 = 0; g0 < GPAD; g0 += GPWQ) {
      const int g = g0 + gq;
      const bool valid = g < p.G;
      float x[EQ];
      const __half* src = p.q + ((int64_t)b * p.Hq + (int64_t)kvh * p.G + g) * D + rq * EQ;
#pragma unroll
      for (int e = 0; e < EQ; ++e) x[e] = valid ? __half2float(src[e]) : 0.0f;
      rotate_forward<EQ, LQ>(x, rq, sgn_q, quat_q, p.inv_sqrt_d, so4);
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
      if (g < GPAD) {
#pragma unroll
        for (int e = 0; e < EQ; ++e) qs[g * D + rq * EQ + e] = x[e] * sc;
        if (rq == 0) qinv_s[g] = ldexpf(1.0f, -ex);
      }
    }
    __syncwarp();
#pragma unroll
    for (int tq = 0; tq < NTQ; ++tq) {
      const int head = 4 * tq + (r >> 1);
      const int part = r & 1;
#pragma unroll
      for (int s = 0; s < KS; ++s) {
        const int b = s / KSB, sp = s % KSB;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int k = 2 * sp + hf;
          const int dlo = b * BLOCK + j * FQ + kq_lo_field(k);
          const int dhi = dlo + 4;
          const float vlo = qs[head * D + dlo] * (1.0f / (float)(1 << kq_lo_off(k)));
          const float vhi = qs[head * D + dhi] * (1.0f / (float)(1 << kq_hi_off(k)));
          const __half hlo = __float2half_rn(vlo), hhi = __float2half_rn(vhi);
          float olo, ohi;
          if (part == 0) {
            olo = __half2float(hlo);
            ohi = __half2float(hhi);
          } else {
            olo = vlo - __half2float(hlo);
            ohi = vhi - __half2float(hhi);
          }
          qf[tq][s][hf] = pack_half2(olo, ohi);
        }
      }
      qinv[tq] = qinv_s[4 * tq + j];
    }
    __syncwarp();
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
        for (int reg = 0; reg < 4; ++reg) acc[mt][tp][reg] = 0.0f;
  };

  const int stype = p.g.scale_type;
  for (int64_t i = 0; i < npg; ++i) {
    const int stage = (int)(i % S);
    const uint32_t parity = (uint32_t)((i / S) & 1);
    const int unit = cc.b * p.g.hkv + cc.kvh;
    if (unit != cur_unit) {
      if (cur_unit >= 0) flush(cur_unit);
      setup_unit(cc.b, cc.kvh);
      cur_unit = unit;
    }
    if (!mbar_wait(&bars[stage], parity, p.wait_limit)) {
      // a copy never arrived: flag it, wait (bounded) for the copies still in
      // flight so no asynchronous write outlives this warp, and stop
      if (lane == 0) set_status(p.status, KVQ3_DEV_TIMEOUT);
      for (int64_t k = i + 1; k < npg && k < i + S; ++k)
        mbar_wait(&bars[k % S], (uint32_t)((k / S) & 1), p.wait_limit);
      return;
    }
    const int64_t page = page_of(p.g, p.page_table, cc.b, cc.lp);
    if (page >= 0) {
      const int64_t len = p.seq_lens[cc.b];
      const int n_valid = (int)min((int64_t)p.g.page_size, len - cc.lp * p.g.page_size);
      const uint8_t* st = stg + (size_t)stage * p.stage_bytes;
      const uint8_t* kS = st;
      const uint8_t* kC = st + p.g.scale_hdr_bytes;
      const uint8_t* vS = st + p.g.record_bytes;
      const uint8_t* vC = vS + p.g.scale_hdr_bytes;
      for (int t0 = 0; t0 < n_valid; t0 += 16) {
        // ------------------------------------------------ S = K q1 (per block)
        float accq[NB][NTQ][4];
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int tq = 0; tq < NTQ; ++tq)
#pragma unroll
            for (int c = 0; c < 4; ++c) accq[b][tq][c] = 0.0f;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          uint32_t h0[FQ / 2], h1[FQ / 2];
          uint32_t lo, hi;
          const int boff = 3 * (b * BLOCK + j * FQ);
          load_bits(kC + (t0 + r) * CB, boff, lo, hi);
          k_codes_to_half2<FQ>(lo, hi, h0);
          load_bits(kC + (t0 + r + 8) * CB, boff, lo, hi);
          k_codes_to_half2<FQ>(lo, hi, h1);
#pragma unroll
          for (int sp = 0; sp < KSB; ++sp) {
            const uint32_t a[4] = {h0[2 * sp], h1[2 * sp], h0[2 * sp + 1], h1[2 * sp + 1]};
#pragma unroll
            for (int tq = 0; tq < NTQ; ++tq)
              mma_16816(accq[b][tq], a, qf[tq][b * KSB + sp][0], qf[tq][b * KSB + sp][1]);
          }
        }
        float skr[NB], skr8[NB];
        load_scales<NB>(kS, t0 + r, stype, skr);
        load_scales<NB>(kS, t0 + r + 8, stype, skr8);
        const bool vr = t0 + r < n_valid, vr8 = t0 + r + 8 < n_valid;
        // ------------------------------------------------ online softmax
        float pr[NTQ], pr8[NTQ];
        bool changed = false;
        float alpha[NTQ];
#pragma unroll
        for (int tq = 0; tq < NTQ; ++tq) {
          float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            s0 += skr[b] * (accq[b][tq][0] + accq[b][tq][1]);
            s1 += skr8[b] * (accq[b][tq][2] + accq[b][tq][3]);
          }
          s0 = vr ? s0 * qinv[tq] : -INFINITY;
          s1 = vr8 ? s1 * qinv[tq] : -INFINITY;
          float mx = fmaxf(s0, s1);
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
          const float mn = fmaxf(m[tq], mx);
          if (mn == -INFINITY) {
            alpha[tq] = 1.0f;
            pr[tq] = 0.0f;
            pr8[tq] = 0.0f;
          } else {
            alpha[tq] = ex2(m[tq] - mn);
            pr[tq] = ex2(s0 - mn);
            pr8[tq] = ex2(s1 - mn);
          }
          l[tq] = l[tq] * alpha[tq] + pr[tq] + pr8[tq];
          m[tq] = mn;
          changed |= alpha[tq] != 1.0f;
        }
        if constexpr (PSPLIT) {
          // this lane's PV columns belong to its own QK head 4tp + j
          if (__any_sync(kFull, changed)) {
#pragma unroll
            for (int tp = 0; tp < NTP; ++tp)
#pragma unroll
              for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[mt][tp][c] *= alpha[tp];
          }
        } else if (__any_sync(kFull, changed)) {
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
        // ------------------------------------------------ P' = p * s_v (B of PV)
        const int T0 = t0 + 2 * j;
        float x0[NTQ], x1[NTQ], x2[NTQ], x3[NTQ];
        {
          // B element (token T, column r) comes from the QK lane 4*(T%8) + head%4
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
        float sv0[NB], sv1[NB], sv2[NB], sv3[NB];
        load_scales<NB>(vS, T0, stype, sv0);
        load_scales<NB>(vS, T0 + 1, stype, sv1);
        load_scales<NB>(vS, T0 + 8, stype, sv2);
        load_scales<NB>(vS, T0 + 9, stype, sv3);
        const bool v0 = T0 < n_valid, v1 = T0 + 1 < n_valid, v2 = T0 + 8 < n_valid,
                   v3 = T0 + 9 < n_valid;
        uint32_t pb[NB][NTP][2];
        if constexpr (PSPLIT) {
#pragma unroll
          for (int tp = 0; tp < NTP; ++tp) {
            const bool hv = 4 * tp + (r >> 1) < p.G;
            const bool lo_part = (r & 1) != 0;
            auto part = [&](float v) {
              const float hi = __half2float(__float2half_rn(v));
              return lo_part ? v - hi : hi;
            };
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const float y0 = hv && v0 ? x0[tp] * sv0[b] : 0.0f;
              const float y1 = hv && v1 ? x1[tp] * sv1[b] : 0.0f;
              const float y2 = hv && v2 ? x2[tp] * sv2[b] : 0.0f;
              const float y3 = hv && v3 ? x3[tp] * sv3[b] : 0.0f;
              pb[b][tp][0] = pack_half2(part(y0), part(y1));
              pb[b][tp][1] = pack_half2(part(y2), part(y3));
            }
          }
        } else {
#pragma unroll
        for (int tp = 0; tp < NTP; ++tp) {
          const int hp = 8 * tp + r;
          const int tsel = hp >> 2;
          float y0 = 0.0f, y1 = 0.0f, y2 = 0.0f, y3 = 0.0f;
#pragma unroll
          for (int tq = 0; tq < NTQ; ++tq)
            if (tq == tsel) {
              y0 = x0[tq];
              y1 = x1[tq];
              y2 = x2[tq];
              y3 = x3[tq];
            }
          const bool hv = hp < p.G;
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            pb[b][tp][0] = pack_half2(hv && v0 ? y0 * sv0[b] : 0.0f, hv && v1 ? y1 * sv1[b] : 0.0f);
            pb[b][tp][1] = pack_half2(hv && v2 ? y2 * sv2[b] : 0.0f, hv && v3 ? y3 * sv3[b] : 0.0f);
          }
        }
        }
        // ------------------------------------------------ o1^T += V^T P'^T
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const int boff = 3 * (b * BLOCK + r * FV);
          uint32_t c0, c1, c2, c3, dummy;
          load_bits(vC + T0 * CB, boff, c0, dummy);
          load_bits(vC + (T0 + 1) * CB, boff, c1, dummy);
          load_bits(vC + (T0 + 8) * CB, boff, c2, dummy);
          load_bits(vC + (T0 + 9) * CB, boff, c3, dummy);
          uint32_t hv01[FV], hv89[FV];
          v_codes_to_half2<FV>(c0, c1, hv01);
          v_codes_to_half2<FV>(c2, c3, hv89);
#pragma unroll
          for (int mp = 0; mp < KSB; ++mp) {
            const uint32_t a[4] = {hv01[2 * mp], hv01[2 * mp + 1], hv89[2 * mp], hv89[2 * mp + 1]};
#pragma unroll
            for (int tp = 0; tp < NTP; ++tp) mma_16816(acc[b * KSB + mp][tp], a, pb[b][tp][0], pb[b][tp][1]);
          }
        }
      }
    }
    __syncwarp();
    if (i + S < npg) {
      fence_proxy_async();
      issue(cp, stage);
      cursor_next(p, cp);
    }
    cursor_next(p, cc);
  }
  if (cur_unit >= 0) flush(cur_unit);
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
  float4 qt[E / 4];
  lane_quats<E>(rp, rr, qt);
  const bool so4 = (rp.flags & KVQ3_ROT_SO4) != 0;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)p.g.batch * p.Hq;
  const int64_t T = total_pages(p, false);
  const int64_t W = p.total_warps;
  for (int64_t it = warp; it < items; it += nwarps) {
    const int b = (int)(it / p.Hq);
    const int h = (int)(it % p.Hq);
    const int kvh = h / p.G, g = h % p.G;
    const int64_t np = seq_pages(p, b, false);
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.0f;
    if (np > 0) {
      const int64_t pu = pages_before(p, b) + (int64_t)kvh * np;
      const int unit = b * p.g.hkv + kvh;
      const int64_t wlo = ((pu + 1) * W - 1) / T;
      const int64_t whi = ((pu + np) * W - 1) / T;
      float M = -INFINITY;
      // warps with an empty page range wrote nothing: skip them
      for (int64_t w = wlo; w <= whi; ++w) {
        if (w * T / W == (w + 1) * T / W) continue;
        const float* slot = p.ws + (size_t)(w + unit) * p.slot_floats;
        M = fmaxf(M, slot[p.G * D + g]);
      }
      if (M != -INFINITY) {
        float lsum = 0.0f;
        for (int64_t w = wlo; w <= whi; ++w) {
          if (w * T / W == (w + 1) * T / W) continue;
          const float* slot = p.ws + (size_t)(w + unit) * p.slot_floats;
          const float c = ex2(slot[p.G * D + g] - M);
          lsum += c * slot[p.G * D + p.G + g];
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] += c * slot[g * D + rr * E + e];
        }
        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] *= inv;
      }
    }
    rotate_inverse<E, L>(o, rr, sgn, qt, p.inv_sqrt_d, so4);
    if (grp == 0) {
#pragma unroll
      for (int e = 0; e < E; ++e) out[((int64_t)b * p.Hq + h) * D + rr * E + e] = o[e];
    }
  }
}

// ------------------------------------------------------------------ host
struct DecodePlan {
  int gpad;
  bool psplit;
  int warps_per_cta;
  int ctas;
  int stages;
  uint32_t stage_bytes, copy_bytes, warp_smem;
  size_t ws_bytes;
  const void* kernel;
};

template <int D, int BLOCK, int GPAD, bool PSPLIT>
const void* decode_kernel_ptr() {
  return reinterpret_cast<const void*>(&decode_split_kernel<D, BLOCK, GPAD, PSPLIT>);
}

// Sizes the launch for the current device.
template <int D, int BLOCK, int GPAD, bool PSPLIT>
kvq3_status decode_plan_t(const CacheGeom& g, int G, DecodePlan* plan) {
  using SM = DecodeSmem<D, GPAD>;
  plan->gpad = GPAD;
  plan->psplit = PSPLIT;
  plan->copy_bytes = (uint32_t)(2 * g.record_bytes);
  plan->stage_bytes = (plan->copy_bytes + 16 + 15) / 16 * 16;
  int stages = (int)(24576 / plan->stage_bytes);
  stages = stages < 2 ? 2 : (stages > 8 ? 8 : stages);
  int wpc = 4;
  uint32_t warp_smem = 0;
  for (;;) {
    warp_smem = (uint32_t)((SM::kStageOff + (size_t)stages * plan->stage_bytes + 127) / 128 * 128);
    if ((size_t)wpc * warp_smem <= 220 * 1024) break;
    if (stages > 2) --stages;
    else if (wpc > 1) wpc >>= 1;
    else return KVQ3_ERR_UNSUPPORTED;  // pages too large for a two-stage ring
  }
  plan->stages = stages;
  plan->warps_per_cta = wpc;
  plan->warp_smem = warp_smem;
  const void* k = decode_kernel_ptr<D, BLOCK, GPAD, PSPLIT>();
  plan->kernel = k;
  const int smem = wpc * (int)warp_smem;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return KVQ3_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 32 * wpc, smem) != cudaSuccess)
    return KVQ3_ERR_CUDA;
  if (per_sm < 1) return KVQ3_ERR_UNSUPPORTED;
  plan->ctas = sm_count() * per_sm;
  const size_t slots = (size_t)plan->ctas * wpc + (size_t)g.batch * g.hkv;
  plan->ws_bytes = slots * (size_t)G * (D + 2) * sizeof(float);
  return KVQ3_OK;
}

template <int D, int BLOCK, int GPAD, bool PSPLIT>
kvq3_status decode_run_t(const DecodePlan& plan, DecodeParams prm, const RotParams& rp, float* out,
                         cudaStream_t st) {
  prm.stages = plan.stages;
  prm.stage_bytes = plan.stage_bytes;
  prm.copy_bytes = plan.copy_bytes;
  prm.total_warps = plan.ctas * plan.warps_per_cta;
  prm.warps_per_cta = plan.warps_per_cta;
  prm.warp_smem = plan.warp_smem;
  decode_split_kernel<D, BLOCK, GPAD, PSPLIT><<<plan.ctas, 32 * plan.warps_per_cta,
                                        plan.warps_per_cta * plan.warp_smem, st>>>(prm, rp);
  if (cudaGetLastError() != cudaSuccess) return KVQ3_ERR_CUDA;
  const int64_t items = (int64_t)prm.g.batch * prm.Hq;
  int64_t blocks = (items + 7) / 8;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap > 0 ? cap : 1;
  decode_combine_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(prm, rp, out);
  return cudaGetLastError() == cudaSuccess ? KVQ3_OK : KVQ3_ERR_CUDA;
}

// Per-head-dim entry points (one translation unit each).
kvq3_status decode_plan_d64(const CacheGeom& g, int G, DecodePlan* plan);
kvq3_status decode_plan_d128(const CacheGeom& g, int G, DecodePlan* plan);
kvq3_status decode_plan_d256(const CacheGeom& g, int G, DecodePlan* plan);
kvq3_status decode_run_d64(const DecodePlan&, const DecodeParams&, const RotParams&, float*, cudaStream_t);
kvq3_status decode_run_d128(const DecodePlan&, const DecodeParams&, const RotParams&, float*, cudaStream_t);
kvq3_status decode_run_d256(const DecodePlan&, const DecodeParams&, const RotParams&, float*, cudaStream_t);

// Variant choice: P' split for G <= 4 (free) and for fp32 value scales.
#define KVQ3_DECODE_PICK(D, BLK, FN, ...)                                                      \
  {                                                                                           \
    const bool f32 = g.scale_type == KVQ3_SCALE_F32;                                          \
    if (gp == 4) return FN<D, BLK, 4, true>(__VA_ARGS__);                                     \
    if (gp == 8) return f32 ? FN<D, BLK, 8, true>(__VA_ARGS__) : FN<D, BLK, 8, false>(__VA_ARGS__); \
    return f32 ? FN<D, BLK, 16, true>(__VA_ARGS__) : FN<D, BLK, 16, false>(__VA_ARGS__);       \
  }

#define KVQ3_DECODE_INSTANCES(D)                                                              \
  kvq3_status decode_plan_d##D(const CacheGeom& g, int G, DecodePlan* plan) {                \
    const int gp = G <= 4 ? 4 : (G <= 8 ? 8 : 16);                                            \
    if (g.block == 32) KVQ3_DECODE_PICK(D, 32, decode_plan_t, g, G, plan)                     \
    KVQ3_DECODE_PICK(D, 64, decode_plan_t, g, G, plan)                                        \
  }                                                                                           \
  kvq3_status decode_run_d##D(const DecodePlan& plan, const DecodeParams& prm,                \
                              const RotParams& rp, float* out, cudaStream_t st) {             \
    const CacheGeom& g = prm.g;                                                               \
    const int gp = plan.gpad;                                                                 \
    if (g.block == 32) KVQ3_DECODE_PICK(D, 32, decode_run_t, plan, prm, rp, out, st)          \
    KVQ3_DECODE_PICK(D, 64, decode_run_t, plan, prm, rp, out, st)                             \
  }

}  // namespace kvq3
