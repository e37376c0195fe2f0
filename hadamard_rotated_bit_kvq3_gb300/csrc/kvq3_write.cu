// Write path of the rotated 3-bit KV cache and its debug read-back.
//
// "Orthogonally mixed 3-bit KV cache", Implementation notes: on every new
// token compute k1 = U(k), v1 = U(v), split into quantisation blocks, one
// scale per block, round to signed 3-bit integers, pack the codes into bytes,
// store only packed codes and scales.  Key formulas: s = (max|x| + eps)/3,
// x_hat = s * clip(round(x/s), -3, 3) -- for b-bit codes (b = 2, 3, 4;
// "Orthogonal Invariance in Activation Space", 3.3, 4.2, 5.1) the divisor and
// the clip bound are 2^(b-1) - 1.  "Orthogonal Invariance in Activation
// Space", 3.3 "Retrieve" for the read-back.
//
// One group of L = D/E lanes handles one (token, kv head, K|V) vector, E
// consecutive elements per lane: 128-bit-or-smaller coalesced fp16 loads,
// the sign flip, the Walsh-Hadamard butterfly (log2 E register stages, log2 L
// shuffle stages), 1/sqrt(d), the SO(4) 4x4 products in registers, the block
// maximum by an xor-shuffle reduction, the scale rounded to its storage type,
// the codes, and the 32-bit words of the code string assembled by shuffles
// and stored by the first NBIT*D/32 lanes of the group.
#include <string.h>

#include "kvq3_internal.h"

using namespace kvq3;

namespace {

template <int D, int E, int BLOCK, int NBIT>
__global__ void __launch_bounds__(256) write_kernel(
    const __grid_constant__ RotParams rp, const __grid_constant__ CacheGeom g,
    uint8_t* __restrict__ pool, const int32_t* __restrict__ page_table,
    const __half* __restrict__ kin, const __half* __restrict__ vin,
    const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ pos, int64_t n_tok,
    int32_t* __restrict__ status, float inv_sqrt_d) {
  constexpr int L = D / E;            // lanes per vector
  constexpr int GPW = 32 / L;         // vectors per warp
  constexpr int LPB = BLOCK / E;      // lanes per quantisation block
  constexpr int BITS = NBIT * E;      // code bits per lane
  constexpr int WORDS = NBIT * D / 32;  // 32-bit words of a code string
  constexpr int QMAX = (1 << (NBIT - 1)) - 1;
  static_assert(E <= BLOCK && BITS <= 32 && WORDS <= L, "lane layout");
  // a kernel launched after this one as a programmatic dependent (the decode)
  // may start now; it waits for this grid's writes before it reads anything
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int r = lane % L, grp = lane / L;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t sgn = lane_signs<E>(rp, r);
  float4 q[E / 4];
  float4 qr[E / 4];
  lane_quats<E>(rp, r, q);
  lane_quats_r<E>(rp, r, qr);
  const bool so4 = rot_so4(rp), pair = rot_pair(rp);
  const int64_t per_which = n_tok * g.hkv;
  const int64_t total = 2 * per_which;
  const int64_t cap = (int64_t)g.max_pages * g.page_size;

  for (int64_t base = warp * GPW; base < total; base += nwarps * GPW) {
    const int64_t item = base + grp;
    const bool in_range = item < total;
    int which = 0, head = 0;
    int64_t tok = 0;
    if (in_range) {   // item = (which, token, head); below 2^31 (n_tok * Hkv is checked on the host)
      which = item >= per_which;
      const uint32_t rem = (uint32_t)(item - which * per_which);
      tok = rem / (uint32_t)g.hkv;
      head = (int)(rem - (uint32_t)tok * (uint32_t)g.hkv);
    }
    // the vector's load and quantisation do not wait for the position and
    // page lookups: only the store does
    float x[E];
    if (in_range) {
      const __half* src = (which ? vin : kin) + (tok * g.hkv + head) * D + r * E;
      if constexpr (E == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(src);
        const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(h[i]);
          x[2 * i] = f.x;
          x[2 * i + 1] = f.y;
        }
      } else if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float2 f = __half22float2(h[i]);
          x[2 * i] = f.x;
          x[2 * i + 1] = f.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = __half2float(src[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) x[e] = 0.0f;
    }
    bool ok = in_range;
    int64_t rec = 0;
    int slot = 0;
    if (ok) {
      const int s = seq_idx[tok];
      const int64_t p = pos[tok];
      int bad = 0;
      int64_t page = -1;
      if (s < 0 || s >= g.batch) bad = KVQ3_DEV_BAD_SEQ;
      else if (p < 0 || p >= cap) bad = KVQ3_DEV_BAD_POS;
      else {   // 0 <= p < max_pages * page_size; p is an int32 position
        page = page_of(g, page_table, s, (int64_t)((uint32_t)p / (uint32_t)g.page_size));
        if (page < 0) bad = KVQ3_DEV_BAD_PAGE;
      }
      if (bad) {
        if (r == 0) set_status(status, bad);
        ok = false;
      } else {
        slot = (int)((uint32_t)p % (uint32_t)g.page_size);
        rec = record_offset(g, page, head, which);
      }
    }
    rotate_forward<E, L>(x, r, sgn, q, qr, inv_sqrt_d, so4, pair);

    // this lane's E elements lie in one block of LPB lanes
    uint32_t sbits, bits = 0;
    if (g.scale_type != KVQ3_SCALE_E4M3_ZP) {
      // block maximum -> symmetric scale, two's-complement codes
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
      for (int m = 1; m < LPB; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
      const float s = __fdiv_rn(amax + g.eps, (float)QMAX);
      const float sq = round_scale(s, g.scale_type, sbits);
      const float inv = sq > 0.0f ? __frcp_rn(sq) : 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float c = fminf(fmaxf(rintf(x[e] * inv), -(float)QMAX), (float)QMAX);
        bits |= ((uint32_t)(int)c & ((1u << NBIT) - 1u)) << (NBIT * e);
      }
    } else {
      // asymmetric variant: block minimum and maximum -> E4M3 scale
      // (max - min + eps)/(2^b - 1) and E4M3 zero point min, unsigned codes
      constexpr float UMAX = (float)((1 << NBIT) - 1);
      float mx = -INFINITY, mn = INFINITY;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        mx = fmaxf(mx, x[e]);
        mn = fminf(mn, x[e]);
      }
#pragma unroll
      for (int m = 1; m < LPB; m <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
        mn = fminf(mn, __shfl_xor_sync(kFull, mn, m));
      }
      uint32_t sb8, zb8;
      const float sq = round_scale(__fdiv_rn((mx - mn) + g.eps, UMAX), KVQ3_SCALE_E4M3, sb8);
      const float zq = round_scale(mn, KVQ3_SCALE_E4M3, zb8);
      sbits = sb8 | (zb8 << 8);       // scale byte, then zero-point byte
      const float inv = sq > 0.0f ? __frcp_rn(sq) : 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float u = fminf(fmaxf(rintf((x[e] - zq) * inv), 0.0f), UMAX);
        bits |= (uint32_t)u << (NBIT * e);
      }
    }
    // word w of the code string collects bits [32w, 32w+32) from the lanes
    // whose [BITS*r, BITS*r + BITS) ranges overlap it
    uint32_t word = 0;
    const int first = (32 * r) / BITS;
#pragma unroll
    for (int k = 0; k < 32 / BITS + 2; ++k) {
      int src = first + k;
      const bool in = src < L;
      src = in ? src : L - 1;
      const uint32_t v = __shfl_sync(kFull, bits, grp * L + src);
      const int sh = BITS * src - 32 * r;
      if (in && sh > -BITS && sh < 32) word |= sh >= 0 ? (v << sh) : (v >> (-sh));
    }
    if (ok && KVQ3_CHECK(status, ::kvq3::in_range(rec, g.record_bytes, g.num_pages * g.page_bytes) &&
                                     slot >= 0 && slot < g.page_size)) {
      uint8_t* base_p = pool + rec;
      if (r < WORDS)
        *reinterpret_cast<uint32_t*>(base_p + g.scale_hdr_bytes + (int64_t)slot * g.cb + 4 * r) = word;
      if (r % LPB == 0) {
        const int blk = r / LPB;
        uint8_t* sp = base_p + ((int64_t)slot * g.nb + blk) * g.sb;
        if (g.sb == 4) *reinterpret_cast<uint32_t*>(sp) = sbits;
        else if (g.sb == 2) *reinterpret_cast<uint16_t*>(sp) = (uint16_t)sbits;
        else *sp = (uint8_t)sbits;
      }
    }
  }
}

template <int D, int BLOCK, int NBIT>
cudaError_t launch_write_b(const RotParams& rp, const CacheGeom& g, const kvq3_cache* c,
                           const __half* k, const __half* v, const int32_t* si, const int32_t* pos,
                           int64_t n_tok, int32_t* st, cudaStream_t stream) {
  constexpr int E = D >= 128 ? D / 32 : 4;
  constexpr int GPW = 32 / (D / E);
  const int64_t items = 2 * n_tok * g.hkv;
  const int64_t warps = (items + GPW - 1) / GPW;
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap > 0 ? cap : 1;
  write_kernel<D, E, BLOCK, NBIT><<<(unsigned)blocks, 256, 0, stream>>>(
      rp, g, static_cast<uint8_t*>(c->pool), c->page_table, k, v, si, pos, n_tok, st,
      inv_sqrt(D));
  return cudaGetLastError();
}

template <int D, int BLOCK>
cudaError_t launch_write(const RotParams& rp, const CacheGeom& g, const kvq3_cache* c,
                         const __half* k, const __half* v, const int32_t* si, const int32_t* pos,
                         int64_t n_tok, int32_t* st, cudaStream_t stream) {
  if (g.bits == 2) return launch_write_b<D, BLOCK, 2>(rp, g, c, k, v, si, pos, n_tok, st, stream);
  if (g.bits == 4) return launch_write_b<D, BLOCK, 4>(rp, g, c, k, v, si, pos, n_tok, st, stream);
  return launch_write_b<D, BLOCK, 3>(rp, g, c, k, v, si, pos, n_tok, st, stream);
}

// ------------------------------------------------------------ read-back
template <int D>
__global__ void __launch_bounds__(256) dequant_kernel(
    const __grid_constant__ RotParams rp, int use_rot, const __grid_constant__ CacheGeom g,
    const uint8_t* __restrict__ pool, const int32_t* __restrict__ page_table, int seq, int kvh,
    int which, int64_t t0, int64_t nt, float* __restrict__ out, int32_t* __restrict__ codes_out,
    int32_t* __restrict__ status, float inv_sqrt_d) {
  constexpr int E = D >= 128 ? D / 32 : 4;
  constexpr int L = D / E;
  constexpr int GPW = 32 / L;
  const int lane = threadIdx.x & 31;
  const int r = lane % L, grp = lane / L;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t sgn = lane_signs<E>(rp, r);
  float4 q[E / 4];
  float4 qr[E / 4];
  lane_quats<E>(rp, r, q);
  lane_quats_r<E>(rp, r, qr);
  const bool so4 = rot_so4(rp), pair = rot_pair(rp);
  const int64_t cap = (int64_t)g.max_pages * g.page_size;
  for (int64_t base = warp * GPW; base < nt; base += nwarps * GPW) {
    const int64_t t = base + grp;
    bool ok = t < nt;
    int bad = 0;
    float x[E];
    int c[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = 0.0f;
      c[e] = 0;
    }
    if (ok) {
      const int64_t p = t0 + t;
      int64_t page = -1;
      if (seq < 0 || seq >= g.batch) bad = KVQ3_DEV_BAD_SEQ;
      else if (p < 0 || p >= cap) bad = KVQ3_DEV_BAD_POS;
      else if ((page = page_of(g, page_table, seq, p / g.page_size)) < 0) bad = KVQ3_DEV_BAD_PAGE;
      if (!bad && !KVQ3_CHECK(status, ::kvq3::in_range(record_offset(g, page, kvh, which), g.record_bytes,
                                               g.num_pages * g.page_bytes)))
        bad = KVQ3_DEV_CHECK;
      if (!bad) {
        const int slot = (int)(p % g.page_size);
        const uint8_t* rec = pool + record_offset(g, page, kvh, which);
        const uint8_t* codes = rec + g.scale_hdr_bytes + (int64_t)slot * g.cb;
        const int blk = (r * E) / g.block;
        const uint8_t* sp = rec + ((int64_t)slot * g.nb + blk) * g.sb;
        uint32_t sbits = 0;
        for (int i = 0; i < g.sb; ++i) sbits |= (uint32_t)sp[i] << (8 * i);
        const bool asym = g.scale_type == KVQ3_SCALE_E4M3_ZP;   // x_hat = s_q u + z_q
        const float sq = decode_scale(sbits & (asym ? 0xffu : ~0u), g.scale_type);
        const float zq = asym ? decode_scale(sbits >> 8, KVQ3_SCALE_E4M3) : 0.0f;
        const int nbit = g.bits, half = 1 << (nbit - 1);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int bit = nbit * (r * E + e);
          const uint32_t two = (uint32_t)codes[bit / 8] |
                               ((bit / 8 + 1 < g.cb) ? (uint32_t)codes[bit / 8 + 1] << 8 : 0u);
          const int f = (int)((two >> (bit % 8)) & ((1u << nbit) - 1u));
          if (asym) {
            c[e] = f;
            x[e] = fmaf(sq, (float)f, zq);
            continue;
          }
          int cv = f >= half ? f - 2 * half : f;
          if (cv == -half) {   // the value the quantiser never writes
            bad |= KVQ3_DEV_BAD_CODE;
            cv = 0;
          }
          c[e] = cv;
          x[e] = sq * (float)cv;
        }
      }
      if (bad) set_status(status, bad);
    }
    if (use_rot) rotate_inverse<E, L>(x, r, sgn, q, qr, inv_sqrt_d, so4, pair);
    if (ok) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        out[t * D + r * E + e] = (bad & ~KVQ3_DEV_BAD_CODE) ? 0.0f : x[e];
        if (codes_out) codes_out[t * D + r * E + e] = c[e];
      }
    }
  }
}

template <int D>
cudaError_t launch_dequant(const RotParams& rp, int use_rot, const CacheGeom& g,
                           const kvq3_cache* c, int seq, int kvh, int which, int64_t t0,
                           int64_t nt, float* out, int32_t* codes, int32_t* st,
                           cudaStream_t stream) {
  constexpr int E = D >= 128 ? D / 32 : 4;
  constexpr int GPW = 32 / (D / E);
  const int64_t warps = (nt + GPW - 1) / GPW;
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap > 0 ? cap : 1;
  dequant_kernel<D><<<(unsigned)blocks, 256, 0, stream>>>(
      rp, use_rot, g, static_cast<const uint8_t*>(c->pool), c->page_table, seq, kvh, which, t0,
      nt, out, codes, st, inv_sqrt(D));
  return cudaGetLastError();
}

}  // namespace

extern "C" {

kvq3_status kvq3_write(kvq3_rotation rot, const kvq3_cache_desc* desc, const kvq3_cache* cache,
                       const void* k, const void* v, const int32_t* seq_idx, const int32_t* pos,
                       int64_t n_tok, int32_t* dev_status, void* stream) {
  CacheGeom g;
  kvq3_status s = make_geom(desc, &g);
  if (s != KVQ3_OK) return s;
  if (!rot || rot->d != g.d || n_tok < 0) return KVQ3_ERR_INVALID_ARG;
  if ((s = check_cache(g, cache, false)) != KVQ3_OK) return s;
  if (n_tok == 0) return KVQ3_OK;
  if (n_tok >= ((int64_t)1 << 31) / (2 * g.hkv)) return KVQ3_ERR_UNSUPPORTED;  // 32-bit item index
  if (!k || !v || !seq_idx || !pos) return KVQ3_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16 != 0)
    return KVQ3_ERR_INVALID_ARG;
  const __half* kh = static_cast<const __half*>(k);
  const __half* vh = static_cast<const __half*>(v);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const int key = g.d * 1000 + g.block;
  switch (key) {
    case 64032: e = launch_write<64, 32>(rot->params, g, cache, kh, vh, seq_idx, pos, n_tok, dev_status, st); break;
    case 64064: e = launch_write<64, 64>(rot->params, g, cache, kh, vh, seq_idx, pos, n_tok, dev_status, st); break;
    case 128032: e = launch_write<128, 32>(rot->params, g, cache, kh, vh, seq_idx, pos, n_tok, dev_status, st); break;
    case 128064: e = launch_write<128, 64>(rot->params, g, cache, kh, vh, seq_idx, pos, n_tok, dev_status, st); break;
    case 256032: e = launch_write<256, 32>(rot->params, g, cache, kh, vh, seq_idx, pos, n_tok, dev_status, st); break;
    case 256064: e = launch_write<256, 64>(rot->params, g, cache, kh, vh, seq_idx, pos, n_tok, dev_status, st); break;
    default: return KVQ3_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}

kvq3_status kvq3_dequant_debug(kvq3_rotation rot, const kvq3_cache_desc* desc,
                               const kvq3_cache* cache, int32_t seq, int32_t kv_head,
                               int32_t which, int64_t t0, int64_t nt, float* out,
                               int32_t* codes_out, int32_t* dev_status, void* stream) {
  CacheGeom g;
  kvq3_status s = make_geom(desc, &g);
  if (s != KVQ3_OK) return s;
  if ((s = check_cache(g, cache, false)) != KVQ3_OK) return s;
  if (nt < 0 || kv_head < 0 || kv_head >= g.hkv || (which != 0 && which != 1))
    return KVQ3_ERR_INVALID_ARG;
  if (rot && rot->d != g.d) return KVQ3_ERR_INVALID_ARG;
  if (nt == 0) return KVQ3_OK;
  if (!out) return KVQ3_ERR_INVALID_ARG;
  RotParams rp;
  memset(&rp, 0, sizeof(rp));
  if (rot) rp = rot->params;
  const int use_rot = rot ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (g.d) {
    case 64: e = launch_dequant<64>(rp, use_rot, g, cache, seq, kv_head, which, t0, nt, out, codes_out, dev_status, st); break;
    case 128: e = launch_dequant<128>(rp, use_rot, g, cache, seq, kv_head, which, t0, nt, out, codes_out, dev_status, st); break;
    case 256: e = launch_dequant<256>(rp, use_rot, g, cache, seq, kv_head, which, t0, nt, out, codes_out, dev_status, st); break;
    default: return KVQ3_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}

}  // extern "C"
