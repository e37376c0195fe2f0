// Host side of the C ABI: rotation handles, validation, sizes, status
// strings, and the standalone rotation kernel (kvq3_rotate).
//
// The seed -> parameter derivation follows reading R4 of include/kvq3.h
// (SplitMix64, then Marsaglia's 1972 point on S^3).  This translation unit
// is compiled with -ffp-contract=off so the fp64 steps are the plain IEEE
// operations, bit-reproducible on every host.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "kvq3_internal.h"

using namespace kvq3;

namespace {

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014).
struct SplitMix64 {
  uint64_t state;
  uint64_t next() {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform_pm1() { return (double)(next() >> 11) * 0x1.0p-53 * 2.0 - 1.0; }
};

// Marsaglia (1972): uniform point on S^3 from two points in the unit disk.
void marsaglia_s3(SplitMix64& rng, double out[4]) {
  double x1, x2, s1, x3, x4, s2;
  for (;;) {
    x1 = rng.uniform_pm1();
    x2 = rng.uniform_pm1();
    s1 = x1 * x1 + x2 * x2;
    if (s1 > 0.0 && s1 < 1.0) break;
  }
  for (;;) {
    x3 = rng.uniform_pm1();
    x4 = rng.uniform_pm1();
    s2 = x3 * x3 + x4 * x4;
    if (s2 > 0.0 && s2 < 1.0) break;
  }
  const double f = sqrt((1.0 - s1) / s2);
  out[0] = x1;
  out[1] = x2;
  out[2] = x3 * f;
  out[3] = x4 * f;
}

bool pow2_in(int d, int lo, int hi) { return d >= lo && d <= hi && (d & (d - 1)) == 0; }

void fill_params(kvq3_rotation_s* r) {
  RotParams& p = r->params;
  memset(&p, 0, sizeof(p));
  p.d = r->d;
  p.flags = r->flags;
  for (int j = 0; j < r->d; ++j)
    if (r->signs[j] < 0) p.sign_bits[j / 32] |= 1u << (j % 32);
  for (int i = 0; i < r->d / 4; ++i) {
    p.quat[i] = make_float4((float)r->quats64[4 * i], (float)r->quats64[4 * i + 1],
                            (float)r->quats64[4 * i + 2], (float)r->quats64[4 * i + 3]);
    p.quat_r[i] = make_float4((float)r->quats_r64[4 * i], (float)r->quats_r64[4 * i + 1],
                              (float)r->quats_r64[4 * i + 2], (float)r->quats_r64[4 * i + 3]);
  }
}

// Normalises n quaternions into out (fp64); false for a zero or non-finite one.
bool normalise_quats(const float* q, int n, double* out) {
  for (int i = 0; i < n; ++i) {
    double n2 = 0.0;
    for (int c = 0; c < 4; ++c) n2 += (double)q[4 * i + c] * (double)q[4 * i + c];
    if (!(n2 > 0.0) || !isfinite(n2)) return false;
    const double inv = 1.0 / sqrt(n2);
    for (int c = 0; c < 4; ++c) out[4 * i + c] = (double)q[4 * i + c] * inv;
  }
  return true;
}

}  // namespace

namespace kvq3 {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

kvq3_status make_geom(const kvq3_cache_desc* desc, CacheGeom* g) {
  if (!desc || !g) return KVQ3_ERR_INVALID_ARG;
  const int d = desc->head_dim;
  if (!pow2_in(d, 4, kMaxD) || desc->num_kv_heads < 1 || desc->batch < 1 ||
      desc->max_pages_per_seq < 1 || desc->num_pages < 1 || desc->page_size < 16 ||
      desc->page_size % 16 != 0 || desc->page_size > 4096 || desc->reserved != 0 ||
      !(desc->eps >= 0.0f) || !isfinite(desc->eps) || desc->block < 1 || d % desc->block != 0 ||
      desc->scale_type < KVQ3_SCALE_F32 || desc->scale_type > KVQ3_SCALE_E4M3_ZP)
    return KVQ3_ERR_INVALID_ARG;
  if (desc->bits < 2 || desc->bits > 4) return KVQ3_ERR_UNSUPPORTED;
  if (desc->scale_type == KVQ3_SCALE_E4M3_ZP && desc->bits != 3) return KVQ3_ERR_UNSUPPORTED;
  if (d < 64 || (desc->block != 32 && desc->block != 64)) return KVQ3_ERR_UNSUPPORTED;
  g->d = d;
  g->hkv = desc->num_kv_heads;
  g->block = desc->block;
  g->nb = d / desc->block;
  // bytes per block of the scale header: the asymmetric variant stores
  // (scale, zero point) as two E4M3 bytes
  g->sb = desc->scale_type == KVQ3_SCALE_F32 ? 4
        : desc->scale_type == KVQ3_SCALE_F16 || desc->scale_type == KVQ3_SCALE_E4M3_ZP ? 2 : 1;
  g->bits = desc->bits;
  g->cb = desc->bits * d / 8;
  g->page_size = desc->page_size;
  g->batch = desc->batch;
  g->max_pages = desc->max_pages_per_seq;
  g->scale_type = desc->scale_type;
  g->eps = desc->eps;
  g->num_pages = desc->num_pages;
  g->scale_hdr_bytes = (int64_t)g->page_size * g->nb * g->sb;
  g->record_bytes = (int64_t)g->page_size * (g->nb * g->sb + g->cb);
  g->page_bytes = (int64_t)g->hkv * 2 * g->record_bytes;
  if (g->num_pages > ((int64_t)1 << 62) / g->page_bytes) return KVQ3_ERR_INVALID_ARG;
  return KVQ3_OK;
}

kvq3_status check_cache(const CacheGeom& g, const kvq3_cache* cache, bool need_lens) {
  if (!cache || !cache->pool) return KVQ3_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cache->pool) % 16 != 0) return KVQ3_ERR_INVALID_ARG;
  if (need_lens && !cache->seq_lens) return KVQ3_ERR_INVALID_ARG;
  if (!cache->page_table && g.num_pages < (int64_t)g.batch * g.max_pages)
    return KVQ3_ERR_INVALID_ARG;  // a contiguous cache needs batch*max_pages pages
  return KVQ3_OK;
}

}  // namespace kvq3

// ------------------------------------------------------------------ kernels
namespace {

// y = U x or U^T x, one group of L = D/E lanes per vector (E = max(4, D/32)).
template <int D>
__global__ void __launch_bounds__(256) rotate_kernel(const __grid_constant__ RotParams rp,
                                                     const void* __restrict__ x, int x_fp16,
                                                     float* __restrict__ y, int64_t n,
                                                     int inverse, float inv_sqrt_d) {
  constexpr int E = D >= 128 ? D / 32 : 4;
  constexpr int L = D / E;
  constexpr int GPW = 32 / L;
  const int lane = threadIdx.x & 31;
  const int r = lane % L, grp = lane / L;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t sgn = lane_signs<E>(rp, r);
  float4 q[E / 4], qr[E / 4];
  lane_quats<E>(rp, r, q);
  lane_quats_r<E>(rp, r, qr);
  const bool so4 = rot_so4(rp), pair = rot_pair(rp);
  for (int64_t base = warp * GPW; base < n; base += nwarps * GPW) {
    const int64_t vi = base + grp;
    const bool ok = vi < n;
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float t = 0.0f;
      if (ok) {
        const int64_t idx = vi * D + r * E + e;
        t = x_fp16 ? __half2float(static_cast<const __half*>(x)[idx])
                   : static_cast<const float*>(x)[idx];
      }
      v[e] = t;
    }
    if (inverse) rotate_inverse<E, L>(v, r, sgn, q, qr, inv_sqrt_d, so4, pair);
    else rotate_forward<E, L>(v, r, sgn, q, qr, inv_sqrt_d, so4, pair);
    if (ok) {
#pragma unroll
      for (int e = 0; e < E; ++e) y[vi * D + r * E + e] = v[e];
    }
  }
}

template <int D>
cudaError_t launch_rotate(const RotParams& rp, const void* x, int x_fp16, float* y, int64_t n,
                          int inverse, cudaStream_t st) {
  constexpr int E = D >= 128 ? D / 32 : 4;
  constexpr int GPW = 32 / (D / E);
  const int64_t warps = (n + GPW - 1) / GPW;
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = (int64_t)kvq3::sm_count() * 16;
  if (blocks > cap) blocks = cap > 0 ? cap : 1;
  rotate_kernel<D><<<(unsigned)blocks, 256, 0, st>>>(rp, x, x_fp16, y, n, inverse,
                                                      kvq3::inv_sqrt(D));
  return cudaGetLastError();
}

}  // namespace

// ------------------------------------------------------------------ C ABI
extern "C" {

int32_t kvq3_abi_version(void) { return KVQ3_ABI_VERSION; }

const char* kvq3_status_string(kvq3_status s) {
  switch (s) {
    case KVQ3_OK: return "ok";
    case KVQ3_ERR_INVALID_ARG: return "invalid argument";
    case KVQ3_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ3_ERR_CUDA: return "CUDA error";
    case KVQ3_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

kvq3_status kvq3_rotation_create(int32_t d, uint64_t seed, uint32_t flags, kvq3_rotation* out) {
  if (!out || !pow2_in(d, 4, kMaxD) ||
      (flags & ~(uint32_t)(KVQ3_ROT_SIGN | KVQ3_ROT_SO4 | KVQ3_ROT_SO4_PAIR)))
    return KVQ3_ERR_INVALID_ARG;
  if ((flags & KVQ3_ROT_SO4_PAIR) && !(flags & KVQ3_ROT_SO4)) return KVQ3_ERR_INVALID_ARG;
  kvq3_rotation_s* r = static_cast<kvq3_rotation_s*>(calloc(1, sizeof(kvq3_rotation_s)));
  if (!r) return KVQ3_ERR_INVALID_ARG;
  r->d = d;
  r->flags = flags;
  SplitMix64 rng{seed};
  for (int j = 0; j < d; ++j) {
    const bool neg = (rng.next() >> 63) != 0;
    r->signs[j] = (flags & KVQ3_ROT_SIGN) && neg ? -1 : 1;
  }
  for (int i = 0; i < d / 4; ++i) {
    double p[4];
    marsaglia_s3(rng, p);
    for (int c = 0; c < 4; ++c)
      r->quats64[4 * i + c] = (flags & KVQ3_ROT_SO4) ? p[c] : (c == 0 ? 1.0 : 0.0);
  }
  // reading R20: the right quaternions are drawn after every left one
  for (int i = 0; i < d / 4; ++i) {
    double q[4] = {1.0, 0.0, 0.0, 0.0};
    if (flags & KVQ3_ROT_SO4_PAIR) marsaglia_s3(rng, q);
    for (int c = 0; c < 4; ++c) r->quats_r64[4 * i + c] = q[c];
  }
  fill_params(r);
  *out = r;
  return KVQ3_OK;
}

kvq3_status kvq3_rotation_create_from_params(int32_t d, const int8_t* signs, const float* quats,
                                             kvq3_rotation* out) {
  if (!out || !signs || !quats || !pow2_in(d, 4, kMaxD)) return KVQ3_ERR_INVALID_ARG;
  for (int j = 0; j < d; ++j)
    if (signs[j] != 1 && signs[j] != -1) return KVQ3_ERR_INVALID_ARG;
  kvq3_rotation_s* r = static_cast<kvq3_rotation_s*>(calloc(1, sizeof(kvq3_rotation_s)));
  if (!r) return KVQ3_ERR_INVALID_ARG;
  r->d = d;
  r->flags = KVQ3_ROT_SIGN | KVQ3_ROT_SO4;
  for (int j = 0; j < d; ++j) r->signs[j] = signs[j];
  if (!normalise_quats(quats, d / 4, r->quats64)) {
    free(r);
    return KVQ3_ERR_INVALID_ARG;
  }
  for (int i = 0; i < d / 4; ++i) r->quats_r64[4 * i] = 1.0;
  fill_params(r);
  *out = r;
  return KVQ3_OK;
}

kvq3_status kvq3_rotation_create_from_params_pair(int32_t d, const int8_t* signs, const float* quats,
                                                  const float* quats_r, kvq3_rotation* out) {
  if (!out || !signs || !quats || !quats_r || !pow2_in(d, 4, kMaxD)) return KVQ3_ERR_INVALID_ARG;
  for (int j = 0; j < d; ++j)
    if (signs[j] != 1 && signs[j] != -1) return KVQ3_ERR_INVALID_ARG;
  kvq3_rotation_s* r = static_cast<kvq3_rotation_s*>(calloc(1, sizeof(kvq3_rotation_s)));
  if (!r) return KVQ3_ERR_INVALID_ARG;
  r->d = d;
  r->flags = KVQ3_ROT_SIGN | KVQ3_ROT_SO4 | KVQ3_ROT_SO4_PAIR;
  for (int j = 0; j < d; ++j) r->signs[j] = signs[j];
  if (!normalise_quats(quats, d / 4, r->quats64) || !normalise_quats(quats_r, d / 4, r->quats_r64)) {
    free(r);
    return KVQ3_ERR_INVALID_ARG;
  }
  fill_params(r);
  *out = r;
  return KVQ3_OK;
}

kvq3_status kvq3_rotation_destroy(kvq3_rotation rot) {
  free(rot);
  return KVQ3_OK;
}

kvq3_status kvq3_rotation_export(kvq3_rotation rot, int8_t* signs, float* quats, int32_t* d_out) {
  if (!rot) return KVQ3_ERR_INVALID_ARG;
  if (d_out) *d_out = rot->d;
  if (signs)
    for (int j = 0; j < rot->d; ++j) signs[j] = (rot->params.sign_bits[j / 32] >> (j % 32)) & 1u ? -1 : 1;
  if (quats)
    for (int i = 0; i < rot->d / 4; ++i) {
      quats[4 * i] = rot->params.quat[i].x;
      quats[4 * i + 1] = rot->params.quat[i].y;
      quats[4 * i + 2] = rot->params.quat[i].z;
      quats[4 * i + 3] = rot->params.quat[i].w;
    }
  return KVQ3_OK;
}

kvq3_status kvq3_rotation_export_pair(kvq3_rotation rot, int8_t* signs, float* quats, float* quats_r,
                                      int32_t* d_out) {
  const kvq3_status s = kvq3_rotation_export(rot, signs, quats, d_out);
  if (s != KVQ3_OK) return s;
  if (quats_r)
    for (int i = 0; i < rot->d / 4; ++i) {
      quats_r[4 * i] = rot->params.quat_r[i].x;
      quats_r[4 * i + 1] = rot->params.quat_r[i].y;
      quats_r[4 * i + 2] = rot->params.quat_r[i].z;
      quats_r[4 * i + 3] = rot->params.quat_r[i].w;
    }
  return KVQ3_OK;
}

kvq3_status kvq3_cache_sizes(const kvq3_cache_desc* desc, size_t* record_bytes, size_t* page_bytes,
                             size_t* pool_bytes) {
  CacheGeom g;
  const kvq3_status s = make_geom(desc, &g);
  if (s != KVQ3_OK) return s;
  if (record_bytes) *record_bytes = (size_t)g.record_bytes;
  if (page_bytes) *page_bytes = (size_t)g.page_bytes;
  if (pool_bytes) *pool_bytes = (size_t)(g.page_bytes * g.num_pages);
  return KVQ3_OK;
}

kvq3_status kvq3_rotate(kvq3_rotation rot, const void* x, int32_t x_is_fp16, float* y,
                        int64_t n_vec, int32_t inverse, void* stream) {
  if (!rot || n_vec < 0 || (n_vec > 0 && (!x || !y))) return KVQ3_ERR_INVALID_ARG;
  if (n_vec == 0) return KVQ3_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int fp16 = x_is_fp16 ? 1 : 0;
  const int inv = inverse ? 1 : 0;
  cudaError_t e;
  switch (rot->d) {
    case 4: e = launch_rotate<4>(rot->params, x, fp16, y, n_vec, inv, st); break;
    case 8: e = launch_rotate<8>(rot->params, x, fp16, y, n_vec, inv, st); break;
    case 16: e = launch_rotate<16>(rot->params, x, fp16, y, n_vec, inv, st); break;
    case 32: e = launch_rotate<32>(rot->params, x, fp16, y, n_vec, inv, st); break;
    case 64: e = launch_rotate<64>(rot->params, x, fp16, y, n_vec, inv, st); break;
    case 128: e = launch_rotate<128>(rot->params, x, fp16, y, n_vec, inv, st); break;
    case 256: e = launch_rotate<256>(rot->params, x, fp16, y, n_vec, inv, st); break;
    default: return KVQ3_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}

}  // extern "C"
