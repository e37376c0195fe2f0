// Device helpers shared by the kernels of the rotated 3-bit KV cache.
//
// Sources: "Orthogonally mixed 3-bit KV cache" (Mathematical statement, Key
// formulas, Implementation notes) and "Orthogonal Invariance in Activation
// Space" (sections 3.1-3.4, 4.2); the readings R1-R15 and the cache layout
// are those written in include/kvq3.h.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/kvq3.h"

namespace kvq3 {

constexpr int kMaxD = 256;
constexpr unsigned kFull = 0xffffffffu;

// Rotation parameters as kernels receive them (by value, ~2 KB of kernel
// parameter space): sign bit j set <=> sigma_j = -1; block i acts on rotated
// coordinates 4i..4i+3 as x -> p_i x (reading R3), or as x -> p_i x conj(q_i)
// with KVQ3_ROT_SO4_PAIR (reading R20; q_i = 1 otherwise).
struct RotParams {
  uint32_t sign_bits[kMaxD / 32];
  float4 quat[kMaxD / 4];     // p_i
  float4 quat_r[kMaxD / 4];   // q_i
  int32_t d;
  uint32_t flags;
};

// Cache geometry derived on the host from kvq3_cache_desc.
struct CacheGeom {
  int32_t d, hkv, block, nb, sb, cb, page_size, batch, max_pages;
  int32_t bits;             // code width b: 2, 3 or 4
  int32_t scale_type;
  float eps;
  int64_t num_pages;
  int64_t record_bytes, page_bytes;
  int64_t scale_hdr_bytes;  // P*nb*sb: offset of the code strings in a record
};

// ---------------------------------------------------------------- FWHT
// Normalised Walsh-Hadamard transform (reading R1) of a vector spread over a
// group of L consecutive lanes, E consecutive elements per lane: element
// index i = r*E + e (r = lane in group, e = register).  log2(E) butterfly
// stages inside the registers, then log2(L) stages across lanes by xor
// shuffles.  Unnormalised here: the caller multiplies by 1/sqrt(d).
// Every lane of the warp must call it (full-warp shuffles).
template <int E, int L>
__device__ __forceinline__ void fwht_group(float (&x)[E], int r) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < L; m <<= 1) {
    const bool upper = (r & m) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float o = __shfl_xor_sync(kFull, x[i], m);
      x[i] = upper ? (o - x[i]) : (x[i] + o);
    }
  }
}

// y = L(p) x: the quaternion product p * x (reading R3).
__device__ __forceinline__ void quat_apply(const float4 p, float& x0, float& x1, float& x2,
                                           float& x3) {
  const float y0 = p.x * x0 - p.y * x1 - p.z * x2 - p.w * x3;
  const float y1 = p.y * x0 + p.x * x1 - p.w * x2 + p.z * x3;
  const float y2 = p.z * x0 + p.w * x1 + p.x * x2 - p.y * x3;
  const float y3 = p.w * x0 - p.z * x1 + p.y * x2 + p.x * x3;
  x0 = y0; x1 = y1; x2 = y2; x3 = y3;
}

// y = L(p)^T x = L(conj p) x (inverse of a unit quaternion block).
__device__ __forceinline__ void quat_apply_t(const float4 p, float& x0, float& x1, float& x2,
                                             float& x3) {
  quat_apply(make_float4(p.x, -p.y, -p.z, -p.w), x0, x1, x2, x3);
}

// y = x * q: the quaternion product with q on the right (reading R20).
__device__ __forceinline__ void quat_apply_right(const float4 q, float& x0, float& x1, float& x2,
                                                 float& x3) {
  const float y0 = x0 * q.x - x1 * q.y - x2 * q.z - x3 * q.w;
  const float y1 = x0 * q.y + x1 * q.x + x2 * q.w - x3 * q.z;
  const float y2 = x0 * q.z - x1 * q.w + x2 * q.x + x3 * q.y;
  const float y3 = x0 * q.w + x1 * q.z - x2 * q.y + x3 * q.x;
  x0 = y0; x1 = y1; x2 = y2; x3 = y3;
}

// y = x * conj(q) (the right half of a two-quaternion block; its inverse is
// quat_apply_right with q).
__device__ __forceinline__ void quat_apply_right_conj(const float4 q, float& x0, float& x1,
                                                      float& x2, float& x3) {
  quat_apply_right(make_float4(q.x, -q.y, -q.z, -q.w), x0, x1, x2, x3);
}

// Forward U = B H D on the E elements this lane holds (dims r*E .. r*E+E-1).
// sgn: E sign bits of this lane; q, qr: the E/4 left and right quaternions of
// this lane; pair: two-quaternion blocks (reading R20).
template <int E, int L>
__device__ __forceinline__ void rotate_forward(float (&x)[E], int r, uint32_t sgn,
                                               const float4 (&q)[E / 4], const float4 (&qr)[E / 4],
                                               float inv_sqrt_d, bool so4, bool pair) {
#pragma unroll
  for (int e = 0; e < E; ++e)
    if ((sgn >> e) & 1u) x[e] = -x[e];
  fwht_group<E, L>(x, r);
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] *= inv_sqrt_d;
  if (so4) {
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      quat_apply(q[i], x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
      if (pair) quat_apply_right_conj(qr[i], x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    }
  }
}

// Inverse U^T = D H B^T.
template <int E, int L>
__device__ __forceinline__ void rotate_inverse(float (&x)[E], int r, uint32_t sgn,
                                               const float4 (&q)[E / 4], const float4 (&qr)[E / 4],
                                               float inv_sqrt_d, bool so4, bool pair) {
  if (so4) {
#pragma unroll
    for (int i = 0; i < E / 4; ++i) {
      if (pair) quat_apply_right(qr[i], x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
      quat_apply_t(q[i], x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    }
  }
  fwht_group<E, L>(x, r);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    x[e] *= inv_sqrt_d;
    if ((sgn >> e) & 1u) x[e] = -x[e];
  }
}

// This lane's E sign bits and E/4 quaternions (dims r*E ..).
template <int E>
__device__ __forceinline__ uint32_t lane_signs(const RotParams& rp, int r) {
  const int j0 = r * E;
  if (E >= 32) return rp.sign_bits[j0 / 32];  // E == 32 only (not used above 32)
  return (rp.sign_bits[j0 / 32] >> (j0 % 32)) & ((1u << E) - 1u);
}

template <int E>
__device__ __forceinline__ void lane_quats(const RotParams& rp, int r, float4 (&q)[E / 4]) {
#pragma unroll
  for (int i = 0; i < E / 4; ++i) q[i] = rp.quat[r * (E / 4) + i];
}

template <int E>
__device__ __forceinline__ void lane_quats_r(const RotParams& rp, int r, float4 (&q)[E / 4]) {
#pragma unroll
  for (int i = 0; i < E / 4; ++i) q[i] = rp.quat_r[r * (E / 4) + i];
}

// Flags of a rotation as the kernels test them.
__device__ __forceinline__ bool rot_so4(const RotParams& rp) { return (rp.flags & KVQ3_ROT_SO4) != 0; }
__device__ __forceinline__ bool rot_pair(const RotParams& rp) {
  return (rp.flags & (KVQ3_ROT_SO4 | KVQ3_ROT_SO4_PAIR)) == (KVQ3_ROT_SO4 | KVQ3_ROT_SO4_PAIR);
}

// ---------------------------------------------------------------- scales
// Round an fp32 scale to its storage type (reading R7; round to nearest even,
// fp16 and E4M3 saturating) and return (stored value as fp32, raw bits).
__device__ __forceinline__ float round_scale(float s, int scale_type, uint32_t& bits) {
  if (scale_type == KVQ3_SCALE_F32) {
    bits = __float_as_uint(s);
    return s;
  }
  if (scale_type == KVQ3_SCALE_F16) {
    const __half h = __float2half_rn(fminf(s, 65504.0f));
    bits = __half_as_ushort(h);
    return __half2float(h);
  }
  const __nv_fp8_storage_t b = __nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
  bits = b;
  const __half_raw hr = __nv_cvt_fp8_to_halfraw(b, __NV_E4M3);
  return __half2float(__half(hr));
}

// Decode a stored scale (raw little-endian bits of width sb) to fp32.
__device__ __forceinline__ float decode_scale(uint32_t bits, int scale_type) {
  if (scale_type == KVQ3_SCALE_F32) return __uint_as_float(bits);
  if (scale_type == KVQ3_SCALE_F16) return __half2float(__ushort_as_half((unsigned short)bits));
  const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(bits & 0xff), __NV_E4M3);
  return __half2float(__half(hr));
}

// ---------------------------------------------------------------- addressing
// Physical page of (b, logical page lp); -1 when the page id is out of range.
__device__ __forceinline__ int64_t page_of(const CacheGeom& g, const int32_t* page_table, int b,
                                           int64_t lp) {
  int64_t pg;
  if (page_table) pg = page_table[(int64_t)b * g.max_pages + lp];
  else pg = (int64_t)b * g.max_pages + lp;
  return (pg >= 0 && pg < g.num_pages) ? pg : -1;
}

__device__ __forceinline__ int64_t record_offset(const CacheGeom& g, int64_t page, int kvh,
                                                 int which) {
  return page * g.page_bytes + (int64_t)(kvh * 2 + which) * g.record_bytes;
}

__device__ __forceinline__ void set_status(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

// Bounds checks of a checked build (compiled with -DKVQ3_CHECKED): a check
// that fails sets KVQ3_DEV_CHECK in the status word and its caller skips the
// access.  In the normal build every check is the constant true.
#ifdef KVQ3_CHECKED
__device__ __forceinline__ bool checked(int32_t* st, bool ok) {
  if (!ok) set_status(st, KVQ3_DEV_CHECK);
  return ok;
}
#define KVQ3_CHECK(st, cond) ::kvq3::checked((st), (cond))
#else
#define KVQ3_CHECK(st, cond) true
#endif

// [base, base + n) lies inside [0, size)
__device__ __forceinline__ bool in_range(int64_t base, int64_t n, int64_t size) {
  return base >= 0 && n >= 0 && base <= size - n;
}

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bounded wait for phase `parity` of an mbarrier.  Returns false when the
// bound ran out (the caller flags KVQ3_DEV_TIMEOUT and winds down).
// Programmatic dependent launch (griddepcontrol): a grid launched with
// programmatic stream serialisation may start before the preceding grid ends;
// griddep_wait blocks until that grid has completed and its writes are
// visible, griddep_launch_dependents lets the following grid start.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t it = 0; it < max_iter; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Packed pairs of fp32 (sm_100 family f32x2 arithmetic): one instruction for two lanes' worth.
typedef unsigned long long u64;
__device__ __forceinline__ float2 f2add(float2 a, float2 b) {
  u64 d, x = *reinterpret_cast<u64*>(&a), y = *reinterpret_cast<u64*>(&b);
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 f2sub(float2 a, float2 b) {
  u64 d, x = *reinterpret_cast<u64*>(&a), y = *reinterpret_cast<u64*>(&b);
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) {
  u64 d, x = *reinterpret_cast<u64*>(&a), y = *reinterpret_cast<u64*>(&b);
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) {
  u64 d, x = *reinterpret_cast<u64*>(&a), y = *reinterpret_cast<u64*>(&b),
         z = *reinterpret_cast<u64*>(&c);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(y), "l"(z));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace kvq3
