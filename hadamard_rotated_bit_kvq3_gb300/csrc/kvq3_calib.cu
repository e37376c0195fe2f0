// SO(4) calibration: choose the quaternions of B that minimise the
// reconstruction error of the quantised rotated vectors on a sample.
//
// "Orthogonally mixed 3-bit KV cache", Implementation notes: start from fixed
// random rotations and calibrate them on representative sequences by
// minimising the reconstruction MSE after quantisation, each SO(4) block a
// normalised quaternion.  The search itself is not given by the page; this
// library's reading (include/kvq3.h, kvq3_calibrate_so4):
//  * objective: sum over the sample and the rotated coordinates of
//    (y - y_hat)^2, y = U x and y_hat its quantised value (the same rounding
//    as the write path); since U is orthogonal this equals the error of
//    U^T y_hat against x;
//  * it separates over quantisation blocks: block j of y depends only on
//    H D x and the m/4 quaternions of the SO(4) blocks inside it;
//  * random local search: each round evaluates the current quaternions and
//    P - 1 perturbed copies (every quaternion moved by a uniform step of
//    size sigma in R^4 and renormalised) in one launch, and every
//    quantisation block keeps the candidate with the lowest error; sigma
//    falls linearly over the rounds.
//
// calib_sse_kernel evaluates the objective per (candidate, quantisation
// block): one group of L = D/E lanes per sample vector, as in the write path.
#include <math.h>
#include <string.h>

#include <vector>

#include "kvq3_internal.h"

using namespace kvq3;

namespace {

// quats_r (nullable): candidate right quaternions of two-quaternion blocks
// (reading R20); without them every block is the left multiplication L(p).
template <int D, int E, int BLOCK, int NBIT, bool ASYM>
__global__ void __launch_bounds__(256) calib_sse_kernel(const __grid_constant__ RotParams rp,
                                                        const float4* __restrict__ quats,
                                                        const float4* __restrict__ quats_r,
                                                        const __half* __restrict__ x, int64_t n,
                                                        int scale_type, float eps,
                                                        double* __restrict__ sse, float inv_sqrt_d) {
  constexpr int L = D / E;
  constexpr int GPW = 32 / L;
  constexpr int LPB = BLOCK / E;
  constexpr int NBQ = D / BLOCK;
  constexpr float QMAX = (float)((1 << (NBIT - 1)) - 1);
  constexpr float UMAX = (float)((1 << NBIT) - 1);
  __shared__ float part[NBQ];
  if (threadIdx.x < NBQ) part[threadIdx.x] = 0.0f;
  __syncthreads();
  const int cand = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int r = lane % L, grp = lane / L;
  const uint32_t sgn = lane_signs<E>(rp, r);
  float4 q[E / 4], qr[E / 4];
  const bool pair = quats_r != nullptr;
#pragma unroll
  for (int i = 0; i < E / 4; ++i) {
    q[i] = quats[(size_t)cand * (D / 4) + r * (E / 4) + i];
    qr[i] = pair ? quats_r[(size_t)cand * (D / 4) + r * (E / 4) + i] : make_float4(1.0f, 0.0f, 0.0f, 0.0f);
  }
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float err = 0.0f;
  for (int64_t base = warp * GPW; base < n; base += nwarps * GPW) {
    const int64_t v = base + grp;
    float xv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) xv[e] = v < n ? __half2float(x[v * D + r * E + e]) : 0.0f;
    rotate_forward<E, L>(xv, r, sgn, q, qr, inv_sqrt_d, true, pair);
    // a zero (padding) vector quantises to zero in both variants: no error
    if constexpr (!ASYM) {
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(xv[e]));
#pragma unroll
      for (int m = 1; m < LPB; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, m));
      uint32_t bits;
      const float sq = round_scale(__fdiv_rn(amax + eps, QMAX), scale_type, bits);
      const float inv = sq > 0.0f ? __frcp_rn(sq) : 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float c = fminf(fmaxf(rintf(xv[e] * inv), -QMAX), QMAX);
        const float dlt = xv[e] - sq * c;
        err = fmaf(dlt, dlt, err);
      }
    } else {
      float mx = -INFINITY, mn = INFINITY;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        mx = fmaxf(mx, xv[e]);
        mn = fminf(mn, xv[e]);
      }
#pragma unroll
      for (int m = 1; m < LPB; m <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
        mn = fminf(mn, __shfl_xor_sync(kFull, mn, m));
      }
      uint32_t sb, zb;
      const float sq = round_scale(__fdiv_rn((mx - mn) + eps, UMAX), KVQ3_SCALE_E4M3, sb);
      const float zq = round_scale(mn, KVQ3_SCALE_E4M3, zb);
      const float inv = sq > 0.0f ? __frcp_rn(sq) : 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float u = fminf(fmaxf(rintf((xv[e] - zq) * inv), 0.0f), UMAX);
        const float dlt = xv[e] - fmaf(sq, u, zq);
        err = fmaf(dlt, dlt, err);
      }
    }
  }
  atomicAdd(&part[(r * E) / BLOCK], err);
  __syncthreads();
  if (threadIdx.x < NBQ) atomicAdd(&sse[(size_t)cand * NBQ + threadIdx.x], (double)part[threadIdx.x]);
}

template <int D, int BLOCK, int NBIT, bool ASYM>
cudaError_t launch_sse(const RotParams& rp, const CacheGeom& g, const float* quats, const float* quats_r, int P,
                       const __half* x, int64_t n, double* sse, cudaStream_t st) {
  constexpr int E = D >= 128 ? D / 32 : 4;
  constexpr int GPW = 32 / (D / E);
  int64_t blocks = (n + 8 * GPW - 1) / (8 * GPW);   // 8 warps per CTA
  const int64_t cap = (int64_t)sm_count() * 8 / P > 0 ? (int64_t)sm_count() * 8 / P : 1;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  calib_sse_kernel<D, E, BLOCK, NBIT, ASYM><<<dim3((unsigned)blocks, (unsigned)P), 256, 0, st>>>(
      rp, reinterpret_cast<const float4*>(quats), reinterpret_cast<const float4*>(quats_r), x, n, g.scale_type,
      g.eps, sse, inv_sqrt(D));
  return cudaGetLastError();
}

template <int D, int BLOCK>
cudaError_t dispatch_sse(const RotParams& rp, const CacheGeom& g, const float* quats, const float* quats_r,
                         int P, const __half* x, int64_t n, double* sse, cudaStream_t st) {
  if (g.scale_type == KVQ3_SCALE_E4M3_ZP)
    return launch_sse<D, BLOCK, 3, true>(rp, g, quats, quats_r, P, x, n, sse, st);
  if (g.bits == 2) return launch_sse<D, BLOCK, 2, false>(rp, g, quats, quats_r, P, x, n, sse, st);
  if (g.bits == 4) return launch_sse<D, BLOCK, 4, false>(rp, g, quats, quats_r, P, x, n, sse, st);
  return launch_sse<D, BLOCK, 3, false>(rp, g, quats, quats_r, P, x, n, sse, st);
}

kvq3_status calib_sse(const kvq3_rotation rot, const CacheGeom& g, const float* quats, const float* quats_r,
                      int32_t P, const void* x, int64_t n, double* sse, cudaStream_t st) {
  const int nbq = g.d / g.block;
  if (cudaMemsetAsync(sse, 0, (size_t)P * nbq * sizeof(double), st) != cudaSuccess) return KVQ3_ERR_CUDA;
  if (n == 0) return KVQ3_OK;
  const __half* xh = static_cast<const __half*>(x);
  cudaError_t e;
  switch (g.d * 1000 + g.block) {
    case 64032: e = dispatch_sse<64, 32>(rot->params, g, quats, quats_r, P, xh, n, sse, st); break;
    case 64064: e = dispatch_sse<64, 64>(rot->params, g, quats, quats_r, P, xh, n, sse, st); break;
    case 128032: e = dispatch_sse<128, 32>(rot->params, g, quats, quats_r, P, xh, n, sse, st); break;
    case 128064: e = dispatch_sse<128, 64>(rot->params, g, quats, quats_r, P, xh, n, sse, st); break;
    case 256032: e = dispatch_sse<256, 32>(rot->params, g, quats, quats_r, P, xh, n, sse, st); break;
    case 256064: e = dispatch_sse<256, 64>(rot->params, g, quats, quats_r, P, xh, n, sse, st); break;
    default: return KVQ3_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}

kvq3_status check_calib(const kvq3_rotation rot, const kvq3_cache_desc* desc, const void* x, int64_t n,
                        CacheGeom* g) {
  kvq3_status s = make_geom(desc, g);
  if (s != KVQ3_OK) return s;
  if (!rot || rot->d != g->d || n < 0 || (n > 0 && !x)) return KVQ3_ERR_INVALID_ARG;
  if (n >= ((int64_t)1 << 40)) return KVQ3_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return KVQ3_ERR_INVALID_ARG;
  return KVQ3_OK;
}

// SplitMix64 (reading R4's generator) for the proposal steps.
struct Mix64 {
  uint64_t s;
  uint64_t next() {
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform_pm1() { return (double)(next() >> 11) * 0x1p-53 * 2.0 - 1.0; }
};

// Random local search of reading R19 over one-quaternion blocks (quats_r_out
// == nullptr) or two-quaternion blocks (reading R20).  Candidate 0 of every
// round is the current set; candidates 1.. move every quaternion of the set
// by sigma * uniform [-1,1)^4 (left first, then right, per block) and
// renormalise; every quantisation block keeps its best candidate.
kvq3_status calibrate(kvq3_rotation rot, const CacheGeom& g, const void* x, int64_t n, int32_t rounds, int32_t P,
                      float step, uint64_t seed, void* workspace, float* quats_out, float* quats_r_out,
                      double* sse_out, cudaStream_t st) {
  const bool pair = quats_r_out != nullptr;
  const int d = g.d, nq = d / 4, nbq = d / g.block, per = g.block / 4;
  const size_t qbytes = ((size_t)P * d * sizeof(float) + 255) / 256 * 256;
  float* dq = static_cast<float*>(workspace);
  float* dqr = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + qbytes);
  double* dsse = reinterpret_cast<double*>(static_cast<uint8_t*>(workspace) + 2 * qbytes);
  std::vector<float> cur(4 * nq), cur_r(4 * nq), prop((size_t)P * 4 * nq), prop_r((size_t)P * 4 * nq);
  std::vector<double> hs((size_t)P * nbq);
  for (int i = 0; i < 4 * nq; ++i) {
    cur[i] = (float)rot->quats64[i];
    cur_r[i] = (float)rot->quats_r64[i];
  }
  Mix64 rng{seed};
  auto evaluate = [&](int ncand) -> kvq3_status {
    const size_t nb = (size_t)ncand * 4 * nq * sizeof(float);
    if (cudaMemcpyAsync(dq, prop.data(), nb, cudaMemcpyHostToDevice, st) != cudaSuccess) return KVQ3_ERR_CUDA;
    if (pair && cudaMemcpyAsync(dqr, prop_r.data(), nb, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return KVQ3_ERR_CUDA;
    kvq3_status r = calib_sse(rot, g, dq, pair ? dqr : nullptr, ncand, x, n, dsse, st);
    if (r != KVQ3_OK) return r;
    if (cudaMemcpyAsync(hs.data(), dsse, (size_t)ncand * nbq * sizeof(double), cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return KVQ3_ERR_CUDA;
    return KVQ3_OK;
  };
  auto perturb = [&](const float* from, float* to, double sigma) {
    double v[4], nrm = 0.0;
    for (int c = 0; c < 4; ++c) {
      v[c] = (double)from[c] + sigma * rng.uniform_pm1();
      nrm += v[c] * v[c];
    }
    nrm = sqrt(nrm);
    for (int c = 0; c < 4; ++c) to[c] = nrm > 0.0 ? (float)(v[c] / nrm) : from[c];
  };
  kvq3_status s;
  for (int t = 0; t < rounds; ++t) {
    const double sigma = (double)step * (1.0 - (double)t / rounds);
    memcpy(prop.data(), cur.data(), cur.size() * sizeof(float));   // candidate 0: the current set
    memcpy(prop_r.data(), cur_r.data(), cur_r.size() * sizeof(float));
    for (int p = 1; p < P; ++p)
      for (int i = 0; i < nq; ++i) {
        perturb(&cur[4 * i], &prop[(size_t)p * 4 * nq + 4 * i], sigma);
        if (pair) perturb(&cur_r[4 * i], &prop_r[(size_t)p * 4 * nq + 4 * i], sigma);
      }
    if ((s = evaluate(P)) != KVQ3_OK) return s;
    // each quantisation block keeps its best candidate (ties: the lower index)
    for (int j = 0; j < nbq; ++j) {
      int best = 0;
      for (int p = 1; p < P; ++p)
        if (hs[(size_t)p * nbq + j] < hs[(size_t)best * nbq + j]) best = p;
      if (best) {
        memcpy(&cur[4 * j * per], &prop[(size_t)best * 4 * nq + 4 * j * per], 4 * per * sizeof(float));
        memcpy(&cur_r[4 * j * per], &prop_r[(size_t)best * 4 * nq + 4 * j * per], 4 * per * sizeof(float));
      }
    }
  }
  memcpy(quats_out, cur.data(), cur.size() * sizeof(float));
  if (pair) memcpy(quats_r_out, cur_r.data(), cur_r.size() * sizeof(float));
  if (sse_out) {
    memcpy(prop.data(), cur.data(), cur.size() * sizeof(float));
    memcpy(prop_r.data(), cur_r.data(), cur_r.size() * sizeof(float));
    if ((s = evaluate(1)) != KVQ3_OK) return s;
    memcpy(sse_out, hs.data(), (size_t)nbq * sizeof(double));
  }
  return KVQ3_OK;
}

}  // namespace

extern "C" {

kvq3_status kvq3_calib_sse(kvq3_rotation rot, const kvq3_cache_desc* desc, const float* quats,
                           int32_t num_candidates, const void* x, int64_t n, double* sse,
                           void* stream) {
  CacheGeom g;
  kvq3_status s = check_calib(rot, desc, x, n, &g);
  if (s != KVQ3_OK) return s;
  if (num_candidates < 1 || num_candidates > 65535 || !quats || !sse) return KVQ3_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(quats) % 16 != 0) return KVQ3_ERR_INVALID_ARG;
  return calib_sse(rot, g, quats, nullptr, num_candidates, x, n, sse, static_cast<cudaStream_t>(stream));
}

kvq3_status kvq3_calib_sse_pair(kvq3_rotation rot, const kvq3_cache_desc* desc, const float* quats,
                                const float* quats_r, int32_t num_candidates, const void* x, int64_t n,
                                double* sse, void* stream) {
  CacheGeom g;
  kvq3_status s = check_calib(rot, desc, x, n, &g);
  if (s != KVQ3_OK) return s;
  if (num_candidates < 1 || num_candidates > 65535 || !quats || !quats_r || !sse) return KVQ3_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(quats) % 16 != 0 || reinterpret_cast<uintptr_t>(quats_r) % 16 != 0)
    return KVQ3_ERR_INVALID_ARG;
  return calib_sse(rot, g, quats, quats_r, num_candidates, x, n, sse, static_cast<cudaStream_t>(stream));
}

kvq3_status kvq3_calibrate_workspace_size(const kvq3_cache_desc* desc, int32_t num_candidates,
                                          size_t* bytes) {
  CacheGeom g;
  kvq3_status s = make_geom(desc, &g);
  if (s != KVQ3_OK) return s;
  if (num_candidates < 2 || num_candidates > 65535 || !bytes) return KVQ3_ERR_INVALID_ARG;
  // left and right candidate quaternions, then the per-block errors
  const size_t qb = ((size_t)num_candidates * g.d * sizeof(float) + 255) / 256 * 256;
  *bytes = 2 * qb + (size_t)num_candidates * (g.d / g.block) * sizeof(double);
  return KVQ3_OK;
}

static kvq3_status calibrate_checked(kvq3_rotation rot, const kvq3_cache_desc* desc, const void* x, int64_t n,
                                     int32_t rounds, int32_t num_candidates, float step, uint64_t seed,
                                     void* workspace, size_t ws_bytes, float* quats_out, float* quats_r_out,
                                     double* sse_out, void* stream) {
  CacheGeom g;
  kvq3_status s = check_calib(rot, desc, x, n, &g);
  if (s != KVQ3_OK) return s;
  size_t need = 0;
  if ((s = kvq3_calibrate_workspace_size(desc, num_candidates, &need)) != KVQ3_OK) return s;
  if (rounds < 0 || !(step >= 0.0f) || !isfinite(step) || !quats_out) return KVQ3_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256)
    return KVQ3_ERR_WORKSPACE;
  return calibrate(rot, g, x, n, rounds, num_candidates, step, seed, workspace, quats_out, quats_r_out, sse_out,
                   static_cast<cudaStream_t>(stream));
}

kvq3_status kvq3_calibrate_so4(kvq3_rotation rot, const kvq3_cache_desc* desc, const void* x, int64_t n,
                               int32_t rounds, int32_t num_candidates, float step, uint64_t seed,
                               void* workspace, size_t ws_bytes, float* quats_out, double* sse_out,
                               void* stream) {
  return calibrate_checked(rot, desc, x, n, rounds, num_candidates, step, seed, workspace, ws_bytes, quats_out,
                           nullptr, sse_out, stream);
}

kvq3_status kvq3_calibrate_so4_pair(kvq3_rotation rot, const kvq3_cache_desc* desc, const void* x, int64_t n,
                                    int32_t rounds, int32_t num_candidates, float step, uint64_t seed,
                                    void* workspace, size_t ws_bytes, float* quats_out, float* quats_r_out,
                                    double* sse_out, void* stream) {
  if (!quats_r_out) return KVQ3_ERR_INVALID_ARG;
  return calibrate_checked(rot, desc, x, n, rounds, num_candidates, step, seed, workspace, ws_bytes, quats_out,
                           quats_r_out, sse_out, stream);
}

}  // extern "C"
