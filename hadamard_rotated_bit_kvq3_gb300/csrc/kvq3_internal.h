// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>

#include "kvq3_common.cuh"

struct kvq3_rotation_s {
  int32_t d;
  uint32_t flags;
  int8_t signs[kvq3::kMaxD];      // as used (all +1 without KVQ3_ROT_SIGN)
  double quats64[kvq3::kMaxD];    // [d/4][4] p_i, unit length (identity without KVQ3_ROT_SO4)
  double quats_r64[kvq3::kMaxD];  // [d/4][4] q_i, unit length (identity without KVQ3_ROT_SO4_PAIR)
  kvq3::RotParams params;         // what the kernels receive
};

namespace kvq3 {

// Validates a cache description for the cache kernels (d in {64,128,256},
// block in {32,64}, bits in {2,3,4}, ...) and derives the geometry.
kvq3_status make_geom(const kvq3_cache_desc* desc, CacheGeom* g);

// Validates the device buffers of a cache against its geometry.
kvq3_status check_cache(const CacheGeom& g, const kvq3_cache* cache, bool need_lens);

// Number of streaming multiprocessors of the current device (cached).
int sm_count();

// Bound on the polls of a drain after a timed-out wait (the normal waits take
// the kernel's wait limit).
constexpr uint32_t kDrainPolls = 1u << 22;
// Default bound on the polls of an mbarrier wait.
constexpr uint32_t kWaitPolls = 1u << 22;

// tcgen05 path of kvq3_prefill_attn: d = 128, 3-bit symmetric codes, blocks
// of 64, at most 128 query heads per kv head (arguments already checked).
bool prefill_tc_supported(const CacheGeom& g, int32_t hq);
size_t prefill_tc_workspace(const CacheGeom& g, int32_t hq, int64_t n_q);
kvq3_status prefill_tc(const CacheGeom& g, const kvq3_cache* cache, int32_t seq, int64_t pos0, int64_t n_q,
                       const void* q, int32_t hq, float qk_scale, float* out, void* workspace, size_t ws_bytes,
                       int32_t* dev_status, const RotParams& rp, uint32_t wait_limit, cudaStream_t st);

// Tile-kernel path of kvq3_prefill_attn (d = 128; arguments already checked).
kvq3_status prefill_tiles(const CacheGeom& g, const kvq3_cache* cache, int32_t seq, int64_t pos0,
                          int64_t n_q, const void* q, int32_t hq, float qk_scale, float* out,
                          int32_t* dev_status, const RotParams& rp, cudaStream_t st);

inline kvq3_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ3_OK : KVQ3_ERR_CUDA; }

inline float inv_sqrt(int d) { return (float)(1.0 / __builtin_sqrt((double)d)); }

// Block i of B as a row-major 4x4 matrix in fp64: L(p_i), or L(p_i) R(conj q_i)
// for two-quaternion blocks (readings R3, R20); the identity without SO(4).
inline void so4_block_matrix(const kvq3_rotation_s* r, int i, double M[16]) {
  const double* p = &r->quats64[4 * i];
  const double* q = &r->quats_r64[4 * i];
  const double a = p[0], b = p[1], c = p[2], e = p[3];
  const double Lp[16] = {a, -b, -c, -e, b, a, -e, c, c, e, a, -b, e, -c, b, a};
  // x -> x * conj(q): the right-multiplication matrix of conj(q)
  const double w = q[0], x = -q[1], y = -q[2], z = -q[3];
  const double Rq[16] = {w, -x, -y, -z, x, w, z, -y, y, -z, w, x, z, y, -x, w};
  const bool pair = (r->flags & KVQ3_ROT_SO4_PAIR) != 0;
  for (int row = 0; row < 4; ++row)
    for (int col = 0; col < 4; ++col) {
      double v = 0.0;
      if (pair) {
        for (int k = 0; k < 4; ++k) v += Lp[4 * row + k] * Rq[4 * k + col];
      } else {
        v = Lp[4 * row + col];
      }
      M[4 * row + col] = v;
    }
}

}  // namespace kvq3
