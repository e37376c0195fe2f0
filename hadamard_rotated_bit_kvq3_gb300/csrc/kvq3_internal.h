// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>

#include "kvq3_common.cuh"

struct kvq3_rotation_s {
  int32_t d;
  uint32_t flags;
  int8_t signs[kvq3::kMaxD];      // as used (all +1 without KVQ3_ROT_SIGN)
  double quats64[kvq3::kMaxD];    // [d/4][4], unit length (identity without KVQ3_ROT_SO4)
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

// Tile-kernel path of kvq3_prefill_attn (d = 128; arguments already checked).
kvq3_status prefill_tiles(const CacheGeom& g, const kvq3_cache* cache, int32_t seq, int64_t pos0,
                          int64_t n_q, const void* q, int32_t hq, float qk_scale, float* out,
                          int32_t* dev_status, const RotParams& rp, cudaStream_t st);

inline kvq3_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ3_OK : KVQ3_ERR_CUDA; }

inline float inv_sqrt(int d) { return (float)(1.0 / __builtin_sqrt((double)d)); }

}  // namespace kvq3
