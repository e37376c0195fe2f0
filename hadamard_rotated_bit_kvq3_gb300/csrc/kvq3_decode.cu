// C ABI of the decode path: argument checks, launch planning, workspace size.
#include <math.h>
#include <string.h>

#include "kvq3_decode.cuh"

using namespace kvq3;

namespace {

#define KVQ3_BY_SCALE(D, FN, ...)                                  \
  switch (g.scale_type) {                                          \
    case KVQ3_SCALE_F32: return FN##_d##D##_f32(__VA_ARGS__);      \
    case KVQ3_SCALE_F16: return FN##_d##D##_f16(__VA_ARGS__);      \
    default: return FN##_d##D##_e4m3(__VA_ARGS__);                 \
  }

kvq3_status plan_for(const CacheGeom& g, int G, DecodePlan* plan) {
  switch (g.d) {
    case 64: KVQ3_BY_SCALE(64, decode_plan, g, G, plan)
    case 128: KVQ3_BY_SCALE(128, decode_plan, g, G, plan)
    case 256: KVQ3_BY_SCALE(256, decode_plan, g, G, plan)
  }
  return KVQ3_ERR_UNSUPPORTED;
}

kvq3_status run_for(const CacheGeom& g, const DecodePlan& plan, const DecodeParams& prm,
                    const RotParams& rp, float* out, cudaStream_t st) {
  switch (g.d) {
    case 64: KVQ3_BY_SCALE(64, decode_run, plan, prm, rp, out, st)
    case 128: KVQ3_BY_SCALE(128, decode_run, plan, prm, rp, out, st)
    case 256: KVQ3_BY_SCALE(256, decode_run, plan, prm, rp, out, st)
  }
  return KVQ3_ERR_UNSUPPORTED;
}

kvq3_status check_heads(const CacheGeom& g, int32_t hq) {
  if (hq < 1 || hq % g.hkv != 0) return KVQ3_ERR_INVALID_ARG;
  if (hq / g.hkv > 16) return KVQ3_ERR_UNSUPPORTED;
  return KVQ3_OK;
}

}  // namespace

extern "C" {

kvq3_status kvq3_decode_workspace_size(const kvq3_cache_desc* desc, int32_t num_q_heads,
                                       size_t* bytes) {
  CacheGeom g;
  kvq3_status s = make_geom(desc, &g);
  if (s != KVQ3_OK) return s;
  if (!bytes) return KVQ3_ERR_INVALID_ARG;
  if ((s = check_heads(g, num_q_heads)) != KVQ3_OK) return s;
  DecodePlan plan;
  if ((s = plan_for(g, num_q_heads / g.hkv, &plan)) != KVQ3_OK) return s;
  *bytes = plan.ws_bytes;
  return KVQ3_OK;
}

kvq3_status kvq3_decode_attn(kvq3_rotation rot, const kvq3_cache_desc* desc,
                             const kvq3_cache* cache, const void* q, int32_t num_q_heads,
                             float sm_scale, float* out, void* workspace, size_t ws_bytes,
                             int32_t* dev_status, void* stream) {
  CacheGeom g;
  kvq3_status s = make_geom(desc, &g);
  if (s != KVQ3_OK) return s;
  if (!rot || rot->d != g.d || !q || !out) return KVQ3_ERR_INVALID_ARG;
  if ((s = check_cache(g, cache, true)) != KVQ3_OK) return s;
  if ((s = check_heads(g, num_q_heads)) != KVQ3_OK) return s;
  if (!(sm_scale <= 0.0f || isfinite(sm_scale))) return KVQ3_ERR_INVALID_ARG;
  const int G = num_q_heads / g.hkv;
  DecodePlan plan;
  if ((s = plan_for(g, G, &plan)) != KVQ3_OK) return s;
  if (!workspace || ws_bytes < plan.ws_bytes || reinterpret_cast<uintptr_t>(workspace) % 256)
    return KVQ3_ERR_WORKSPACE;
  DecodeParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = g;
  prm.pool = static_cast<const uint8_t*>(cache->pool);
  prm.page_table = cache->page_table;
  prm.seq_lens = cache->seq_lens;
  prm.q = static_cast<const __half*>(q);
  prm.ws = static_cast<float*>(workspace);
  prm.status = dev_status;
  prm.G = G;
  prm.Hq = num_q_heads;
  const double sc = sm_scale > 0.0f ? (double)sm_scale : 1.0 / sqrt((double)g.d);
  prm.qk_scale = (float)(sc * 1.4426950408889634);  // log2(e): softmax in base 2
  prm.inv_sqrt_d = inv_sqrt(g.d);
  prm.slot_floats = (uint32_t)(G * (g.d + 2));
  prm.wait_limit = 1u << 22;
  return run_for(g, plan, prm, rot->params, out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
