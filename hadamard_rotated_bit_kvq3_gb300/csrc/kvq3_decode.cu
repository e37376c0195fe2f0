// C ABI of the decode path: argument checks, launch planning, workspace size.
#include <math.h>
#include <string.h>

#include <algorithm>

#include <mutex>

#include "kvq3_decode.cuh"

using namespace kvq3;

namespace {

#define KVQ3_BY_BITS(D, SN, FN, ...)                               \
  switch (g.bits) {                                                \
    case 2: return FN##_d##D##_##SN##_b2(__VA_ARGS__);             \
    case 4: return FN##_d##D##_##SN##_b4(__VA_ARGS__);             \
    default: return FN##_d##D##_##SN##_b3(__VA_ARGS__);            \
  }
#define KVQ3_BY_SCALE(D, FN, ...)                                  \
  switch (g.scale_type) {                                          \
    case KVQ3_SCALE_F32: KVQ3_BY_BITS(D, f32, FN, __VA_ARGS__)     \
    case KVQ3_SCALE_F16: KVQ3_BY_BITS(D, f16, FN, __VA_ARGS__)     \
    case KVQ3_SCALE_E4M3_ZP: return FN##_d##D##_e4m3zp_b3(__VA_ARGS__); \
    default: KVQ3_BY_BITS(D, e4m3, FN, __VA_ARGS__)                \
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

kvq3_status prefill_plan_for(const CacheGeom& g, int G, DecodePlan* plan) {
  switch (g.d) {
    case 64: KVQ3_BY_SCALE(64, prefill_plan, g, G, plan)
    case 128: KVQ3_BY_SCALE(128, prefill_plan, g, G, plan)
    case 256: KVQ3_BY_SCALE(256, prefill_plan, g, G, plan)
  }
  return KVQ3_ERR_UNSUPPORTED;
}

kvq3_status prefill_run_for(const CacheGeom& g, const DecodePlan& plan, const DecodeParams& prm,
                            const RotParams& rp, float* out, cudaStream_t st) {
  switch (g.d) {
    case 64: KVQ3_BY_SCALE(64, prefill_run, plan, prm, rp, out, st)
    case 128: KVQ3_BY_SCALE(128, prefill_run, plan, prm, rp, out, st)
    case 256: KVQ3_BY_SCALE(256, prefill_run, plan, prm, rp, out, st)
  }
  return KVQ3_ERR_UNSUPPORTED;
}

kvq3_status check_heads(const CacheGeom& g, int32_t hq) {
  if (hq < 1 || hq % g.hkv != 0) return KVQ3_ERR_INVALID_ARG;
  if (hq / g.hkv > 16) return KVQ3_ERR_UNSUPPORTED;
  return KVQ3_OK;
}

// Prefill geometry: the G query heads of a kv head form hb blocks of hpb
// <= 8 heads; n_q query tokens form ceil(n_q / qt) blocks of qt = 8 / hpb
// tokens; a tile (token block, head block) is a unit of gcols = qt * hpb
// logit columns per kv head.  *vg is the cache geometry with the tiles as
// its batch.
kvq3_status prefill_geom(const kvq3_cache_desc* desc, int32_t hq, int64_t n_q, CacheGeom* vg,
                         int* qt, int* gcols, int* hb = nullptr, int* hpb = nullptr) {
  kvq3_status s = make_geom(desc, vg);
  if (s != KVQ3_OK) return s;
  if ((s = check_heads(*vg, hq)) != KVQ3_OK) return s;
  if (n_q < 0 || n_q >= ((int64_t)1 << 31)) return KVQ3_ERR_INVALID_ARG;
  const int G = hq / vg->hkv;
  const int nhb = (G + 7) / 8, per = (G + nhb - 1) / nhb;
  *qt = 8 / per;
  *gcols = *qt * per;
  if (hb) *hb = nhb;
  if (hpb) *hpb = per;
  const int64_t tiles = (n_q + *qt - 1) / *qt * nhb;
  if (tiles * vg->hkv >= ((int64_t)1 << 31)) return KVQ3_ERR_UNSUPPORTED;
  vg->batch = (int32_t)(tiles > 0 ? tiles : 1);
  return KVQ3_OK;
}

kvq3_status decode_attn_impl(kvq3_rotation rot, const kvq3_cache_desc* desc, const kvq3_cache* cache,
                             const void* q, int32_t num_q_heads, float sm_scale, float* out,
                             void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream,
                             uint32_t wait_polls) {
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
  prm.unit_cta = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) +
                                            ((size_t)plan.ctas + (size_t)g.batch * g.hkv) * G * (g.d + 2) *
                                                sizeof(float));
  prm.status = dev_status;
  prm.G = G;
  prm.Hq = num_q_heads;
  const double sc = sm_scale > 0.0f ? (double)sm_scale : 1.0 / sqrt((double)g.d);
  prm.qk_scale = (float)(sc * 1.4426950408889634);  // log2(e): softmax in base 2
  prm.inv_sqrt_d = inv_sqrt(g.d);
  prm.slot_floats = (uint32_t)(G * (g.d + 2));
  prm.wait_limit = wait_polls;
  return run_for(g, plan, prm, rot->params, out, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

kvq3_status kvq3_prefill_workspace_size(const kvq3_cache_desc* desc, int32_t num_q_heads,
                                        int64_t n_q, size_t* bytes) {
  CacheGeom vg;
  int qt = 0, gcols = 0;
  kvq3_status s = prefill_geom(desc, num_q_heads, n_q, &vg, &qt, &gcols);
  if (s != KVQ3_OK) return s;
  if (!bytes) return KVQ3_ERR_INVALID_ARG;
  DecodePlan plan;
  if ((s = prefill_plan_for(vg, gcols, &plan)) != KVQ3_OK) return s;
  *bytes = plan.ws_bytes;
  CacheGeom g;
  make_geom(desc, &g);
  if (prefill_tc_supported(g, num_q_heads))   // the tcgen05 path: split units' partials
    *bytes = std::max(*bytes, prefill_tc_workspace(g, num_q_heads, n_q));
  return KVQ3_OK;
}

static kvq3_status prefill_attn_impl(kvq3_rotation rot, const kvq3_cache_desc* desc,
                                     const kvq3_cache* cache, int32_t seq, int64_t pos0, int64_t n_q,
                                     const void* q, int32_t num_q_heads, float sm_scale, float* out,
                                     void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream,
                                     uint32_t wait_limit) {
  CacheGeom vg;
  int qt = 0, gcols = 0, hb = 0, hpb = 0;
  kvq3_status s = prefill_geom(desc, num_q_heads, n_q, &vg, &qt, &gcols, &hb, &hpb);
  if (s != KVQ3_OK) return s;
  if (!rot || rot->d != vg.d || !cache) return KVQ3_ERR_INVALID_ARG;
  if (seq < 0 || seq >= desc->batch || pos0 < 0 ||
      pos0 + n_q > (int64_t)vg.max_pages * vg.page_size || pos0 + n_q >= ((int64_t)1 << 31))
    return KVQ3_ERR_INVALID_ARG;
  if (n_q == 0) return KVQ3_OK;
  if (!q || !out || (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return KVQ3_ERR_INVALID_ARG;   // 16-byte accesses to both
  {
    CacheGeom g;   // the real geometry for the cache checks (lengths unused)
    make_geom(desc, &g);
    if ((s = check_cache(g, cache, false)) != KVQ3_OK) return s;
  }
  if (!(sm_scale <= 0.0f || isfinite(sm_scale))) return KVQ3_ERR_INVALID_ARG;
  DecodePlan plan;
  if ((s = prefill_plan_for(vg, gcols, &plan)) != KVQ3_OK) return s;
  if (!workspace || ws_bytes < plan.ws_bytes || reinterpret_cast<uintptr_t>(workspace) % 256)
    return KVQ3_ERR_WORKSPACE;
  const double qks = (sm_scale > 0.0f ? (double)sm_scale : 1.0 / sqrt((double)vg.d)) * 1.4426950408889634;
  {
    // shared dequantised tiles: each K/V tile is unpacked once for 128 query
    // rows on the tcgen05 path (d = 128, blocks of 64, b = 2-4), for 64 on
    // the mma.sync one (d = 128, blocks of 32, b = 3)
    CacheGeom g;
    make_geom(desc, &g);
    if (prefill_tc_supported(g, num_q_heads))
      return prefill_tc(g, cache, seq, pos0, n_q, q, num_q_heads, (float)qks, out, workspace, ws_bytes,
                        dev_status, rot->params, wait_limit, static_cast<cudaStream_t>(stream));
  }
  if (vg.d == 128 && vg.bits == 3 && vg.scale_type != KVQ3_SCALE_E4M3_ZP) {
    CacheGeom g;
    make_geom(desc, &g);
    return prefill_tiles(g, cache, seq, pos0, n_q, q, num_q_heads, (float)qks, out, dev_status,
                         rot->params, static_cast<cudaStream_t>(stream));
  }
  DecodeParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.g = vg;
  prm.pool = static_cast<const uint8_t*>(cache->pool);
  prm.page_table = cache->page_table;
  prm.seq_lens = nullptr;
  prm.q = static_cast<const __half*>(q);
  prm.ws = static_cast<float*>(workspace);
  prm.unit_cta = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) +
                                            ((size_t)plan.ctas + (size_t)vg.batch * vg.hkv) * gcols *
                                                (vg.d + 2) * sizeof(float));
  prm.status = dev_status;
  prm.G = gcols;
  prm.Hq = num_q_heads;
  const double sc = sm_scale > 0.0f ? (double)sm_scale : 1.0 / sqrt((double)vg.d);
  prm.qk_scale = (float)(sc * 1.4426950408889634);  // log2(e): softmax in base 2
  prm.inv_sqrt_d = inv_sqrt(vg.d);
  prm.slot_floats = (uint32_t)(gcols * (vg.d + 2));
  prm.wait_limit = wait_limit;
  prm.pf_n = (int32_t)n_q;
  prm.pf_qt = qt;
  prm.pf_hb = hb;
  prm.pf_hpb = hpb;
  prm.pf_gkv = num_q_heads / vg.hkv;
  prm.pf_seq = seq;
  prm.pf_pos0 = pos0;
  return prefill_run_for(vg, plan, prm, rot->params, out, static_cast<cudaStream_t>(stream));
}

kvq3_status kvq3_prefill_attn(kvq3_rotation rot, const kvq3_cache_desc* desc,
                              const kvq3_cache* cache, int32_t seq, int64_t pos0, int64_t n_q,
                              const void* q, int32_t num_q_heads, float sm_scale, float* out,
                              void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return prefill_attn_impl(rot, desc, cache, seq, pos0, n_q, q, num_q_heads, sm_scale, out, workspace,
                           ws_bytes, dev_status, stream, kWaitPolls);
}

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
  return decode_attn_impl(rot, desc, cache, q, num_q_heads, sm_scale, out, workspace, ws_bytes,
                          dev_status, stream, kWaitPolls);
}

// Test hook, not part of the public header: kvq3_decode_attn with the bound
// on each stage wait set to `polls` mbarrier polls.  With polls = 0 no wait
// can succeed, so every CTA takes its time-out path (flag KVQ3_DEV_TIMEOUT,
// drain its copies in flight, return) while every copy still targets valid
// memory: the time-out path runs without any fault or hang.
kvq3_status kvq3_test_decode_attn_polls(kvq3_rotation rot, const kvq3_cache_desc* desc,
                                        const kvq3_cache* cache, const void* q, int32_t num_q_heads,
                                        float sm_scale, float* out, void* workspace, size_t ws_bytes,
                                        int32_t* dev_status, void* stream, uint32_t polls) {
  return decode_attn_impl(rot, desc, cache, q, num_q_heads, sm_scale, out, workspace, ws_bytes,
                          dev_status, stream, polls);
}

// Test hook, not part of the public header: kvq3_prefill_attn with the bound
// on each mbarrier wait set to `polls` polls (the tcgen05 path and the decode
// kernel's prefill variant; the mma.sync tile kernel has no waits).  With
// polls = 0 every CTA takes its time-out path: it flags KVQ3_DEV_TIMEOUT,
// drains the copies and MMAs it issued, frees its tensor memory and returns.
kvq3_status kvq3_test_prefill_attn_polls(kvq3_rotation rot, const kvq3_cache_desc* desc,
                                         const kvq3_cache* cache, int32_t seq, int64_t pos0, int64_t n_q,
                                         const void* q, int32_t num_q_heads, float sm_scale, float* out,
                                         void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream,
                                         uint32_t polls) {
  return prefill_attn_impl(rot, desc, cache, seq, pos0, n_q, q, num_q_heads, sm_scale, out, workspace,
                           ws_bytes, dev_status, stream, polls);
}

}  // extern "C"

// ------------------------------------------------------------------ no-alloc
// Workspace of kvq3_decode_attn_noalloc: a fixed array in the library's
// device image, so the call itself never allocates.  Every GPU that loads the
// library holds it until the process exits.
namespace {

constexpr size_t kNoAllocBytes = (size_t)8 << 20;  // 8 MiB: KVQ3_DECODE_NOALLOC_MAX_BYTES
static_assert(kNoAllocBytes == KVQ3_DECODE_NOALLOC_MAX_BYTES, "header and library disagree");
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices];  // device address of g_noalloc_ws, per device

// Device address of the array on the current device.  The name g_noalloc_ws
// in host code is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and kept.
kvq3_status noalloc_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ3_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ3_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) return KVQ3_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return KVQ3_OK;
}

}  // namespace

extern "C" kvq3_status kvq3_decode_attn_noalloc(kvq3_rotation rot, const kvq3_cache_desc* desc,
                                                const kvq3_cache* cache, const void* q,
                                                int32_t num_q_heads, float sm_scale, float* out,
                                                int32_t* dev_status, void* stream) {
  size_t need = 0;
  kvq3_status s = kvq3_decode_workspace_size(desc, num_q_heads, &need);
  if (s != KVQ3_OK) return s;
  if (need > kNoAllocBytes) return KVQ3_ERR_WORKSPACE;
  void* ws = nullptr;
  if ((s = noalloc_workspace(&ws)) != KVQ3_OK) return s;
  return kvq3_decode_attn(rot, desc, cache, q, num_q_heads, sm_scale, out, ws, kNoAllocBytes,
                          dev_status, stream);
}
