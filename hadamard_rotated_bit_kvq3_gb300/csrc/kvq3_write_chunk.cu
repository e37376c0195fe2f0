// Write path for a contiguous chunk of positions of one sequence (prefill):
// rotate, quantise and pack every K and V vector of tokens pos0..pos0+n-1.
//
// "Orthogonally mixed 3-bit KV cache", Implementation notes (write path) and
// Key formulas; "Orthogonal Invariance in Activation Space", 3.1-3.4.  Same
// arithmetic and stored format as kvq3_write (include/kvq3.h R1-R9), laid out
// for throughput:
//  * one thread per vector (d = 64 or 128 values in registers), 128 vectors
//    (consecutive tokens of one kv head, K or V) per CTA tile;
//  * the tile's fp16 rows are staged through shared memory with cp.async
//    (16-byte pieces, XOR-swizzled so both the coalesced fill and the
//    row-per-thread read are bank-conflict free), double-buffered;
//  * sign flip D as an XOR of fp16 sign bits with masks from the constant
//    bank; the Walsh-Hadamard butterfly with packed f32x2 adds (element i
//    and i + d/2 share a register pair, so every stage but the last is packed);
//    SO(4) blocks as 4x4 matrices (one- or two-quaternion blocks alike),
//    blocks i and i + d/8 packed;
//  * 1/sqrt(d) is folded into the block maximum and the reciprocal scale;
//  * codes by one fused multiply-add against the 1.5*2^23 rounding constant
//    (round half to even), packed in-thread into 32-bit words (b-bit codes,
//    b = 2, 3, 4: divisor and clip bound 2^(b-1) - 1), stored with 16-byte
//    stores.
#include <string.h>

#include "kvq3_internal.h"

using namespace kvq3;

namespace {

constexpr int kTile = 128;  // vectors per CTA tile = threads per CTA
constexpr int kChunkMaxD = 128;  // head dimensions this path serves: 64, 128

struct ChunkParams {
  CacheGeom g;
  uint8_t* pool;
  const int32_t* page_table;
  const __half* k;
  const __half* v;
  int32_t* status;
  int64_t pos0, n_tok;
  int32_t seq;
  int32_t tiles_per_head;     // ceil(n_tok / kTile)
  int64_t n_tiles;            // 2 * hkv * tiles_per_head
  float inv_sqrt_d;
  uint32_t sign_xor[kMaxD / 2];   // fp16-pair sign masks of the input order
  float2 mat2[kChunkMaxD / 8][16];  // SO(4) block matrices of blocks (i, i + d/8), row-major
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}

// tile -> (K|V, kv head, first token); all counts fit 32 bits (checked on the host)
struct TileId {
  int which, head;
  uint32_t tok0;
};
__device__ __forceinline__ TileId tile_id(const ChunkParams& p, uint32_t tile) {
  const uint32_t per_which = (uint32_t)p.g.hkv * (uint32_t)p.tiles_per_head;
  TileId id;
  id.which = tile >= per_which;
  const uint32_t rem = tile - (id.which ? per_which : 0u);
  id.head = (int)(rem / (uint32_t)p.tiles_per_head);
  id.tok0 = (rem - (uint32_t)id.head * (uint32_t)p.tiles_per_head) * kTile;
  return id;
}

template <int D, int BLOCK, int SCALE, bool SO4, int NBIT>
__global__ void __launch_bounds__(kTile) write_chunk_kernel(const __grid_constant__ ChunkParams p) {
  constexpr int H = D / 2;              // register pairs: x2[k] = (x[k], x[k + H])
  constexpr int ROWB = 2 * D;           // bytes per input row
  constexpr int PIECES = ROWB / 16;     // 16-byte pieces per row (8 or 16)
  constexpr int NB = D / BLOCK;
  constexpr int CB = NBIT * D / 8;      // code bytes (16 .. 64)
  constexpr int QMAX = (1 << (NBIT - 1)) - 1;
  constexpr int SB = SCALE == KVQ3_SCALE_F32 ? 4 : (SCALE == KVQ3_SCALE_F16 || SCALE == KVQ3_SCALE_E4M3_ZP) ? 2 : 1;
  // a kernel launched after this one as a programmatic dependent may start
  // now; it waits for this grid's writes before it reads anything
  griddep_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  const int t = threadIdx.x;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const CacheGeom& g = p.g;

  // stage the rows of tile `tile` into buffer `buf`
  auto load_tile = [&](uint32_t tile, int buf) {
    const TileId id = tile_id(p, tile);
    const uint32_t tok0 = id.tok0;
    const __half* src = (id.which ? p.v : p.k) + id.head * D;
    const uint32_t dst = sbase + (uint32_t)buf * kTile * ROWB;
#pragma unroll
    for (int i = 0; i < PIECES; ++i) {
      const int idx = i * kTile + t;            // piece index in the tile
      const int row = idx / PIECES, pc = idx % PIECES;
      const uint32_t tok = tok0 + row;
      const bool valid = tok < (uint32_t)p.n_tok;
      const __half* s = src + (size_t)(valid ? tok : 0u) * (uint32_t)(g.hkv * D) + pc * 8;
      cp_async16(dst + row * ROWB + ((pc ^ (row & (PIECES - 1))) * 16), s, valid);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  const uint32_t n_tiles = (uint32_t)p.n_tiles;
  uint32_t tile = blockIdx.x;
  if (tile >= n_tiles) return;
  load_tile(tile, 0);
  for (int it = 0; tile < n_tiles; ++it, tile += gridDim.x) {
    const int buf = it & 1;
    const uint32_t next = tile + gridDim.x;
    if (next < n_tiles) load_tile(next, buf ^ 1);
    else asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();

    // ---- this thread's vector: row t of the tile
    const TileId id = tile_id(p, tile);
    const int which = id.which, head = id.head;
    const uint32_t tok = id.tok0 + t;
    float2 x2[H];
    {
      const uint32_t rowa = sbase + (uint32_t)buf * kTile * ROWB + t * ROWB;
#pragma unroll
      for (int pc = 0; pc < PIECES; ++pc) {
        uint4 w;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "r"(rowa + ((pc ^ (t & (PIECES - 1))) * 16)));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = pc * 8 + 2 * q;          // elements e, e+1
          const uint32_t h = ww[q] ^ p.sign_xor[e / 2];
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
          if (e < H) {
            x2[e].x = f.x;
            x2[e + 1].x = f.y;
          } else {
            x2[e - H].y = f.x;
            x2[e + 1 - H].y = f.y;
          }
        }
      }
    }
    __syncthreads();  // the buffer is refilled two tiles later

    // ---- Walsh-Hadamard butterfly: stages h < H packed, stage H inside pairs
#pragma unroll
    for (int h = 1; h < H; h <<= 1) {
#pragma unroll
      for (int i = 0; i < H; ++i) {
        if ((i & h) == 0) {
          const float2 a = x2[i], b = x2[i + h];
          x2[i] = f2add(a, b);
          x2[i + h] = f2sub(a, b);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const float a = x2[i].x, b = x2[i].y;
      x2[i].x = a + b;
      x2[i].y = a - b;
    }
    // ---- SO(4) blocks (matrix entries carry 1/sqrt(d) when present)
    if constexpr (SO4) {
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const float2 x0 = x2[4 * i], x1 = x2[4 * i + 1], xx2 = x2[4 * i + 2], x3 = x2[4 * i + 3];
#pragma unroll
        for (int row = 0; row < 4; ++row) {
          const float2* m = &p.mat2[i][4 * row];
          x2[4 * i + row] = f2fma(m[0], x0, f2fma(m[1], x1, f2fma(m[2], xx2, f2mul(m[3], x3))));
        }
      }
    }
    // x2 now holds sqrt(d) * (U x) (or U x when SO4 folded 1/sqrt(d) in)
    const float post = SO4 ? 1.0f : p.inv_sqrt_d;

    // ---- scales and codes, block by block
    const bool ok_tok = tok < (uint32_t)p.n_tok;
    const uint32_t pos = (uint32_t)p.pos0 + tok;        // < capacity < 2^31
    const uint32_t lp = pos / (uint32_t)g.page_size;
    int64_t page = -1;
    if (ok_tok) {
      page = page_of(g, p.page_table, p.seq, lp);
      if (page < 0) set_status(p.status, KVQ3_DEV_BAD_PAGE);
    }
    uint32_t words[CB / 4];
#pragma unroll
    for (int w = 0; w < CB / 4; ++w) words[w] = 0;
    uint32_t sbits[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if constexpr (SCALE == KVQ3_SCALE_E4M3_ZP) {
        // asymmetric variant: E4M3 scale (max - min + eps)/(2^b - 1) and E4M3
        // zero point min; unsigned codes round((x - z_q)/s_q) clipped to [0, 2^b - 1]
        constexpr float UMAX = (float)((1 << NBIT) - 1);
        float mx = -INFINITY, mn = INFINITY;
#pragma unroll
        for (int j = b * BLOCK; j < (b + 1) * BLOCK; ++j) {
          const float xv = j < H ? x2[j].x : x2[j - H].y;
          mx = fmaxf(mx, xv);
          mn = fminf(mn, xv);
        }
        uint32_t sb8, zb8;
        const float sq = round_scale(__fdiv_rn((mx - mn) * post + g.eps, UMAX), KVQ3_SCALE_E4M3, sb8);
        const float zq = round_scale(mn * post, KVQ3_SCALE_E4M3, zb8);
        sbits[b] = sb8 | (zb8 << 8);
        const float r = sq > 0.0f ? __frcp_rn(sq) : 0.0f;
        const float inv = r * post, zoff = -zq * r;
#pragma unroll
        for (int j = b * BLOCK; j < (b + 1) * BLOCK; ++j) {
          const float xv = j < H ? x2[j].x : x2[j - H].y;
          float tq = fmaf(xv, inv, zoff) + 12582912.0f;      // 1.5 * 2^23 + rint((x - z_q) / s_q)
          tq = fminf(fmaxf(tq, 12582912.0f), 12582912.0f + UMAX);
          const uint32_t c = __float_as_uint(tq) & ((1u << NBIT) - 1u);
          const int bit = NBIT * j;
          words[bit / 32] |= c << (bit % 32);
          if (bit % 32 > 32 - NBIT) words[bit / 32 + 1] |= c >> (32 - bit % 32);
        }
        continue;
      }
      float amax = 0.0f;
#pragma unroll
      for (int j = b * BLOCK; j < (b + 1) * BLOCK; ++j)
        amax = fmaxf(amax, fabsf(j < H ? x2[j].x : x2[j - H].y));
      const float s = __fdiv_rn(amax * post + g.eps, (float)QMAX);
      uint32_t bits;
      const float sq = round_scale(s, SCALE, bits);
      sbits[b] = bits;
      const float inv = sq > 0.0f ? __frcp_rn(sq) * post : 0.0f;
#pragma unroll
      for (int j = b * BLOCK; j < (b + 1) * BLOCK; ++j) {
        const float xv = j < H ? x2[j].x : x2[j - H].y;
        float tq = fmaf(xv, inv, 12582912.0f);            // 1.5 * 2^23 + rint(x / s_q)
        if constexpr (SCALE != KVQ3_SCALE_F32)   // clip to [-QMAX, QMAX]
          tq = fminf(fmaxf(tq, 12582912.0f - QMAX), 12582912.0f + QMAX);
        const uint32_t c = __float_as_uint(tq) & ((1u << NBIT) - 1u);   // b-bit two's complement
        const int bit = NBIT * j;
        words[bit / 32] |= c << (bit % 32);
        if (bit % 32 > 32 - NBIT) words[bit / 32 + 1] |= c >> (32 - bit % 32);
      }
    }
    if (page >= 0 && KVQ3_CHECK(p.status, in_range(record_offset(g, page, head, which), g.record_bytes,
                                                  g.num_pages * g.page_bytes) &&
                                         pos - lp * (uint32_t)g.page_size < (uint32_t)g.page_size)) {
      const int slot = (int)(pos - lp * (uint32_t)g.page_size);
      uint8_t* rec = p.pool + record_offset(g, page, head, which);
      uint8_t* cp = rec + g.scale_hdr_bytes + (int64_t)slot * CB;
      if constexpr (CB % 16 == 0) {   // 16-byte multiples (all but 3-bit d = 64), 16-byte aligned
        uint4* cd = reinterpret_cast<uint4*>(cp);
#pragma unroll
        for (int w = 0; w < CB / 16; ++w)
          cd[w] = make_uint4(words[4 * w], words[4 * w + 1], words[4 * w + 2], words[4 * w + 3]);
      } else {                        // d = 64: 24-byte strings, 8-byte aligned
        uint2* cd = reinterpret_cast<uint2*>(cp);
#pragma unroll
        for (int w = 0; w < CB / 8; ++w) cd[w] = make_uint2(words[2 * w], words[2 * w + 1]);
      }
      uint8_t* sp = rec + (int64_t)slot * NB * SB;
      if constexpr (SCALE == KVQ3_SCALE_E4M3_ZP) {   // (scale, zero point) byte pairs
#pragma unroll
        for (int b = 0; b < NB; ++b) reinterpret_cast<uint16_t*>(sp)[b] = (uint16_t)sbits[b];
      } else if constexpr (SB == 4) {
#pragma unroll
        for (int b = 0; b < NB; ++b) reinterpret_cast<uint32_t*>(sp)[b] = sbits[b];
      } else if constexpr (SB == 2) {
#pragma unroll
        for (int b = 0; b < NB; ++b) reinterpret_cast<uint16_t*>(sp)[b] = (uint16_t)sbits[b];
      } else {
#pragma unroll
        for (int b = 0; b < NB; ++b) sp[b] = (uint8_t)sbits[b];
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int D, int BLOCK, int SCALE, bool SO4, int NBIT>
cudaError_t launch_chunk_b(const ChunkParams& p, cudaStream_t st) {
  const size_t smem = 2 * (size_t)kTile * 2 * D;
  auto k = write_chunk_kernel<D, BLOCK, SCALE, SO4, NBIT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTile, smem);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
  if (grid > p.n_tiles) grid = p.n_tiles;
  k<<<(unsigned)grid, kTile, smem, st>>>(p);
  return cudaGetLastError();
}

template <int D, int BLOCK, int SCALE, bool SO4>
cudaError_t launch_chunk(const ChunkParams& p, cudaStream_t st) {
  if constexpr (SCALE == KVQ3_SCALE_E4M3_ZP) return launch_chunk_b<D, BLOCK, SCALE, SO4, 3>(p, st);   // 3-bit only
  if (p.g.bits == 2) return launch_chunk_b<D, BLOCK, SCALE, SO4, 2>(p, st);
  if (p.g.bits == 4) return launch_chunk_b<D, BLOCK, SCALE, SO4, 4>(p, st);
  return launch_chunk_b<D, BLOCK, SCALE, SO4, 3>(p, st);
}

template <int D, int BLOCK>
cudaError_t dispatch_chunk(const ChunkParams& p, int scale, bool so4, cudaStream_t st) {
  if (scale == KVQ3_SCALE_F32)
    return so4 ? launch_chunk<D, BLOCK, KVQ3_SCALE_F32, true>(p, st) : launch_chunk<D, BLOCK, KVQ3_SCALE_F32, false>(p, st);
  if (scale == KVQ3_SCALE_F16)
    return so4 ? launch_chunk<D, BLOCK, KVQ3_SCALE_F16, true>(p, st) : launch_chunk<D, BLOCK, KVQ3_SCALE_F16, false>(p, st);
  if (scale == KVQ3_SCALE_E4M3_ZP)
    return so4 ? launch_chunk<D, BLOCK, KVQ3_SCALE_E4M3_ZP, true>(p, st) : launch_chunk<D, BLOCK, KVQ3_SCALE_E4M3_ZP, false>(p, st);
  return so4 ? launch_chunk<D, BLOCK, KVQ3_SCALE_E4M3, true>(p, st) : launch_chunk<D, BLOCK, KVQ3_SCALE_E4M3, false>(p, st);
}

}  // namespace

extern "C" kvq3_status kvq3_write_chunk(kvq3_rotation rot, const kvq3_cache_desc* desc,
                                        const kvq3_cache* cache, const void* k, const void* v,
                                        int32_t seq, int64_t pos0, int64_t n_tok,
                                        int32_t* dev_status, void* stream) {
  CacheGeom g;
  kvq3_status s = make_geom(desc, &g);
  if (s != KVQ3_OK) return s;
  if (!rot || rot->d != g.d || n_tok < 0) return KVQ3_ERR_INVALID_ARG;
  if ((s = check_cache(g, cache, false)) != KVQ3_OK) return s;
  if (n_tok == 0) return KVQ3_OK;
  if (!k || !v || seq < 0 || seq >= g.batch || pos0 < 0 ||
      pos0 + n_tok > (int64_t)g.max_pages * g.page_size)
    return KVQ3_ERR_INVALID_ARG;
  // 32-bit position, token and tile arithmetic on the device
  if (pos0 + n_tok >= ((int64_t)1 << 31) || n_tok * g.hkv * g.d >= ((int64_t)1 << 32))
    return KVQ3_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16 != 0)
    return KVQ3_ERR_INVALID_ARG;
  if (g.d > 128) {
    // d = 256 does not fit one thread: the general path handles it
    return KVQ3_ERR_UNSUPPORTED;
  }
  ChunkParams p;
  memset(&p, 0, sizeof(p));
  p.g = g;
  p.pool = static_cast<uint8_t*>(cache->pool);
  p.page_table = cache->page_table;
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.status = dev_status;
  p.pos0 = pos0;
  p.n_tok = n_tok;
  p.seq = seq;
  p.tiles_per_head = (int32_t)((n_tok + kTile - 1) / kTile);
  p.n_tiles = 2 * (int64_t)g.hkv * p.tiles_per_head;
  p.inv_sqrt_d = inv_sqrt(g.d);
  const int d = g.d;
  for (int e = 0; e < d / 2; ++e) {
    uint32_t m = 0;
    if (rot->signs[2 * e] < 0) m |= 0x8000u;
    if (rot->signs[2 * e + 1] < 0) m |= 0x80000000u;
    p.sign_xor[e] = m;
  }
  const bool so4 = (rot->flags & KVQ3_ROT_SO4) != 0;
  const double isd = 1.0 / sqrt((double)d);
  if (d > kChunkMaxD) return KVQ3_ERR_UNSUPPORTED;
  for (int i = 0; i < d / 8; ++i) {
    double Ma[16], Mb[16];
    so4_block_matrix(rot, i, Ma);
    so4_block_matrix(rot, i + d / 8, Mb);
    for (int c = 0; c < 16; ++c) p.mat2[i][c] = make_float2((float)(Ma[c] * isd), (float)(Mb[c] * isd));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const int key = g.d * 1000 + g.block;
  switch (key) {
    case 64032: e = dispatch_chunk<64, 32>(p, g.scale_type, so4, st); break;
    case 64064: e = dispatch_chunk<64, 64>(p, g.scale_type, so4, st); break;
    case 128032: e = dispatch_chunk<128, 32>(p, g.scale_type, so4, st); break;
    case 128064: e = dispatch_chunk<128, 64>(p, g.scale_type, so4, st); break;
    default: return KVQ3_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}
