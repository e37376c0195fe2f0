/*
 * kvq3.h -- C ABI of the orthogonally rotated 3-bit KV cache (GB300, sm_103a).
 *
 * Method.  Every key and value head vector is rotated by an orthogonal
 * U = B . H_d . D and stored as signed 3-bit codes with one scale per block
 * of m rotated coordinates; decode attention rotates the query by the same U,
 * reads the packed cache directly (unpack, scale and dot product fused), runs
 * an online softmax, multiplies by the dequantised values and rotates the
 * output back with U^T.
 *
 * Sources (page title, then section):
 *   [OMC] "Orthogonally mixed 3-bit KV cache" -- Mathematical statement
 *         (H_d^T H_d = I, R_i in SO(4), B = diag(R_1..R_{d/4}), U = B H_d,
 *         (Uq)^T(Uk) = q^T k, v' = Uv rotated back with U^T, the scale
 *         s = (max_j|x_j| + eps)/(2^(b-1)-1) and the code
 *         clip(round(x/s), -(2^(b-1)-1), 2^(b-1)-1) with b = 3); Key formulas
 *         (Attn = softmax(QK^T/sqrt d) V); Implementation notes (write path:
 *         k1 = U(k), v1 = U(v), one scale per block, signed 3-bit codes packed
 *         into bytes, only codes and scales stored; read path: q1 = U(q),
 *         keys unpacked and scaled inside the dot product, softmax, multiply
 *         by reconstructed values, y = U^T y1, with no full-precision K/V ever
 *         formed; SO(4) blocks from normalised quaternions, fixed random
 *         rotations for a first version).
 *   [OIQ] "Orthogonal Invariance in Activation Space: Fast Walsh-Hadamard
 *         Transforms for KV Quantization" -- 3.1 (normalised FWHT, self
 *         inverse), 3.2 (random sign flip D applied before the FWHT, generated
 *         once and stored as a fixed parameter), 3.3 (store / retrieve /
 *         attention pipeline), 3.4 (per-group scales, default g = 32),
 *         4.2 (record = scale header followed by packed codes),
 *         4.3 (dequantisation fused into the attention kernel).
 *   [HFF] "Hardware-Fused Fast Hadamard Transforms Enable Lossless 3-Bit
 *         KV-Cache Compression at 128K Context" -- 64-element sub-blocks with
 *         an FP8 scale header, 3.125 effective bits per element.
 *
 * Readings fixed by this library where the pages are silent or disagree:
 *   R1  H_d is the normalised Walsh-Hadamard matrix in natural (Sylvester)
 *       order, H[i][j] = (-1)^popcount(i&j) / sqrt(d).
 *   R2  U = B . H_d . D: sign flip first, then H_d, then the SO(4) blocks.
 *   R3  R_i is the left-multiplication matrix of the unit quaternion
 *       p_i = (a, b, c, e) (x -> p_i * x as a quaternion product):
 *       [[a,-b,-c,-e],[b,a,-e,c],[c,e,a,-b],[e,-c,b,a]]; it acts on rotated
 *       coordinates 4i..4i+3.  With KVQ3_ROT_SO4_PAIR, R20 instead.
 *   R20 The general element of SO(4) ([OMC] Mathematical statement: R_i in
 *       SO(4)) as a pair of unit quaternions: R_i x = p_i * x * conj(q_i),
 *       i.e. L(p_i) R(conj q_i) with R(q) the right-multiplication matrix
 *       x -> x * q = [[a,-b,-c,-e],[b,a,e,-c],[c,-e,a,b],[e,c,-b,a]].  From a
 *       seed, q_i is one more Marsaglia point per block drawn after all the
 *       p_i (R4), so the signs and p_i are those of the one-quaternion
 *       rotation with the same seed.
 *   R4  Seed -> parameters: SplitMix64 (Steele, Lea & Flood 2014) seeded with
 *       the seed.  Draws 0..d-1 give the signs (sign -1 when the top bit is
 *       set); then for each block i a uniform point of S^3 by Marsaglia's 1972
 *       method, with uniforms u = (next() >> 11) * 2^-53 * 2 - 1, pairs with
 *       s = x^2 + y^2 outside (0, 1) rejected, all in IEEE fp64 without fused
 *       multiply-add; the device uses the fp32 roundings of the quaternions.
 *       Flags choose whether the drawn signs / quaternions are used
 *       (otherwise +1 / identity); the draws are made either way.
 *   R5  eps is taken as given (1e-6 by default) and kept in the formula.
 *   R6  round = round half to even.
 *   R7  The scale is rounded to its storage type first (fp32, or fp16 / OCP
 *       FP8-E4M3 with round-to-nearest-even saturating to the largest finite
 *       value) and the codes are computed with the stored scale s_q:
 *       c = clip(round(x / s_q), -3, 3); c = 0 where s_q == 0.  Dequantisation
 *       is exactly s_q * c.
 *   R8  Codes are 3-bit two's complement (-3 = 0b101); 0b100 (-4) is never
 *       written.
 *   R9  Code string of a vector: element j at bits 3j..3j+2 of a
 *       little-endian bit stream of 3d/8 bytes (bit k of the stream is bit
 *       k%8 of byte k/8).  Blocks are consecutive rotated coordinates
 *       [0,m), [m,2m), ...
 *   R18 The asymmetric variant of [HFF] (per 64-element sub-block: unsigned
 *       3-bit codes and an FP8 header with a scale and a zero point), scale
 *       type KVQ3_SCALE_E4M3_ZP: per block z = min x and
 *       s = (max x - min x + eps)/7, each stored as one E4M3 byte (RNE,
 *       saturating; scale byte first), unsigned codes
 *       u = clip(round((x - z_q)/s_q), 0, 7) (u = 0 where s_q == 0) in the
 *       R9 bit stream, x_hat = s_q*u + z_q.  Two header bytes per block
 *       (3.25 bits per element at m = 64): the page's 3.125-bit figure would
 *       leave one byte for both and is not followed.  3-bit codes only.
 *   R19 SO(4) calibration (kvq3_calibrate_so4): the page asks for the
 *       quaternions that minimise the post-quantisation reconstruction MSE
 *       on sample vectors and names no search; taken as a random local
 *       search that keeps, per quantisation block, the best of the current
 *       set and perturbed copies: one quaternion per block
 *       (kvq3_calibrate_so4) or the pair of R20 (kvq3_calibrate_so4_pair).
 *   R17 Other code widths b = 2 and 4 ([OIQ] 3.3 stores d*b bits per
 *       vector, 4.2 packs INT3/INT4 values, 5.1 evaluates b = 4, 3, 2; [OMC]
 *       writes its quantiser for any b): divisor and clip bound
 *       2^(b-1) - 1 (1, 3, 7) in R7, b-bit two's complement in R8 (-2^(b-1)
 *       is never written), element j at bits b*j..b*j+b-1 of a b*d/8-byte
 *       string in R9.
 *   R10 One scale per block and no per-vector scale ([OMC]); [OIQ] 4.2's
 *       header count does not add up and is not followed.
 *   R11 The query is rotated by the same U as the keys ([OMC] q1 = U(q)).
 *   R12 Logits are scaled by sm_scale, 1/sqrt(d) by default ([OMC] Key
 *       formulas; the page's Implementation notes sketch writes the logits
 *       without the scale, and the formula is taken over the sketch).
 *   R13 Decode attends to positions [0, seq_lens[b]); the caller appends the
 *       current token with kvq3_write and advances seq_lens itself.
 *   R14 Query head h reads kv head h / (Hq/Hkv) (consecutive grouping).
 *   R15 The output is fp32 and unrotated; an empty sequence gives zeros.
 *
 * Cache layout (the "chunk record" of [OIQ] 4.2, one per page, kv head and
 * K|V).  P = page_size tokens per page (a multiple of 16), nb = d/m blocks,
 * sb = scale bytes (4, 2, 1), cb = b*d/8 code bytes (3d/8 at b = 3):
 *   record  = [ scales: P*nb entries, token-major (slot t, block j at t*nb+j),
 *                       sb bytes each, little-endian ]
 *             [ codes : P code strings of cb bytes (slot t at t*cb) ]
 *             R = P*(nb*sb + cb) bytes
 *   page    = for kv head 0..Hkv-1: K record, V record   (Hkv*2*R bytes)
 *   pool    = num_pages pages
 * Position pos of sequence b lives in slot pos % P of logical page pos / P.
 * The physical page is page_table[b*max_pages_per_seq + pos/P] for a paged
 * cache, or b*max_pages_per_seq + pos/P for a contiguous cache (no table).
 * Every record and page size is a multiple of 16 bytes.
 *
 * Ownership.  The caller owns every buffer: pool, page table, lengths,
 * inputs, outputs and the decode workspace (all device memory unless stated).
 * The library's only allocation is the rotation handle itself (host memory,
 * in kvq3_rotation_create*).  No entry point synchronises the device.
 * Every device-side call is asynchronous on the given stream (a
 * cudaStream_t passed as void*, NULL = legacy default stream) and runs on
 * the device that is current for the calling thread.
 *
 * Errors.  Argument checks run on the host before any launch and return a
 * kvq3_status; nothing is launched then.  Launch failures return
 * KVQ3_ERR_CUDA.  Bad data found on the device (a position or page id out of
 * range, a length above capacity, a stored code of -4, a wait that ran out)
 * sets bits of the optional caller-provided device word *dev_status
 * (atomicOr) and the kernel skips the affected unit; kernels never trap.
 */
#ifndef KVQ3_H_
#define KVQ3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ3_ABI_VERSION 3   /* 2: code widths 2-4, the asymmetric scale type, calibration;
                                3: two-quaternion SO(4) blocks (KVQ3_ROT_SO4_PAIR) */

typedef enum {
  KVQ3_OK = 0,
  KVQ3_ERR_INVALID_ARG = 1,   /* a pointer, size or layout field is invalid */
  KVQ3_ERR_UNSUPPORTED = 2,   /* valid, but not compiled in (d, m, bits, G) */
  KVQ3_ERR_CUDA = 3,          /* a CUDA call or kernel launch failed */
  KVQ3_ERR_WORKSPACE = 4      /* decode workspace missing or too small */
} kvq3_status;

typedef enum {
  KVQ3_SCALE_F32 = 0,
  KVQ3_SCALE_F16 = 1,
  KVQ3_SCALE_E4M3 = 2,
  KVQ3_SCALE_E4M3_ZP = 3      /* asymmetric variant (R18): E4M3 scale and E4M3
                                 zero point per block, unsigned codes; b = 3 */
} kvq3_scale_type;

/* Rotation flags.  H_d is always applied.  KVQ3_ROT_SO4_PAIR (with
 * KVQ3_ROT_SO4) makes every SO(4) block the general two-quaternion rotation
 * of R20. */
enum { KVQ3_ROT_SIGN = 1u, KVQ3_ROT_SO4 = 2u, KVQ3_ROT_SO4_PAIR = 4u };

/* Bits of the device status word. */
enum {
  KVQ3_DEV_BAD_SEQ = 1,      /* sequence index outside [0, batch) */
  KVQ3_DEV_BAD_POS = 2,      /* position outside [0, max_pages_per_seq*P) */
  KVQ3_DEV_BAD_PAGE = 4,     /* page id outside [0, num_pages) */
  KVQ3_DEV_BAD_LEN = 8,      /* seq_lens[b] outside [0, capacity] */
  KVQ3_DEV_BAD_CODE = 16,    /* a stored code of -2^(b-1), e.g. -4 at b = 3 (never written) */
  KVQ3_DEV_TIMEOUT = 32,     /* an asynchronous copy did not arrive in time */
  KVQ3_DEV_CHECK = 64        /* a bounds check of a checked build failed (the
                                library compiled with KVQ3_CHECKED); the
                                access was skipped */
};

/* Opaque, immutable rotation U = B . H_d . D (host memory). */
typedef struct kvq3_rotation_s *kvq3_rotation;

/* Static description of a cache. */
typedef struct {
  int32_t head_dim;          /* d: 64, 128 or 256 for the cache kernels;
                                any power of two 4..256 for kvq3_rotate */
  int32_t num_kv_heads;      /* Hkv >= 1 */
  int32_t block;             /* m: 32 or 64, divides d */
  int32_t bits;              /* b: code width, 2, 3 or 4 (R17) */
  int32_t scale_type;        /* kvq3_scale_type */
  float eps;                 /* eps of the scale formula (1e-6) */
  int32_t page_size;         /* P: tokens per page, a positive multiple of 16 */
  int32_t batch;             /* number of sequences */
  int32_t max_pages_per_seq; /* page-table row length (capacity / P) */
  int32_t reserved;          /* 0 */
  int64_t num_pages;         /* pages in the pool */
} kvq3_cache_desc;

/* Device buffers of a cache. */
typedef struct {
  void *pool;                /* num_pages * page_bytes, 16-byte aligned */
  const int32_t *page_table; /* [batch][max_pages_per_seq] or NULL: contiguous */
  const int32_t *seq_lens;   /* [batch] attended lengths (decode only) */
} kvq3_cache;

/* ABI version of the loaded library (KVQ3_ABI_VERSION). */
int32_t kvq3_abi_version(void);

/* Human-readable name of a status code (static string). */
const char *kvq3_status_string(kvq3_status s);

/* Creates the rotation of head dimension d (a power of two, 4 <= d <= 256)
 * from a seed (reading R4; [OIQ] 3.2: the signs are drawn once and kept as a
 * fixed parameter; [OMC] Implementation notes: fixed random rotations built
 * from normalised quaternions).  flags: KVQ3_ROT_SIGN | KVQ3_ROT_SO4.  *out receives a handle
 * owned by the caller (free with kvq3_rotation_destroy).  Host only. */
kvq3_status kvq3_rotation_create(int32_t d, uint64_t seed, uint32_t flags,
                                 kvq3_rotation *out);

/* Creates a rotation from explicit parameters (host arrays): signs[d] in
 * {+1,-1}, quats[d/4][4] (a, b, c, e) -- each is normalised to unit length in
 * fp64 before use; a zero quaternion is rejected.  Host only. */
kvq3_status kvq3_rotation_create_from_params(int32_t d, const int8_t *signs,
                                             const float *quats,
                                             kvq3_rotation *out);

/* Creates a two-quaternion rotation (R20) from explicit parameters (host
 * arrays): signs[d], quats[d/4][4] (p_i) and quats_r[d/4][4] (q_i), each
 * quaternion normalised in fp64 (a zero one is rejected).  Flags of the
 * handle: KVQ3_ROT_SIGN | KVQ3_ROT_SO4 | KVQ3_ROT_SO4_PAIR.  Host only. */
kvq3_status kvq3_rotation_create_from_params_pair(int32_t d, const int8_t *signs,
                                                  const float *quats, const float *quats_r,
                                                  kvq3_rotation *out);

/* Frees a rotation handle (NULL is accepted). */
kvq3_status kvq3_rotation_destroy(kvq3_rotation rot);

/* Copies the parameters the device uses into host arrays: signs[d] and
 * quats[d/4][4] (fp32); *d_out (nullable) receives d. */
kvq3_status kvq3_rotation_export(kvq3_rotation rot, int8_t *signs, float *quats,
                                 int32_t *d_out);

/* As kvq3_rotation_export, plus quats_r[d/4][4] (nullable), the right
 * quaternions q_i the device uses ((1,0,0,0) for a one-quaternion rotation). */
kvq3_status kvq3_rotation_export_pair(kvq3_rotation rot, int8_t *signs, float *quats,
                                      float *quats_r, int32_t *d_out);

/* Byte sizes of a record, a page and the whole pool for a description. */
kvq3_status kvq3_cache_sizes(const kvq3_cache_desc *desc, size_t *record_bytes,
                             size_t *page_bytes, size_t *pool_bytes);

/* y = U x (inverse = 0) or y = U^T x (inverse != 0) for n_vec vectors of
 * dimension d ([OMC] k1 = U(k), q1 = U(q), y = U.T @ y1).
 * x: device [n_vec][d], fp32 (x_is_fp16 = 0) or fp16 (x_is_fp16 = 1);
 * y: device fp32 [n_vec][d].  fp32 arithmetic.  n_vec = 0 is a no-op. */
kvq3_status kvq3_rotate(kvq3_rotation rot, const void *x, int32_t x_is_fp16,
                        float *y, int64_t n_vec, int32_t inverse, void *stream);

/* Write path ([OMC] Implementation notes: each new token's key and value are
 * rotated by U, split into quantisation blocks with one scale each, rounded
 * to signed 3-bit codes and packed; only codes and scales are kept): for
 * every token i and kv head, the K and V vectors are rotated, quantised (R7)
 * and stored in the slot of (seq_idx[i], pos[i]).  Appends one token per
 * sequence (decode) or a prefill chunk (many positions of one or more
 * sequences).
 * k, v: device fp16 [n_tok][Hkv][d], 16-byte aligned; seq_idx, pos: device
 * int32 [n_tok].  2 * n_tok * Hkv must stay below 2^31 (KVQ3_ERR_UNSUPPORTED
 * otherwise).  Tokens whose slot is invalid are skipped and flagged in
 * *dev_status (nullable).  Two tokens with the same slot race (last writer
 * unspecified). */
kvq3_status kvq3_write(kvq3_rotation rot, const kvq3_cache_desc *desc,
                       const kvq3_cache *cache, const void *k, const void *v,
                       const int32_t *seq_idx, const int32_t *pos, int64_t n_tok,
                       int32_t *dev_status, void *stream);

/* Write path for a prefill chunk: positions pos0 .. pos0+n_tok-1 of sequence
 * seq, with k, v: device fp16 [n_tok][Hkv][d] (row i is position pos0 + i).
 * The same formula as kvq3_write ([OMC] Implementation notes, write path),
 * without per-token index arrays: one thread per vector, rows staged through
 * shared memory, packed f32x2 butterfly.  Both are fp32 computations with
 * different summation orders, so the stored bytes agree except where an
 * element's |x/s_q| lies within about 1e-6 relative of a rounding boundary
 * (or a block's scale at a rounding midpoint of its storage type), where
 * either neighbour may be stored.  d must be 64 or 128
 * (KVQ3_ERR_UNSUPPORTED otherwise; kvq3_write covers d = 256).  The position
 * range must lie inside the sequence's capacity (KVQ3_ERR_INVALID_ARG);
 * invalid page ids are skipped and flagged in *dev_status. */
kvq3_status kvq3_write_chunk(kvq3_rotation rot, const kvq3_cache_desc *desc,
                             const kvq3_cache *cache, const void *k, const void *v,
                             int32_t seq, int64_t pos0, int64_t n_tok,
                             int32_t *dev_status, void *stream);

/* Bytes of device workspace kvq3_decode_attn needs for num_q_heads query
 * heads on the current device (0 < *bytes, a few MB). */
kvq3_status kvq3_decode_workspace_size(const kvq3_cache_desc *desc,
                                       int32_t num_q_heads, size_t *bytes);

/* Read path ([OMC] Implementation notes: the query is rotated to q1 = U(q);
 * keys are unpacked and scaled inside the attention dot product, logits come
 * from q1 and the reconstructed rotated keys, then softmax, then the product
 * with the reconstructed rotated values, and the output is rotated back with
 * U^T; [OIQ] 4.3 fused dequantisation): one decode step of all sequences.
 * q: device fp16 [batch][Hq][d]; out: device fp32 [batch][Hq][d];
 * sm_scale <= 0 means 1/sqrt(d); Hq must be a multiple of Hkv with
 * Hq/Hkv <= 16.  The attended length of sequence b is seq_lens[b]
 * (device int32), 0 <= seq_lens[b] <= max_pages_per_seq*P.
 * workspace: device, ws_bytes >= kvq3_decode_workspace_size (256-byte
 * aligned); it holds split partials between the two kernels of one call, so
 * calls that share a workspace must not overlap.  A sequence with a bad
 * length is skipped (zero output, KVQ3_DEV_BAD_LEN); a bad page id masks that
 * page (KVQ3_DEV_BAD_PAGE). */
kvq3_status kvq3_decode_attn(kvq3_rotation rot, const kvq3_cache_desc *desc,
                             const kvq3_cache *cache, const void *q,
                             int32_t num_q_heads, float sm_scale, float *out,
                             void *workspace, size_t ws_bytes,
                             int32_t *dev_status, void *stream);

/* Largest decode workspace kvq3_decode_attn_noalloc can serve (bytes). */
#define KVQ3_DECODE_NOALLOC_MAX_BYTES (8u << 20)

/* kvq3_decode_attn without a caller-provided workspace (none of the pages
 * has a counterpart: this is a deployment convenience).  For callers that
 * cannot allocate device memory when they call -- for instance a serving loop
 * whose memory is entirely reserved by its framework at start-up, or a plugin
 * that is handed tensors but no allocator.  The call allocates nothing: the
 * split partials go to a fixed 8 MiB array built into the library
 * (KVQ3_DECODE_NOALLOC_MAX_BYTES), which every GPU that loads the library
 * keeps until the process exits.  Arguments and results are those of
 * kvq3_decode_attn.
 *   - Returns KVQ3_ERR_WORKSPACE, with nothing launched, when the call would
 *     need more than the array holds (kvq3_decode_workspace_size tells).
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     The address is kept for the life of the process: after a
 *     cudaDeviceReset (or any other teardown of the device's primary
 *     context) the module may load elsewhere, so do not call this entry
 *     point again on that device after such a reset.
 *   - All calls share the one array per device, and it keeps whatever the
 *     last call left in it (nothing needs clearing: every partial the merge
 *     reads is written earlier in the same call).  Calls that overlap on the
 *     GPU -- on different streams, or from several host threads -- race on
 *     it and give wrong results; serialise them. */
kvq3_status kvq3_decode_attn_noalloc(kvq3_rotation rot, const kvq3_cache_desc *desc,
                                     const kvq3_cache *cache, const void *q,
                                     int32_t num_q_heads, float sm_scale, float *out,
                                     int32_t *dev_status, void *stream);

/* Chunked-prefill attention over the packed cache ([OMC] read path and Key
 * formulas with a causal mask; the pages quantise keys and values during the
 * prefill phase as well as decode, and the same fused read applies): query
 * token i, at position pos0 + i of sequence seq, attends to positions
 * [0, pos0 + i] of that sequence -- one decode step of the sequence cut
 * after its own position.  The positions must already be in the cache (e.g.
 * written by kvq3_write_chunk); seq_lens is not read.
 * q: device fp16 [n_q][Hq][d]; out: device fp32 [n_q][Hq][d]; both 16-byte
 * aligned (else KVQ3_ERR_INVALID_ARG); sm_scale <= 0 means 1/sqrt(d); Hq a
 * multiple of Hkv with Hq/Hkv <= 16.  Internally the
 * queries form tiles of up to 8 (query token, head) pairs per kv head; at
 * d = 128 with symmetric codes and blocks of 64, units of 128 such rows, a
 * long unit's keys split in 2 to 16 ranges (one per 8,192 keys) whose
 * partial results meet in the workspace, so the workspace grows with the
 * longest context the cache holds, max_pages_per_seq * P.
 * workspace:
 * device, ws_bytes >= kvq3_prefill_workspace_size(desc, Hq, n_q), 256-byte
 * aligned; calls sharing it must not overlap.  n_q = 0 is a no-op;
 * KVQ3_ERR_INVALID_ARG when seq is out of range or pos0 + n_q exceeds the
 * sequence capacity max_pages_per_seq * P. */
kvq3_status kvq3_prefill_workspace_size(const kvq3_cache_desc *desc, int32_t num_q_heads,
                                        int64_t n_q, size_t *bytes);
kvq3_status kvq3_prefill_attn(kvq3_rotation rot, const kvq3_cache_desc *desc,
                              const kvq3_cache *cache, int32_t seq, int64_t pos0,
                              int64_t n_q, const void *q, int32_t num_q_heads,
                              float sm_scale, float *out, void *workspace, size_t ws_bytes,
                              int32_t *dev_status, void *stream);

/* Reads back positions t0..t0+nt-1 of sequence seq, kv head kv_head, K
 * (which = 0) or V (which = 1) as fp32 out[nt][d]: s_q * c in the rotated
 * domain (rot == NULL) or U^T (s_q * c) (rot != NULL) ([OIQ] 3.3 "Retrieve").
 * codes_out (nullable): int32 [nt][d] raw codes.  Positions without a valid
 * slot give zeros and set *dev_status bits; a stored -2^(b-1) (-4 at b = 3)
 * sets KVQ3_DEV_BAD_CODE and reads as 0.  A debugging and testing aid. */
kvq3_status kvq3_dequant_debug(kvq3_rotation rot, const kvq3_cache_desc *desc,
                               const kvq3_cache *cache, int32_t seq,
                               int32_t kv_head, int32_t which, int64_t t0,
                               int64_t nt, float *out, int32_t *codes_out,
                               int32_t *dev_status, void *stream);

/* ---- SO(4) calibration ([OMC] Implementation notes: calibrate the fixed
 * random rotations on representative sequences by minimising the
 * reconstruction MSE after quantisation, each SO(4) block a normalised
 * quaternion).  Offline tools, not on the decode path.
 *
 * kvq3_calib_sse: for num_candidates (P) quaternion sets, the squared
 * reconstruction error of the sample under each, per quantisation block:
 * sse[p][j] = sum over the n vectors and the coordinates i of block j of
 * (y_i - y_hat_i)^2, y = B_p H D x (the rotation's signs, candidate p's
 * quaternions, SO(4) blocks always applied) and y_hat its quantised value
 * under desc's block size, code width, scale format and eps (the write
 * path's arithmetic, fp32).  Since U is orthogonal, sum_j sse[p][j] is the
 * error of U^T y_hat against x.
 * quats: device fp32 [P][d/4][4], 16-byte aligned; x: device fp16 [n][d],
 * 16-byte aligned; sse: device fp64 [P][d/block], overwritten.  Only d,
 * block, bits, scale_type and eps of desc are used (the rest must still be
 * valid).  1 <= P <= 65535; n = 0 gives zeros. */
kvq3_status kvq3_calib_sse(kvq3_rotation rot, const kvq3_cache_desc *desc, const float *quats,
                           int32_t num_candidates, const void *x, int64_t n, double *sse,
                           void *stream);

/* kvq3_calib_sse for candidate two-quaternion blocks (R20): candidate p's
 * quaternion pair of block i is (quats[p][i], quats_r[p][i]); both device
 * fp32 [P][d/4][4], 16-byte aligned.  Otherwise as kvq3_calib_sse. */
kvq3_status kvq3_calib_sse_pair(kvq3_rotation rot, const kvq3_cache_desc *desc, const float *quats,
                                const float *quats_r, int32_t num_candidates, const void *x, int64_t n,
                                double *sse, void *stream);

/* Device workspace bytes of kvq3_calibrate_so4 and kvq3_calibrate_so4_pair
 * with num_candidates (>= 2). */
kvq3_status kvq3_calibrate_workspace_size(const kvq3_cache_desc *desc, int32_t num_candidates,
                                          size_t *bytes);

/* Random local search over the quaternions of rot (reading R19): each of
 * `rounds` rounds evaluates the current set and num_candidates - 1 copies in
 * which every quaternion moves by sigma * (uniform [-1,1)^4, SplitMix64
 * seeded with `seed`) and is renormalised, with sigma = step * (1 - t/rounds)
 * in round t, in one kvq3_calib_sse launch; every quantisation block keeps
 * the candidate with the lowest error (ties: the current set), which is
 * possible because block j of y depends only on its own m/4 quaternions.
 * So no block's error ever rises.  quats_out: host fp32 [d/4][4] (the rotation
 * itself is not changed: kvq3_rotation_create_from_params makes the
 * calibrated one); sse_out (nullable): host fp64 [d/block], the final error.
 * workspace: device, >= kvq3_calibrate_workspace_size bytes, 256-byte
 * aligned.  Synchronises the stream once per round (host decisions). */
kvq3_status kvq3_calibrate_so4(kvq3_rotation rot, const kvq3_cache_desc *desc, const void *x,
                               int64_t n, int32_t rounds, int32_t num_candidates, float step,
                               uint64_t seed, void *workspace, size_t ws_bytes, float *quats_out,
                               double *sse_out, void *stream);

/* The search of kvq3_calibrate_so4 over two-quaternion blocks (R20): every
 * round perturbs both quaternions of every block (each by its own
 * sigma * uniform [-1,1)^4 step, renormalised) and every quantisation block
 * keeps its best pair.  The start is rot's pairs (q_i = 1 for a
 * one-quaternion rotation).  quats_out, quats_r_out: host fp32 [d/4][4];
 * sse_out (nullable) as in kvq3_calibrate_so4.  Synchronises the stream once
 * per round. */
kvq3_status kvq3_calibrate_so4_pair(kvq3_rotation rot, const kvq3_cache_desc *desc, const void *x,
                                    int64_t n, int32_t rounds, int32_t num_candidates, float step,
                                    uint64_t seed, void *workspace, size_t ws_bytes, float *quats_out,
                                    float *quats_r_out, double *sse_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ3_H_ */
