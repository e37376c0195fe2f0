// Decode-attention kernels for head dimension 256, f32 scales and 2-bit codes
// (both block sizes, all GQA group paddings, the chunked-prefill variant); one
// translation unit per (head dimension, scale type, code width) for a
// parallel build.
#include "kvq3_decode.cuh"

namespace kvq3 {
KVQ3_DECODE_INSTANCES(256, f32, KVQ3_SCALE_F32, 2)
}  // namespace kvq3
