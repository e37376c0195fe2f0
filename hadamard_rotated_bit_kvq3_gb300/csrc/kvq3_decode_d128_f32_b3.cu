// Decode-attention kernels for head dimension 128, f32 scales and 3-bit codes
// (both block sizes, all GQA group paddings, the chunked-prefill variant); one
// translation unit per (head dimension, scale type, code width) for a
// parallel build.
#include "kvq3_decode.cuh"

namespace kvq3 {
KVQ3_DECODE_INSTANCES(128, f32, KVQ3_SCALE_F32, 3)
}  // namespace kvq3
