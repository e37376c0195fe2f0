// Decode-attention kernels for head dimension 256 with f16 scales (both block
// sizes, all GQA group paddings); one translation unit per (head dimension,
// scale type) for a parallel build.
#include "kvq3_decode.cuh"

namespace kvq3 {
KVQ3_DECODE_INSTANCES(256, f16, KVQ3_SCALE_F16)
}  // namespace kvq3
