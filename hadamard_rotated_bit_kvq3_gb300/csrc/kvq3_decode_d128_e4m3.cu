// Decode-attention kernels for head dimension 128 with e4m3 scales (both block
// sizes, all GQA group paddings); one translation unit per (head dimension,
// scale type) for a parallel build.
#include "kvq3_decode.cuh"

namespace kvq3 {
KVQ3_DECODE_INSTANCES(128, e4m3, KVQ3_SCALE_E4M3)
}  // namespace kvq3
