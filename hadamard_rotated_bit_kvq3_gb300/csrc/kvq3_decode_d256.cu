// Decode-attention kernels for head dimension 256 (all block sizes and GQA
// group paddings); one translation unit per head dimension for a parallel
// build.
#include "kvq3_decode.cuh"

namespace kvq3 {
KVQ3_DECODE_INSTANCES(256)
}  // namespace kvq3
