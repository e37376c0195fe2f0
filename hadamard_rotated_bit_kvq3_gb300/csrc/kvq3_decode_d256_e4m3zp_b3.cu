// Decode-attention kernels for head dimension 256 in the asymmetric variant (E4M3
// scale and E4M3 zero point per block, unsigned 3-bit codes): both block
// sizes, all GQA group paddings, the chunked-prefill variant.
#include "kvq3_decode.cuh"

namespace kvq3 {
KVQ3_DECODE_INSTANCES(256, e4m3zp, KVQ3_SCALE_E4M3_ZP, 3)
}  // namespace kvq3
