// bf16 instantiations of the split-KV paged decode kernel for short walks (the
// values pass unrolled a few row groups a trip), block size 16, head_dim 64,
// group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE_SHORT(BF16, 16)
}  // namespace ns
