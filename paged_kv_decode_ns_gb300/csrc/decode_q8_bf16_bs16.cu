// q8_0-pool instantiations of the split-KV paged decode kernel (bf16 q and output), block size 16, group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE_Q(BF16, 16, true)
}  // namespace ns
