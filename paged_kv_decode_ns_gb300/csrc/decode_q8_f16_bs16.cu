// q8_0-pool instantiations of the split-KV paged decode kernel (f16 q and output), block size 16, group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE_Q(F16, 16, true)
}  // namespace ns
