// bf16 instantiations of the split-KV paged decode kernel, block size 8, group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE(BF16, 8)
}  // namespace ns
