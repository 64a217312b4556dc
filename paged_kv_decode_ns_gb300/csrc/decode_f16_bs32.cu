// f16 instantiations of the split-KV paged decode kernel, block size 32, group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE(F16, 32)
}  // namespace ns
