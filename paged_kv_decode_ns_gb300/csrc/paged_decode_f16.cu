// fp16 instantiations of the split-KV paged decode kernel.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE(F16, 4)
NS_INSTANTIATE_DECODE(F16, 8)
NS_INSTANTIATE_DECODE(F16, 16)
NS_INSTANTIATE_DECODE(F16, 32)
}  // namespace ns
