// bf16 instantiations of the split-KV paged decode kernel.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE(BF16, 4)
NS_INSTANTIATE_DECODE(BF16, 8)
NS_INSTANTIATE_DECODE(BF16, 16)
NS_INSTANTIATE_DECODE(BF16, 32)
}  // namespace ns
