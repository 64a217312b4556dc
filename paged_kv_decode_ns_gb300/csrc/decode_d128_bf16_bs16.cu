// head_dim 128 instantiations of the split-KV paged decode kernel (bf16), block size 16, group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE_QD(BF16, 16, false, 128)
}  // namespace ns
