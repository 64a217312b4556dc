// bf16 instantiations of the split-KV paged decode kernel with two-level merges,
// block size 16, head_dim 64, group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE_TWO(BF16, 16)
}  // namespace ns
