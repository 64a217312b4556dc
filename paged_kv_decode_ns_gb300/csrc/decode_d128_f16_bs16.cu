// head_dim 128 instantiations of the split-KV paged decode kernel (f16), block size 16, group sizes 1..8.
#include "paged_decode_launch.cuh"

namespace ns {
NS_INSTANTIATE_DECODE_QD(F16, 16, false, 128)
}  // namespace ns
