// Instantiates the attention kernels for head dims padded to 96.
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_DEFINE_LAUNCH(96)
}  // namespace sdpa09
