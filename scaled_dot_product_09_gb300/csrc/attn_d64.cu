// Instantiates the attention kernels for head dims padded to 64.
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_DEFINE_LAUNCH(64)
}  // namespace sdpa09
