// Instantiates the attention kernels for head dims padded to 32.
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_DEFINE_LAUNCH(32)
}  // namespace sdpa09
