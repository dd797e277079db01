// Instantiates the attention kernels for head dims padded to 80.
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_DEFINE_LAUNCH(80)
}  // namespace sdpa09
