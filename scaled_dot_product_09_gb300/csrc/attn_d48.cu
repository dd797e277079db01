// Instantiates the attention kernels for head dims padded to 48.
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_DEFINE_LAUNCH(48)
}  // namespace sdpa09
