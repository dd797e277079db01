// Instantiates the attention kernels for head dims padded to 128.
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_DEFINE_LAUNCH(128)
}  // namespace sdpa09
