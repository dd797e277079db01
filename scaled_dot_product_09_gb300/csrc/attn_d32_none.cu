// Instantiates the attention kernels for head dims padded to 32, bias kind "none".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(32, kBiasNone, launch_attn_none)
}  // namespace sdpa09
