// Instantiates the attention kernels for head dims padded to 80, bias kind "none".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(80, kBiasNone, launch_attn_none)
}  // namespace sdpa09
