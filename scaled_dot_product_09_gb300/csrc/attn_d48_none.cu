// Instantiates the attention kernels for head dims padded to 48, bias kind "none".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(48, kBiasNone, launch_attn_none)
}  // namespace sdpa09
