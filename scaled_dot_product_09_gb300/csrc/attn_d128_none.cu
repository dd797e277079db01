// Instantiates the attention kernels for head dims padded to 128, bias kind "none".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(128, kBiasNone, launch_attn_none)
}  // namespace sdpa09
