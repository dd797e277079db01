// Instantiates the attention kernels for head dims padded to 64, bias kind "sam".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(64, kBiasSam, launch_attn_sam)
}  // namespace sdpa09
