// Instantiates the attention kernels for head dims padded to 48, bias kind "swin".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(48, kBiasSwin, launch_attn_swin)
}  // namespace sdpa09
