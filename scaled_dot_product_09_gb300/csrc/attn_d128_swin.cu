// Instantiates the attention kernels for head dims padded to 128, bias kind "swin".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(128, kBiasSwin, launch_attn_swin)
}  // namespace sdpa09
