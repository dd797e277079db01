// Instantiates the attention kernels for head dims padded to 80, bias kind "swin".
#include "attn_launch.cuh"

namespace sdpa09 {
SDPA09_INSTANTIATE(80, kBiasSwin, launch_attn_swin)
}  // namespace sdpa09
