// attn_launch.cuh -- per-head-dim launcher of the attention kernel.  Each
// attn_d<DPAD>.cu translation unit instantiates one head-dim block so the
// build compiles them in parallel.
#pragma once
#include <cuda_runtime.h>
#include "attn_fwd_kernel.cuh"

namespace sdpa09 {

// Launches attn_fwd_kernel<DPAD, bias, dbg>.  Returns the cudaError_t of
// the attribute call or the launch.
template <int DPAD>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const AttnParams& p, int bias, bool dbg, int grid, size_t smem,
                        cudaStream_t stream);

#define SDPA09_DEFINE_LAUNCH(DPAD)                                                              \
    template <int BIAS, bool DBG>                                                               \
    static cudaError_t launch_attn_##DPAD##_impl(const CUtensorMap& tq, const CUtensorMap& tk,  \
                                                 const CUtensorMap& tv, const AttnParams& p,    \
                                                 int grid, size_t smem, cudaStream_t stream) {  \
        auto kern = attn_fwd_kernel<DPAD, BIAS, DBG>;                                           \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             (int)smem);                                        \
        if (e != cudaSuccess) return e;                                                         \
        kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);                                  \
        return cudaGetLastError();                                                              \
    }                                                                                           \
    template <>                                                                                 \
    cudaError_t launch_attn<DPAD>(const CUtensorMap& tq, const CUtensorMap& tk,                 \
                                  const CUtensorMap& tv, const AttnParams& p, int bias,         \
                                  bool dbg, int grid, size_t smem, cudaStream_t stream) {       \
        switch (bias * 2 + (dbg ? 1 : 0)) {                                                     \
            case 0: return launch_attn_##DPAD##_impl<kBiasNone, false>(tq, tk, tv, p, grid, smem, stream); \
            case 1: return launch_attn_##DPAD##_impl<kBiasNone, true>(tq, tk, tv, p, grid, smem, stream);  \
            case 2: return launch_attn_##DPAD##_impl<kBiasSwin, false>(tq, tk, tv, p, grid, smem, stream); \
            case 3: return launch_attn_##DPAD##_impl<kBiasSwin, true>(tq, tk, tv, p, grid, smem, stream);  \
            case 4: return launch_attn_##DPAD##_impl<kBiasSam, false>(tq, tk, tv, p, grid, smem, stream);  \
            case 5: return launch_attn_##DPAD##_impl<kBiasSam, true>(tq, tk, tv, p, grid, smem, stream);   \
            default: return cudaErrorInvalidValue;                                              \
        }                                                                                       \
    }

}  // namespace sdpa09
