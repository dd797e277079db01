// Instantiates and launches the packed-windows backward kernel
// (attn_bwd_kernel.cuh) for head dims padded to 32, 48 and 64, no bias or the
// Swin bias, and slots of 32, 64 or 128 rows.
#include <cuda_runtime.h>
#include "attn_bwd_kernel.cuh"

namespace sdpa09 {

template <int DPAD, int BIAS, int SL, bool IMG, bool FAST = false>
static cudaError_t launch_win_one(const BwdMaps& tm, const BwdTcParams& p, int grid, size_t smem,
                                  cudaStream_t stream) {
    auto kern = attn_bwd_win_kernel<DPAD, BIAS, SL, IMG, FAST>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kBwdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tm, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int DPAD, int BIAS, bool IMG>
static cudaError_t launch_win_img(const BwdMaps& tm, const BwdTcParams& p, int grid, size_t smem, cudaStream_t stream) {
    // Swin with bias rows and a shared, non-atomic table-gradient area (slots
    // of at most 64 rows) has an instantiation of its own
    const bool fast = BIAS == kBiasSwin && p.swin_rows && p.swin_acc && !p.swin_acc_atomic;
    switch (p.sl) {
        case 32:
            return fast ? launch_win_one<DPAD, BIAS, 32, IMG, true>(tm, p, grid, smem, stream)
                        : launch_win_one<DPAD, BIAS, 32, IMG>(tm, p, grid, smem, stream);
        case 64:
            return fast ? launch_win_one<DPAD, BIAS, 64, IMG, true>(tm, p, grid, smem, stream)
                        : launch_win_one<DPAD, BIAS, 64, IMG>(tm, p, grid, smem, stream);
        case 128: return launch_win_one<DPAD, BIAS, 128, IMG>(tm, p, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

// the Swin image token layout is a separate instantiation
template <int DPAD, int BIAS>
static cudaError_t launch_win_sl(const BwdMaps& tm, const BwdTcParams& p, int grid, size_t smem, cudaStream_t stream) {
    if constexpr (BIAS == kBiasSwin)
        if (p.swin_image) return launch_win_img<DPAD, BIAS, true>(tm, p, grid, smem, stream);
    return launch_win_img<DPAD, BIAS, false>(tm, p, grid, smem, stream);
}

cudaError_t launch_bwd_win(int dpad, bool swin, const BwdMaps& tm, const BwdTcParams& p, int grid, size_t smem,
                           cudaStream_t stream) {
    switch (dpad) {
        case 32: return swin ? launch_win_sl<32, kBiasSwin>(tm, p, grid, smem, stream)
                             : launch_win_sl<32, kBiasNone>(tm, p, grid, smem, stream);
        case 48: return swin ? launch_win_sl<48, kBiasSwin>(tm, p, grid, smem, stream)
                             : launch_win_sl<48, kBiasNone>(tm, p, grid, smem, stream);
        case 64: return swin ? launch_win_sl<64, kBiasSwin>(tm, p, grid, smem, stream)
                             : launch_win_sl<64, kBiasNone>(tm, p, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdpa09
