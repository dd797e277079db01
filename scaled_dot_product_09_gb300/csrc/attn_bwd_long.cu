// The long-sequence backward: its pre-pass (D = rowsum(dO * O)) and the two
// tensor-core passes (attn_bwd_long.cuh) for head dims padded to 32, 48, 64
// and 80.  The SAM rel-pos parts are in attn_bwd_sam.cu.
#include <cuda_runtime.h>
#include "attn_bwd_long.cuh"

namespace sdpa09 {

// D = rowsum(dO * O) in fp32, one thread per query row.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdPrepParams p) {
    const bool bf = p.is_bf16 != 0;
    for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < p.rows; row += gridDim.x * blockDim.x) {
        const size_t base = (size_t)row * p.d;
        float D = 0.f;
        for (int c = 0; c < p.d; c += 8) {
            const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + base + c);
            const uint4 b = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + base + c);
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 x, y;
                if (bf) {
                    x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
                    y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
                } else {
                    x = __half22float2(*reinterpret_cast<const __half2*>(&wa[e]));
                    y = __half22float2(*reinterpret_cast<const __half2*>(&wb[e]));
                }
                D = fmaf(x.x, y.x, fmaf(x.y, y.y, D));
            }
        }
        p.Dws[row] = D;
    }
}

cudaError_t launch_bwd_prep(const BwdPrepParams& p, int nsm, cudaStream_t stream) {
    const int blocks = std::max(1, std::min((p.rows + 255) / 256, nsm * 8));
    bwd_prep_kernel<<<blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int DPAD, int BIAS, int MODE, int SW>
static cudaError_t launch_long_one(const BwdMaps& tm, const BwdLongParams& p, int grid, size_t smem,
                                   cudaStream_t stream) {
    auto kern = attn_bwd_long_kernel<DPAD, BIAS, MODE, SW>;
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

template <int DPAD>
static cudaError_t launch_long_d(int mode, int sw, const BwdMaps& tm, const BwdLongParams& p, int grid, size_t smem,
                                 cudaStream_t st) {
    if (sw == 0)
        return mode == kBwdKeyPass ? launch_long_one<DPAD, kBiasNone, kBwdKeyPass, 0>(tm, p, grid, smem, st)
                                   : launch_long_one<DPAD, kBiasNone, kBwdQueryPass, 0>(tm, p, grid, smem, st);
    if constexpr (DPAD == 80 || DPAD == 64) {
        if (sw == 64)
            return mode == kBwdKeyPass ? launch_long_one<DPAD, kBiasSam, kBwdKeyPass, 64>(tm, p, grid, smem, st)
                                       : launch_long_one<DPAD, kBiasSam, kBwdQueryPass, 64>(tm, p, grid, smem, st);
        if (sw == 14)
            return mode == kBwdKeyPass ? launch_long_one<DPAD, kBiasSam, kBwdKeyPass, 14>(tm, p, grid, smem, st)
                                       : launch_long_one<DPAD, kBiasSam, kBwdQueryPass, 14>(tm, p, grid, smem, st);
        if (sw == 48)
            return mode == kBwdKeyPass ? launch_long_one<DPAD, kBiasSam, kBwdKeyPass, 48>(tm, p, grid, smem, st)
                                       : launch_long_one<DPAD, kBiasSam, kBwdQueryPass, 48>(tm, p, grid, smem, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_long(int dpad, int mode, int sw, const BwdMaps& tm, const BwdLongParams& p, int grid,
                            size_t smem, cudaStream_t stream) {
    switch (dpad) {
        case 32: return launch_long_d<32>(mode, sw, tm, p, grid, smem, stream);
        case 48: return launch_long_d<48>(mode, sw, tm, p, grid, smem, stream);
        case 64: return launch_long_d<64>(mode, sw, tm, p, grid, smem, stream);
        case 80: return launch_long_d<80>(mode, sw, tm, p, grid, smem, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdpa09
