// attn_launch.cuh -- launchers of the attention kernel instantiations.  Each
// attn_d<DPAD>_<bias>.cu translation unit instantiates one (head-dim block,
// bias kind) pair so the build compiles them in parallel.
#pragma once
#include <cuda_runtime.h>
#include "attn_fwd_kernel.cuh"

namespace sdpa09 {

struct LaunchArgs {
    const TmaMaps* tm;
    const AttnParams* p;
    int mode;   // kModeShared / kModeSeparate
    int sw;     // SAM grid-width specialisation, or the Swin window token count (0 = generic)
    int sl;     // slot rows in separate mode (32, 64, 128)
    bool dbg;
    int grid;
    size_t smem;
    cudaStream_t stream;
    const VarlenTable* vt;  // variable-length batch table, or null
};

template <int DPAD, int BIAS, int MODE, int SW, int SL, bool DBG, bool VL = false, bool IMG = false, bool SWR = false,
          bool NS = false>
cudaError_t launch_one(const LaunchArgs& a) {
    auto kern = attn_fwd_kernel<DPAD, BIAS, MODE, SW, SL, DBG, VL, IMG, SWR, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)a.smem);
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the CTAs may become resident while the
    // previous kernel on the stream drains; the kernel waits for it
    // (griddepcontrol.wait) before touching global memory.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.grid);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = a.smem;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    VarlenArg<VL> vt{};
    if constexpr (VL) static_cast<VarlenTable&>(vt) = *a.vt;
    e = cudaLaunchKernelEx(&cfg, kern, *a.tm, *a.p, vt);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int DPAD, int BIAS, int MODE, int SW, int SL, bool IMG = false, bool SWR = false>
cudaError_t launch_dbg(const LaunchArgs& a) {
    return a.dbg ? launch_one<DPAD, BIAS, MODE, SW, SL, true, false, IMG, SWR>(a)
                 : launch_one<DPAD, BIAS, MODE, SW, SL, false, false, IMG, SWR>(a);
}

// Defined in the per-(DPAD, bias) translation units.
template <int DPAD, int BIAS>
cudaError_t launch_attn(const LaunchArgs& a);

// The packed (separate) tiling keeps three tiles per ring stage; it is built
// for head dims up to 64 only.
// Shared tiling without bias: a scale <= 0 (scaled before the max) is an
// instantiation of its own
template <int DPAD, int SW>
cudaError_t launch_none_shared(const LaunchArgs& a) {
    const bool ns = !(a.p->scale_log2 > 0.f);
    if (a.dbg)
        return ns ? launch_one<DPAD, kBiasNone, kModeShared, SW, 0, true, false, false, false, true>(a)
                  : launch_one<DPAD, kBiasNone, kModeShared, SW, 0, true>(a);
    return ns ? launch_one<DPAD, kBiasNone, kModeShared, SW, 0, false, false, false, false, true>(a)
              : launch_one<DPAD, kBiasNone, kModeShared, SW, 0, false>(a);
}

template <int DPAD>
cudaError_t launch_attn_none(const LaunchArgs& a) {
    if (a.vt) {
        if (a.sw != 0 || a.dbg) return cudaErrorInvalidValue;
        if (a.mode == kModeSeparate) {
            // short sequences packed SL rows per slice
            if constexpr (DPAD <= 64) {
                if (a.sl == 32) return launch_one<DPAD, kBiasNone, kModeSeparate, 0, 32, false, true>(a);
                if (a.sl == 64) return launch_one<DPAD, kBiasNone, kModeSeparate, 0, 64, false, true>(a);
            }
            return cudaErrorInvalidValue;
        }
        return !(a.p->scale_log2 > 0.f) ? launch_one<DPAD, kBiasNone, kModeShared, 0, 0, false, true, false, false, true>(a)
                                        : launch_one<DPAD, kBiasNone, kModeShared, 0, 0, false, true>(a);
    }
    if (a.mode == kModeShared) {
        if constexpr (DPAD <= 64)
            if (a.sw == 80) return launch_none_shared<DPAD, 80>(a);
        return launch_none_shared<DPAD, 0>(a);
    }
    if constexpr (DPAD <= 64) {
        if (a.sl == 32) return launch_dbg<DPAD, kBiasNone, kModeSeparate, 0, 32>(a);
        if (a.sl == 64) return launch_dbg<DPAD, kBiasNone, kModeSeparate, 0, 64>(a);
    }
    return cudaErrorInvalidValue;
}

// packed Swin with slots of 32 or 64 rows (64: also the 49-key softmax)
template <int DPAD, bool IMG, bool SWR>
cudaError_t launch_swin_sl(const LaunchArgs& a) {
    if (a.sl == 32) return launch_dbg<DPAD, kBiasSwin, kModeSeparate, 0, 32, IMG, SWR>(a);
    if (a.sl == 64 && a.sw == 49) return launch_dbg<DPAD, kBiasSwin, kModeSeparate, 49, 64, IMG, SWR>(a);
    if (a.sl == 64) return launch_dbg<DPAD, kBiasSwin, kModeSeparate, 0, 64, IMG, SWR>(a);
    return cudaErrorInvalidValue;
}

template <int DPAD>
cudaError_t launch_attn_swin(const LaunchArgs& a) {
    if constexpr (DPAD <= 64) {
        // the windows and the image token layout, and the bias rows and the
        // bias MMAs (slots of 128 rows take the MMAs only), are separate
        // instantiations
        if (a.mode == kModeSeparate) {
            if (a.sl == 128) {
                if (a.p->swin_rows) return cudaErrorInvalidValue;
                return a.p->swin_image ? launch_dbg<DPAD, kBiasSwin, kModeSeparate, 0, 128, true>(a)
                                       : launch_dbg<DPAD, kBiasSwin, kModeSeparate, 0, 128, false>(a);
            }
            if (a.p->swin_image)
                return a.p->swin_rows ? launch_swin_sl<DPAD, true, true>(a) : launch_swin_sl<DPAD, true, false>(a);
            return a.p->swin_rows ? launch_swin_sl<DPAD, false, true>(a) : launch_swin_sl<DPAD, false, false>(a);
        }
    }
    return cudaErrorInvalidValue;
}

template <int DPAD>
cudaError_t launch_attn_sam(const LaunchArgs& a) {
    if (a.mode != kModeShared) return cudaErrorInvalidValue;
    switch (a.sw) {
        case 64: return launch_dbg<DPAD, kBiasSam, kModeShared, 64, 0>(a);
        case 48: return launch_dbg<DPAD, kBiasSam, kModeShared, 48, 0>(a);
        case 14: return launch_dbg<DPAD, kBiasSam, kModeShared, 14, 0>(a);
        default: return launch_dbg<DPAD, kBiasSam, kModeShared, 0, 0>(a);
    }
}

#define SDPA09_INSTANTIATE(DPAD, BIAS, FN) \
    template <>                            \
    cudaError_t launch_attn<DPAD, BIAS>(const LaunchArgs& a) { return FN<DPAD>(a); }

}  // namespace sdpa09
