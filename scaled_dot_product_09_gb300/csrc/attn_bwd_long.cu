// The long-sequence backward: its pre-pass (D = rowsum(dO * O), and for SAM
// the rel-pos terms of every query row), the two tensor-core passes
// (attn_bwd_long.cuh) for head dims padded to 32, 48, 64 and 80, and the SAM
// post-pass (rel-pos gradients into dQ and the tables).
#include <cuda_runtime.h>
#include "attn_bwd_long.cuh"

namespace sdpa09 {

struct BwdPrepParams {
    const void *q, *o, *dout;  // [BH][Nq][d] 16-bit
    float* Dws;                // [BH][Nq]
    int rows, Nq, d, is_bf16;
    // SAM (square grids, tables of length 2 S - 1): rel terms in log2 units
    const void *rel_h, *rel_w;  // [2 S_h - 1][d], [2 S_w - 1][d]
    __half* rel;                // [rows][rel_stride]: rel_h at 0, rel_w at rw0
    float* d_relh;              // [rows][k_h], zeroed here
    float* d_relw;              // [rows][k_w], zeroed here
    int s_h, s_w, rel_stride, rw0;
};

__device__ __forceinline__ float ld16(const void* base, size_t i, bool bf) {
    const uint16_t u = static_cast<const uint16_t*>(base)[i];
    return bf ? __bfloat162float(__ushort_as_bfloat16(u)) : __half2float(__ushort_as_half(u));
}

// One thread per query row.  The SAM tables are staged in shared memory as
// fp32 rows padded to an odd stride (d + 1 words: rows read by the lanes of a
// warp fall in different banks).
template <bool SAM>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdPrepParams p) {
    extern __shared__ float sR[];  // SAM: R_h rows then R_w rows, stride d + 1
    const bool bf = p.is_bf16 != 0;
    const int ld = p.d + 1;
    const int nrh = 2 * p.s_h - 1, nrw = 2 * p.s_w - 1;
    if constexpr (SAM) {
        for (int i = threadIdx.x; i < (nrh + nrw) * p.d; i += blockDim.x) {
            const int rr = i / p.d, c = i - rr * p.d;
            sR[rr * ld + c] = rr < nrh ? ld16(p.rel_h, (size_t)rr * p.d + c, bf) : ld16(p.rel_w, (size_t)(rr - nrh) * p.d + c, bf);
        }
        __syncthreads();
    }
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
        if constexpr (SAM) {
            // rel_h[kh] = Q . R_h[qh - kh + S_h - 1], rel_w[kw] = Q . R_w[qw - kw + S_w - 1]
            const int tok = row % p.Nq, qh = tok / p.s_w, qw = tok - qh * p.s_w;
            float qv[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) qv[c] = c < p.d ? ld16(p.q, base + c, bf) : 0.f;
            __half* out = p.rel + (size_t)row * p.rel_stride;
            for (int t = 0; t < p.rel_stride; ++t) {
                float a = 0.f;
                const float* rr = nullptr;
                if (t < p.s_h) rr = sR + (qh - t + p.s_h - 1) * ld;
                else if (t >= p.rw0 && t < p.rw0 + p.s_w) rr = sR + (nrh + qw - (t - p.rw0) + p.s_w - 1) * ld;
                if (rr) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c < p.d) a = fmaf(qv[c], rr[c], a);
                }
                out[t] = __float2half_rn(a * kLog2e);
            }
            float* dh = p.d_relh + (size_t)row * p.s_h;
            for (int t = 0; t < p.s_h; ++t) dh[t] = 0.f;
            float* dw = p.d_relw + (size_t)row * p.s_w;
            for (int t = 0; t < p.s_w; ++t) dw[t] = 0.f;
        }
    }
}

cudaError_t launch_bwd_prep(const BwdPrepParams& p, bool sam, int nsm, cudaStream_t stream) {
    const int blocks = std::max(1, std::min((p.rows + 255) / 256, nsm * 8));
    if (sam) {
        const size_t smem = (size_t)(2 * p.s_h - 1 + 2 * p.s_w - 1) * (p.d + 1) * 4;
        cudaError_t e = cudaFuncSetAttribute(bwd_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        bwd_prep_kernel<true><<<blocks, 256, smem, stream>>>(p);
    } else {
        bwd_prep_kernel<false><<<blocks, 256, 0, stream>>>(p);
    }
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

namespace sdpa09 {

// ------------------------------------------------------- SAM post-pass
// With rel_h[q][kh] = Q_q . R_h[qh - kh + S - 1] (and rel_w alike), the
// gradients of those terms are dRelH / dRelW (the sums of dS the query pass
// left): dQ_q gets sum_kh dRelH[q][kh] R_h[qh - kh + S - 1] + the same over
// kw, and table row r gets sum of dRelH[q][kh] Q_q over the (q, kh) that
// address it.  Square grids of side S, tables of length 2 S - 1.
struct BwdSamPostParams {
    const float* dq32;   // [rows][d] scale dS.K
    const float* d_relh; // [rows][S]
    const float* d_relw; // [rows][S]
    const void *q, *rel_h, *rel_w;  // 16-bit
    void* dq;            // 16-bit output [rows][d]
    float* d_bias;       // [2S-1][d] for R_h, then [2S-1][d] for R_w; added to
    int rows, Nq, d, S, BH, groups, is_bf16;
};

// dQ: one thread per query row; the tables in shared memory as fp32 rows of
// odd stride d + 1.
__global__ void __launch_bounds__(256) bwd_sam_dq_kernel(const BwdSamPostParams p) {
    extern __shared__ float sR[];
    const bool bf = p.is_bf16 != 0;
    const int ld = p.d + 1, L = 2 * p.S - 1;
    for (int i = threadIdx.x; i < 2 * L * p.d; i += blockDim.x) {
        const int rr = i / p.d, c = i - rr * p.d;
        sR[rr * ld + c] = rr < L ? ld16(p.rel_h, (size_t)rr * p.d + c, bf) : ld16(p.rel_w, (size_t)(rr - L) * p.d + c, bf);
    }
    __syncthreads();
    for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < p.rows; row += gridDim.x * blockDim.x) {
        const int tok = row % p.Nq, qh = tok / p.S, qw = tok - qh * p.S;
        float acc[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) acc[c] = c < p.d ? p.dq32[(size_t)row * p.d + c] : 0.f;
        const float* gh = p.d_relh + (size_t)row * p.S;
        const float* gw = p.d_relw + (size_t)row * p.S;
        for (int kk = 0; kk < p.S; ++kk) {
            const float wh = gh[kk], ww = gw[kk];
            const float* rh = sR + (qh - kk + p.S - 1) * ld;
            const float* rw = sR + (L + qw - kk + p.S - 1) * ld;
#pragma unroll
            for (int c = 0; c < 128; ++c)
                if (c < p.d) acc[c] = fmaf(wh, rh[c], fmaf(ww, rw[c], acc[c]));
        }
        uint16_t* dst = static_cast<uint16_t*>(p.dq) + (size_t)row * p.d;
#pragma unroll
        for (int c = 0; c < 128; ++c)
            if (c < p.d) dst[c] = to_half_bits(acc[c], bf);
    }
}

// Table gradients: a CTA takes one grid line (blockIdx.y: grid row l for
// R_h when blockIdx.z == 0, grid column l for R_w when 1) and a group of
// slices; over the line's S query rows t it forms Y[kk][c] = sum_t
// dRel[q_t][kk] Q[q_t][c] for each slice of the group, and adds Y[kk] to
// table row l - kk + S - 1 once at the end.
__global__ void __launch_bounds__(256) bwd_sam_dtab_kernel(const BwdSamPostParams p) {
    extern __shared__ float sm[];
    const bool bf = p.is_bf16 != 0;
    const int S = p.S, line = blockIdx.y, axis = blockIdx.z;
    float* sA = sm;           // [S rows t][S kk]
    float* sB = sm + S * S;   // [S rows t][d]
    const int nout = S * p.d;
    constexpr int kMaxOut = 24;  // outputs per thread (S * d <= 256 * 24)
    float y[kMaxOut];
#pragma unroll
    for (int j = 0; j < kMaxOut; ++j) y[j] = 0.f;
    const int per = (p.BH + p.groups - 1) / p.groups;
    const int s0 = blockIdx.x * per, s1 = min(p.BH, s0 + per);
    for (int sl = s0; sl < s1; ++sl) {
        __syncthreads();
        for (int i = threadIdx.x; i < S * S; i += blockDim.x) {
            const int t = i / S, kk = i - t * S;
            const int tok = axis == 0 ? line * S + t : t * S + line;
            sA[i] = (axis == 0 ? p.d_relh : p.d_relw)[((size_t)sl * p.Nq + tok) * S + kk];
        }
        for (int i = threadIdx.x; i < S * p.d; i += blockDim.x) {
            const int t = i / p.d, c = i - t * p.d;
            const int tok = axis == 0 ? line * S + t : t * S + line;
            sB[i] = ld16(p.q, ((size_t)sl * p.Nq + tok) * p.d + c, bf);
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kMaxOut; ++j) {
            const int o = threadIdx.x + j * 256;
            if (o < nout) {
                const int kk = o / p.d, c = o - kk * p.d;
                float a = y[j];
                for (int t = 0; t < S; ++t) a = fmaf(sA[t * S + kk], sB[t * p.d + c], a);
                y[j] = a;
            }
        }
    }
    float* tab = p.d_bias + (size_t)axis * (2 * S - 1) * p.d;
#pragma unroll
    for (int j = 0; j < kMaxOut; ++j) {
        const int o = threadIdx.x + j * 256;
        if (o < nout && s0 < s1) {
            const int kk = o / p.d, c = o - kk * p.d;
            atomicAdd(&tab[(size_t)(line - kk + S - 1) * p.d + c], y[j]);
        }
    }
}

cudaError_t launch_bwd_sam_post(const BwdSamPostParams& p, int nsm, cudaStream_t stream) {
    const int L = 2 * p.S - 1;
    const size_t smem_dq = (size_t)2 * L * (p.d + 1) * 4;
    cudaError_t e = cudaFuncSetAttribute(bwd_sam_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dq);
    if (e != cudaSuccess) return e;
    const int blocks = std::max(1, std::min((p.rows + 255) / 256, nsm * 8));
    bwd_sam_dq_kernel<<<blocks, 256, smem_dq, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_t = (size_t)(p.S * p.S + p.S * p.d) * 4;
    e = cudaFuncSetAttribute(bwd_sam_dtab_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_t);
    if (e != cudaSuccess) return e;
    bwd_sam_dtab_kernel<<<dim3((unsigned)p.groups, (unsigned)p.S, 2), 256, smem_t, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sdpa09
