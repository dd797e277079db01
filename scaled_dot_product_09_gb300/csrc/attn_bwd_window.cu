// attn_bwd_window.cu -- backward pass of the attention forward for short
// sequences (windows: Nq, Nk <= 128, d <= 64), for Swin training ("视觉大模型
// 训练和推理加速" section 二 builds the forward and the backward computation
// of its custom window operators alike).
//
// One CTA handles one (window, head) slice at a time, with every operand of
// the slice in shared memory: S = scale Q.K^T + bias, P = softmax(S) exactly
// (row max and sum over the slice's keys), then
//   dV = P^T dO,  D_i = dO_i . O_i,  dS = P * (dO V^T - D),
//   dQ = scale dS K,  dK = scale dS^T Q,
// and, for the Swin bias, the table gradient: each (query, key) pair of head
// h adds dS to table row idx(i, j) (the shifted-window mask is constant).
// The table gradient is summed per CTA in shared memory and added to the
// caller's fp32 buffer once per CTA.  Products are fp32 on the CUDA cores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_bwd_window.cuh"

namespace sdpa09 {

namespace {

constexpr int kBwdThreads = 256;

__device__ __forceinline__ uint16_t st16(float v, bool bf) {
    return bf ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

// Eight consecutive 16-bit values (16-byte aligned) as floats.
__device__ __forceinline__ void ld8(const uint16_t* p, bool bf, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if (bf) {  // a bfloat16 is the high half of a float
            f[2 * t] = __uint_as_float(w[t] << 16);
            f[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
        } else {
            const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
            f[2 * t] = x.x;
            f[2 * t + 1] = x.y;
        }
    }
}

// Dot product of two rows of d 16-bit values (d % 8 == 0).
__device__ __forceinline__ float dot_rows(const uint16_t* a, const uint16_t* b, int d, bool bf) {
    float acc = 0.f;
    for (int c = 0; c < d; c += 8) {
        float x[8], y[8];
        ld8(a + c, bf, x);
        ld8(b + c, bf, y);
#pragma unroll
        for (int t = 0; t < 8; ++t) acc = fmaf(x[t], y[t], acc);
    }
    return acc;
}

// Eight floats, scaled, rounded to 16 bits and stored as one 16-byte word.
__device__ __forceinline__ void st8(uint16_t* p, const float (&a)[8], float scale, bool bf) {
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
        w[t] = (uint32_t)st16(a[2 * t] * scale, bf) | ((uint32_t)st16(a[2 * t + 1] * scale, bf) << 16);
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Region of a coordinate along one axis of the shifted map: 0 inside, 1 in
// the strip the cyclic shift brought from the far edge's window, 2 past it.
__device__ __forceinline__ int bwd_strip(int pos, int G, int M, int s) {
    return pos < G - M ? 0 : (pos < G - s ? 1 : 2);
}

__global__ void __launch_bounds__(kBwdThreads)
    attn_bwd_window_kernel(const BwdParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int Nq = p.Nq, Nk = p.Nk, d = p.d;
    const int ld = Nk + 1;  // padded row of the score matrix
    uint16_t* sQ = reinterpret_cast<uint16_t*>(smem);
    uint16_t* sK = sQ + Nq * d;
    uint16_t* sV = sK + Nk * d;
    uint16_t* sO = sV + Nk * d;
    uint16_t* sdO = sO + Nq * d;
    float* sP = reinterpret_cast<float*>(sdO + Nq * d);  // [Nq][ld]: S, then P, then dS
    float* sD = sP + Nq * ld;                            // [Nq]
    float* sTab = sD + Nq;                               // Swin table gradient [T][H], T = (2M-1)^2
    const bool bf = p.is_bf16 != 0;
    const int tid = threadIdx.x;
    const int M = p.win, T = (2 * M - 1) * (2 * M - 1);
    const int n_tab = p.swin ? T * p.H : 0;
    for (int e = tid; e < n_tab; e += kBwdThreads) sTab[e] = 0.f;

    for (int slice = blockIdx.x; slice < p.BH; slice += gridDim.x) {
        const int h = slice % p.H;
        __syncthreads();  // the previous slice's reads of shared memory are done
        // ---- operands of the slice (rows of d 16-bit values, d % 8 == 0)
        {
            const int cq = Nq * d / 8, ck = Nk * d / 8;
            const uint4* gq = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + (size_t)slice * Nq * d);
            const uint4* go = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + (size_t)slice * Nq * d);
            const uint4* gdo = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + (size_t)slice * Nq * d);
            const uint4* gk = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k) + (size_t)slice * Nk * d);
            const uint4* gv = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v) + (size_t)slice * Nk * d);
            for (int e = tid; e < cq; e += kBwdThreads) {
                reinterpret_cast<uint4*>(sQ)[e] = gq[e];
                reinterpret_cast<uint4*>(sO)[e] = go[e];
                reinterpret_cast<uint4*>(sdO)[e] = gdo[e];
            }
            for (int e = tid; e < ck; e += kBwdThreads) {
                reinterpret_cast<uint4*>(sK)[e] = gk[e];
                reinterpret_cast<uint4*>(sV)[e] = gv[e];
            }
        }
        // the slice's window and its origin in the shifted map (Swin)
        int wr = 0, wc = 0;
        if (p.swin) {
            const int w = (slice / p.H) % p.n_w;
            wr = w / p.n_ww;
            wc = w - wr * p.n_ww;
        }
        __syncthreads();
        // ---- S = scale Q.K^T + bias
        for (int e = tid; e < Nq * Nk; e += kBwdThreads) {
            const int i = e / Nk, j = e - (e / Nk) * Nk;
            float s = dot_rows(sQ + i * d, sK + j * d, d, bf) * p.scale;
            if (p.swin) {
                const int ri = i / M, ci = i - ri * M, rj = j / M, cj = j - rj * M;
                const int idx = (ri - rj + M - 1) * (2 * M - 1) + (ci - cj + M - 1);
                s += p.table[(size_t)idx * p.H + h];
                if (p.shift > 0) {
                    const int yi = wr * M + ri, xi = wc * M + ci, yj = wr * M + rj, xj = wc * M + cj;
                    if (bwd_strip(yi, p.grid_h, M, p.shift) != bwd_strip(yj, p.grid_h, M, p.shift) ||
                        bwd_strip(xi, p.grid_w, M, p.shift) != bwd_strip(xj, p.grid_w, M, p.shift))
                        s -= 100.f;
                }
            }
            sP[i * ld + j] = s;
        }
        __syncthreads();
        // ---- P = softmax over the row's keys (one warp per row)
        {
            const int warp = tid >> 5, lane = tid & 31;
            for (int i = warp; i < Nq; i += kBwdThreads / 32) {
                float m = -INFINITY;
                for (int j = lane; j < Nk; j += 32) m = fmaxf(m, sP[i * ld + j]);
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                float sum = 0.f;
                for (int j = lane; j < Nk; j += 32) {
                    const float ex = expf(sP[i * ld + j] - m);
                    sP[i * ld + j] = ex;
                    sum += ex;
                }
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                const float inv = 1.f / sum;
                for (int j = lane; j < Nk; j += 32) sP[i * ld + j] *= inv;
            }
        }
        // ---- D_i = dO_i . O_i
        for (int i = tid; i < Nq; i += kBwdThreads) sD[i] = dot_rows(sdO + i * d, sO + i * d, d, bf);
        __syncthreads();
        // ---- dV = P^T dO (each thread: eight adjacent columns of one row)
        const int d8 = d / 8;
        {
            uint16_t* gdv = static_cast<uint16_t*>(p.dv) + (size_t)slice * Nk * d;
            for (int e = tid; e < Nk * d8; e += kBwdThreads) {
                const int j = e / d8, c = (e - (e / d8) * d8) * 8;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int i = 0; i < Nq; ++i) {
                    const float pij = sP[i * ld + j];
                    float x[8];
                    ld8(sdO + i * d + c, bf, x);
#pragma unroll
                    for (int t = 0; t < 8; ++t) acc[t] = fmaf(pij, x[t], acc[t]);
                }
                st8(gdv + j * d + c, acc, 1.f, bf);
            }
        }
        __syncthreads();  // P is read by dV before it becomes dS
        // ---- dS = P * (dO V^T - D), in place
        for (int e = tid; e < Nq * Nk; e += kBwdThreads) {
            const int i = e / Nk, j = e - (e / Nk) * Nk;
            const float ds = sP[i * ld + j] * (dot_rows(sdO + i * d, sV + j * d, d, bf) - sD[i]);
            sP[i * ld + j] = ds;
            if (p.swin) {
                const int ri = i / M, ci = i - ri * M, rj = j / M, cj = j - rj * M;
                const int idx = (ri - rj + M - 1) * (2 * M - 1) + (ci - cj + M - 1);
                atomicAdd(&sTab[idx * p.H + h], ds);
            }
        }
        __syncthreads();
        // ---- dQ = scale dS K,  dK = scale dS^T Q
        {
            uint16_t* gdq = static_cast<uint16_t*>(p.dq) + (size_t)slice * Nq * d;
            for (int e = tid; e < Nq * d8; e += kBwdThreads) {
                const int i = e / d8, c = (e - (e / d8) * d8) * 8;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int j = 0; j < Nk; ++j) {
                    const float sij = sP[i * ld + j];
                    float x[8];
                    ld8(sK + j * d + c, bf, x);
#pragma unroll
                    for (int t = 0; t < 8; ++t) acc[t] = fmaf(sij, x[t], acc[t]);
                }
                st8(gdq + i * d + c, acc, p.scale, bf);
            }
            uint16_t* gdk = static_cast<uint16_t*>(p.dk) + (size_t)slice * Nk * d;
            for (int e = tid; e < Nk * d8; e += kBwdThreads) {
                const int j = e / d8, c = (e - (e / d8) * d8) * 8;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int i = 0; i < Nq; ++i) {
                    const float sij = sP[i * ld + j];
                    float x[8];
                    ld8(sQ + i * d + c, bf, x);
#pragma unroll
                    for (int t = 0; t < 8; ++t) acc[t] = fmaf(sij, x[t], acc[t]);
                }
                st8(gdk + j * d + c, acc, p.scale, bf);
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < n_tab; e += kBwdThreads)
        if (sTab[e] != 0.f) atomicAdd(p.d_table + e, sTab[e]);
}

}  // namespace

size_t bwd_window_smem_bytes(int Nq, int Nk, int d, int win, int H, bool swin) {
    const size_t ops = (size_t)(3 * Nq + 2 * Nk) * d * 2;
    const size_t tab = swin ? (size_t)(2 * win - 1) * (2 * win - 1) * H * 4 : 0;
    return ops + (size_t)Nq * (Nk + 1) * 4 + (size_t)Nq * 4 + tab;
}

cudaError_t launch_bwd_window(const BwdParams& p, int grid, size_t smem, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attn_bwd_window_kernel<<<grid, kBwdThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sdpa09
