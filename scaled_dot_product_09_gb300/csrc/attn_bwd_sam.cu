// attn_bwd_sam.cu -- the SAM decomposed rel-pos gradients of the
// long-sequence backward, on the CUDA cores in fp32 (every product has
// 16-bit inputs or fp32 sums as operands and is accumulated in fp32; nothing
// is rounded to 16 bits before the stored result; the rel terms the two
// tensor-core passes add to their scores come from attn_bwd_sam_rel.cu):
//
//   dQ post-pass:  dQ_q = (scale dS.K)_q + sum_kh dRelH[q][kh] R_h[qh - kh + S - 1]
//                                        + sum_kw dRelW[q][kw] R_w[qw - kw + S - 1];
//   table pass:    dR_h[j] = sum of dRelH[q][kh] Q_q over the (q, kh) with
//                  qh - kh + S - 1 = j, and dR_w[j] alike with qw - kw + S - 1 = j.
//
// (Segment Anything, image encoder: the decomposed relative position terms
// added to the attention logits, and their gradients by the chain rule.)
//
// The grids are square: side S = 14, 48 or 64, tables of 2 S - 1 rows (tables
// of another length are resampled to that first, and their gradients
// resampled back; see the end of this file).  Work is cut in blocks of 64
// query rows of one slice: one grid row when S = 64 (S = 48: one grid row
// padded to 64); four grid rows, each padded from 14 to 16 columns, when
// S = 14 (block row r is grid row bp * LPC + r / QWP, grid column r % QWP;
// padded rows are zero).
// Every product is a small GEMM tiled in registers: a thread keeps an 8 x 4
// (dQ) or 4 x 4 (tables) tile of outputs and reads both operands as float4
// (or four 16-bit values) from shared memory.  For the w terms the index
// j = qw - kw + S - 1 turns the skew into a band that is dense in j: the
// passes spread dRelW[q][kw] to row j of a zero-filled matrix before
// multiplying.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "attn_bwd_sam.cuh"

namespace sdpa09 {

namespace {


template <int S>
struct SamGeom {
    static_assert(S == 14 || S == 48 || S == 64, "SAM backward grids are 14 x 14, 48 x 48 or 64 x 64");
    static constexpr int QWP = S > 16 ? 64 : 16;    // block rows per grid row
    static constexpr int LPC = 64 / QWP;            // grid rows per block
    static constexpr int NBP = (S + LPC - 1) / LPC; // blocks per slice
    static constexpr int NT = 2 * S - 1;            // table rows
    // dQ post-pass: rows j of the spread dRelW matrix
    static constexpr int JW = QWP + S - 1;

    // block row r of block (s, bp): global query row and whether it exists
    __device__ static bool row(int s, int bp, int r, int Nq, int& grow) {
        const int l = r / QWP, qw = r - l * QWP, qh = bp * LPC + l;
        grow = s * Nq + qh * S + qw;
        return qw < S && qh < S;
    }
};

template <bool BF>
__device__ __forceinline__ float4 ld4h(const uint16_t* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    if constexpr (BF) {
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                           __uint_as_float(u.y & 0xffff0000u));
    } else {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
}

template <bool BF>
__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if constexpr (BF) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        } else {
            const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
            f[2 * e] = t.x;
            f[2 * e + 1] = t.y;
        }
    }
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (BF) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

__device__ __forceinline__ void fma8x4(float (&acc)[8][4], const float4 a0, const float4 a1, const float4 b) {
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bb[4] = {b.x, b.y, b.z, b.w};
    // column pairs through the packed FMA (the same rounding per element)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const float2 y = __ffma2_rn(make_float2(a[i], a[i]), make_float2(bb[e], bb[e + 1]),
                                        make_float2(acc[i][e], acc[i][e + 1]));
            acc[i][e] = y.x;
            acc[i][e + 1] = y.y;
        }
}

__device__ __forceinline__ void fma4x4(float (&acc)[4][4], const float4 a, const float4 b) {
    const float aa[4] = {a.x, a.y, a.z, a.w};
    const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const float2 y = __ffma2_rn(make_float2(aa[i], aa[i]), make_float2(bb[e], bb[e + 1]),
                                        make_float2(acc[i][e], acc[i][e + 1]));
            acc[i][e] = y.x;
            acc[i][e + 1] = y.y;
        }
}

// --------------------------------------------------------------- dQ post-pass
// 160 threads: group g of 8 block rows (tid / 20) x group cg of 4 columns of
// d (tid % 20).  Staged per block: dRelH as [kh][block row] and the spread
// dRelW as [j][block row] (row pitch kAP floats), both fp32; the tables as
// 16-bit [terms][j][d] for the CTA's life.
constexpr int kAP = 68;  // pitch: 16-byte rows, and the staging stores below hit distinct banks
constexpr int kDqThreads = 160;

template <int S, bool BF>
__global__ void __launch_bounds__(kDqThreads, S == 64 ? 2 : 4) bwd_sam_dq_kernel(const SamBwdParams p) {
    using G = SamGeom<S>;
    extern __shared__ __align__(16) unsigned char smem[];
    const int d = p.d;
    uint16_t* sT = reinterpret_cast<uint16_t*>(smem);
    float* sAh = reinterpret_cast<float*>(smem + (size_t)2 * G::NT * d * 2);
    float* sAw = sAh + S * kAP;
    const int tid = threadIdx.x, nt = blockDim.x;
    {
        const uint16_t* tab_h = static_cast<const uint16_t*>(p.rel_h);
        const uint16_t* tab_w = static_cast<const uint16_t*>(p.rel_w);
        for (int i = tid; i < G::NT * d; i += nt) {
            sT[i] = tab_h[i];
            sT[G::NT * d + i] = tab_w[i];
        }
    }
    const int g = tid / 20, cg = tid - g * 20;
    const bool act = 4 * cg < d;
    const int r0 = 8 * g, l = r0 / G::QWP, qw0 = r0 - l * G::QWP;
    const size_t rows = (size_t)p.BH * p.Nq;
    const float* drw1 = p.d_relw + rows * S;
    const int nblk = p.BH * G::NBP;
    for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int s = blk / G::NBP, bp = blk - s * G::NBP;
        const int qh = bp * G::LPC + l;
        __syncthreads();  // the previous block is done with sAh and sAw
        for (int i = tid; i < G::JW * kAP / 4; i += nt) reinterpret_cast<float4*>(sAw)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (S == 64) {
            // dRelH rows as float4: a warp takes 16 rows x 2 column groups
            for (int i = tid; i < 64 * 16; i += nt) {
                const int rr = i & 15, kb = (i >> 4) & 1, rest = i >> 5, kp = rest & 7, rb = rest >> 3;
                const int r = 16 * rb + rr, k4 = 2 * kp + kb;
                int grow;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (G::row(s, bp, r, p.Nq, grow)) v = *reinterpret_cast<const float4*>(p.d_relh + (size_t)grow * S + 4 * k4);
                sAh[(4 * k4 + 0) * kAP + r] = v.x;
                sAh[(4 * k4 + 1) * kAP + r] = v.y;
                sAh[(4 * k4 + 2) * kAP + r] = v.z;
                sAh[(4 * k4 + 3) * kAP + r] = v.w;
            }
        } else {
            for (int i = tid; i < 64 * S; i += nt) {
                const int r = i & 63, kh = i >> 6;
                int grow;
                sAh[kh * kAP + r] = G::row(s, bp, r, p.Nq, grow) ? p.d_relh[(size_t)grow * S + kh] : 0.f;
            }
        }
        __syncthreads();
        // dRelW (both halves) spread to row j = qw + S - 1 - kw
        if constexpr (S == 64) {
            for (int i = tid; i < 64 * 16; i += nt) {
                const int rr = i & 15, kb = (i >> 4) & 1, rest = i >> 5, kp = rest & 7, rb = rest >> 3;
                const int r = 16 * rb + rr, k4 = 2 * kp + kb;
                int grow;
                if (G::row(s, bp, r, p.Nq, grow)) {
                    const float4 a = *reinterpret_cast<const float4*>(p.d_relw + (size_t)grow * S + 4 * k4);
                    const float4 b = *reinterpret_cast<const float4*>(drw1 + (size_t)grow * S + 4 * k4);
                    const int j0 = r + S - 1 - 4 * k4;  // qw = r on 64-wide grids
                    sAw[(j0 - 0) * kAP + r] = a.x + b.x;
                    sAw[(j0 - 1) * kAP + r] = a.y + b.y;
                    sAw[(j0 - 2) * kAP + r] = a.z + b.z;
                    sAw[(j0 - 3) * kAP + r] = a.w + b.w;
                }
            }
        } else {
            for (int i = tid; i < 64 * S; i += nt) {
                const int r = i & 63, kw = i >> 6;
                int grow;
                if (G::row(s, bp, r, p.Nq, grow)) {
                    const int qw = r % G::QWP;
                    sAw[(qw + S - 1 - kw) * kAP + r] =
                        p.d_relw[(size_t)grow * S + kw] + drw1[(size_t)grow * S + kw];
                }
            }
        }
        __syncthreads();
        if (!act) continue;
        float acc[8][4];
        bool ok[8];
        int grows[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ok[i] = G::row(s, bp, r0 + i, p.Nq, grows[i]);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ok[i]) v = *reinterpret_cast<const float4*>(p.dq32 + (size_t)grows[i] * d + 4 * cg);
            acc[i][0] = v.x;
            acc[i][1] = v.y;
            acc[i][2] = v.z;
            acc[i][3] = v.w;
        }
        if (qh < S) {
            const uint16_t* th = sT + (size_t)(qh + S - 1) * d + 4 * cg;  // row qh + S - 1 - kh
#pragma unroll 4
            for (int kh = 0; kh < S; ++kh) {
                const float4 a0 = *reinterpret_cast<const float4*>(sAh + kh * kAP + r0);
                const float4 a1 = *reinterpret_cast<const float4*>(sAh + kh * kAP + r0 + 4);
                fma8x4(acc, a0, a1, ld4h<BF>(th - (size_t)kh * d));
            }
            const uint16_t* tw = sT + (size_t)G::NT * d + 4 * cg;
            const int j1 = min(qw0 + 7 + S - 1, G::NT - 1);
#pragma unroll 4
            for (int j = qw0; j <= j1; ++j) {
                const float4 a0 = *reinterpret_cast<const float4*>(sAw + j * kAP + r0);
                const float4 a1 = *reinterpret_cast<const float4*>(sAw + j * kAP + r0 + 4);
                fma8x4(acc, a0, a1, ld4h<BF>(tw + (size_t)j * d));
            }
        }
        uint16_t* dq16 = static_cast<uint16_t*>(p.dq);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (ok[i])
                *reinterpret_cast<uint2*>(dq16 + (size_t)grows[i] * d + 4 * cg) =
                    make_uint2(pack2<BF>(acc[i][0], acc[i][1]), pack2<BF>(acc[i][2], acc[i][3]));
    }
}

// ----------------------------------------------------------------- table pass
// A CTA takes one block position bp (fixed grid rows) and a group of slices,
// and keeps in registers: Y_h[kh][c] = sum dRelH[q][kh] Q_q[c] over the q of
// one grid row (4 x 4 tile; table row qh - kh + S - 1) and, for two j-groups,
// Y_w[j][c] = sum over the block's rows of the spread dRelW[q][j] Q_q[c]
// (table row j).  Threads: warp w = 5 wr + wc, lane = 4 lr + lc; tile row
// group kg = 8 wr + lr (0..15), column group cg = 4 wc + lc (0..19).
// Staged per slice: dRelH as [block row][KHP], the spread dRelW as
// [block row][JWS] (zeros outside each row's band, written once), Q as fp32
// [block row][d].
constexpr int kTabThreads = 320;

template <int S, bool BF>
__global__ void __launch_bounds__(kTabThreads, 2) bwd_sam_dtab_kernel(const SamBwdParams p) {
    using G = SamGeom<S>;
    constexpr int KHP = S > 16 ? 64 : 16;   // dRelH row pitch
    constexpr int JWS = S > 16 ? 128 : 32;  // spread dRelW row pitch (>= QWP + S - 1, multiple of 4)
    constexpr int JG = (G::NT + 3) / 4;      // j-groups of the w table
    static_assert(G::QWP + S - 1 <= JWS && 4 * JG <= JWS, "pitch");
    extern __shared__ __align__(16) unsigned char smem[];
    const int d = p.d;
    float* sAh = reinterpret_cast<float*>(smem);  // [64][KHP]
    float* sAw = sAh + 64 * KHP;                  // [64][JWS]
    float* sQ = sAw + 64 * JWS;                   // [64][d]
    const int tid = threadIdx.x, nt = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int kg = 8 * (warp / 5) + (lane >> 2), cg = 4 * (warp % 5) + (lane & 3);
    const bool act = 4 * cg < d;
    const int bp = blockIdx.x % G::NBP, grp = blockIdx.x / G::NBP;
    const int per = (p.BH + p.groups - 1) / p.groups;
    const int s0 = grp * per, s1 = min(p.BH, s0 + per);
    const size_t rows = (size_t)p.BH * p.Nq;
    const float* drw1 = p.d_relw + rows * S;
    const uint16_t* q16 = static_cast<const uint16_t*>(p.q);
    // h tile: grid row lh of the block, kh group khg
    const int lh = kg / (KHP / 4), khg = kg - lh * (KHP / 4);
    const int qh = bp * G::LPC + lh;
    float yh[4][4], yw[2][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            yh[i][e] = 0.f;
            yw[0][i][e] = 0.f;
            yw[1][i][e] = 0.f;
        }
    for (int i = tid; i < 64 * (KHP + JWS + d); i += nt) sAh[i] = 0.f;
    for (int s = s0; s < s1; ++s) {
        __syncthreads();  // zeros written / the previous slice is done
        for (int i = tid; i < 64 * S; i += nt) {
            const int r = i / S, kk = i - r * S;
            int grow;
            if (G::row(s, bp, r, p.Nq, grow)) {
                const size_t o = (size_t)grow * S + kk;
                sAh[r * KHP + kk] = p.d_relh[o];
                sAw[r * JWS + (r % G::QWP) + S - 1 - kk] = p.d_relw[o] + drw1[o];
            }
        }
        for (int i = tid; i < 64 * (d / 8); i += nt) {
            const int r = i / (d / 8), c8 = i - r * (d / 8);
            int grow;
            if (G::row(s, bp, r, p.Nq, grow)) {
                float f[8];
                unpack8<BF>(*reinterpret_cast<const uint4*>(q16 + (size_t)grow * d + c8 * 8), f);
                float4* dst = reinterpret_cast<float4*>(sQ + r * d + c8 * 8);
                dst[0] = make_float4(f[0], f[1], f[2], f[3]);
                dst[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
        __syncthreads();
        if (!act) continue;
        if (qh < S && 4 * khg < S) {
            const float* a = sAh + lh * G::QWP * KHP + 4 * khg;
            const float* b = sQ + lh * G::QWP * d + 4 * cg;
#pragma unroll 4
            for (int qw = 0; qw < S; ++qw)
                fma4x4(yh, *reinterpret_cast<const float4*>(a + qw * KHP), *reinterpret_cast<const float4*>(b + qw * d));
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int jg = kg + 16 * t;
            if (jg < JG) {
                const int qa = max(0, 4 * jg - S + 1), qb = min(S - 1, 4 * jg + 3);
                for (int ll = 0; ll < G::LPC; ++ll) {
                    const float* a = sAw + ll * G::QWP * JWS + 4 * jg;
                    const float* b = sQ + ll * G::QWP * d + 4 * cg;
#pragma unroll 4
                    for (int qw = qa; qw <= qb; ++qw)
                        fma4x4(yw[t], *reinterpret_cast<const float4*>(a + qw * JWS),
                               *reinterpret_cast<const float4*>(b + qw * d));
                }
            }
        }
    }
    if (!act || s0 >= s1) return;
    float* dRh = p.d_bias;
    float* dRw = p.d_bias + (size_t)G::NT * d;
    if (qh < S) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int kh = 4 * khg + i;
            if (kh < S) {
                float* row = dRh + (size_t)(qh + S - 1 - kh) * d + 4 * cg;
#pragma unroll
                for (int e = 0; e < 4; ++e) atomicAdd(row + e, yh[i][e]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int jg = kg + 16 * t;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = 4 * jg + i;
            if (jg < JG && j < G::NT) {
                float* row = dRw + (size_t)j * d + 4 * cg;
#pragma unroll
                for (int e = 0; e < 4; ++e) atomicAdd(row + e, yw[t][i][e]);
            }
        }
    }
}

// Grid-stride kernels: as many CTAs as fit on the SMs at once, at most one
// per unit of work.
template <typename K>
cudaError_t launch_k(K kern, int work, int threads, size_t smem, int nsm, cudaStream_t st, const SamBwdParams& p) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(work, std::max(1, per_sm) * nsm));
    kern<<<grid, threads, smem, st>>>(p);
    return cudaGetLastError();
}

template <int S, bool BF>
cudaError_t launch_post(const SamBwdParams& p, int nsm, cudaStream_t st) {
    using G = SamGeom<S>;
    const int nblk = p.BH * G::NBP;
    const size_t smem_dq = (size_t)2 * G::NT * p.d * 2 + (size_t)(S + G::JW) * kAP * 4;
    cudaError_t e = launch_k(bwd_sam_dq_kernel<S, BF>, nblk, kDqThreads, smem_dq, nsm, st, p);
    if (e != cudaSuccess) return e;
    constexpr int KHP = S > 16 ? 64 : 16, JWS = S > 16 ? 128 : 32;
    const size_t smem_t = (size_t)64 * (KHP + JWS + p.d) * 4;
    // one CTA per (block position, slice group): the grid is exactly that
    cudaError_t e2 = cudaFuncSetAttribute(bwd_sam_dtab_kernel<S, BF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_t);
    if (e2 != cudaSuccess) return e2;
    bwd_sam_dtab_kernel<S, BF><<<G::NBP * p.groups, kTabThreads, smem_t, st>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------ table pass, 14 x 14 windows
// On the 14-wide grid a slice (196 query rows) is small, so the table pass
// takes whole slices and forms a dense GEMM against a "spread" matrix: with
// j the table row that a (query, key row / column) pair addresses --
// j = qh - kh + 13 for R_h (j in [0, 27)) and 28 + qw - kw + 13 for R_w
// (j in [28, 55)) -- the row sums dRelH, dRelW are spread to A[q][j] (zero
// where no key row / column addresses j) and dR[j] = sum over slices and q
// of A[q][j] Q_q.  (Per-slice versions of the pre-pass and the dQ pass on
// the same plan measured slower than the block-wise ones: 351 vs 209 us and
// 267 vs 200 us on the SAM window workload; this one 192 vs 307 us.)
constexpr int k14 = 14, k14N = 196, k14J = 56, k14W = 28;  // side, rows per slice, stacked tables, R_w offset

// dR[j] += sum_q A[q][j] Q_q over the CTA's slices; 288 threads: 14 table-row
// groups of 4 x 20 column groups of 4; one atomic add per output at the end.
template <bool BF>
__global__ void __launch_bounds__(288, 2) bwd_sam14_dtab_kernel(const SamBwdParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int d = p.d;
    float* sA = reinterpret_cast<float*>(smem);  // [196][56] spread row sums
    float* sQ = sA + k14N * k14J;                // [196][d]
    const int tid = threadIdx.x, nt = blockDim.x;
    const int jg = tid / 20, cg = tid - jg * 20;
    const bool act = jg < k14J / 4 && 4 * cg < d;
    const size_t rows = (size_t)p.BH * p.Nq;
    const float* drw1 = p.d_relw + rows * k14;
    const uint16_t* q16 = static_cast<const uint16_t*>(p.q);
    float y[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) y[i][e] = 0.f;
    bool any = false;
    for (int s = blockIdx.x; s < p.BH; s += gridDim.x) {
        any = true;
        const size_t row0 = (size_t)s * k14N;
        __syncthreads();
        for (int i = tid; i < k14N * k14J / 4; i += nt) reinterpret_cast<float4*>(sA)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = tid; i < k14N * (d / 8); i += nt) {
            const int r = i / (d / 8), c8 = i - r * (d / 8);
            float f[8];
            unpack8<BF>(*reinterpret_cast<const uint4*>(q16 + (row0 + r) * d + c8 * 8), f);
            float4* dst = reinterpret_cast<float4*>(sQ + r * d + c8 * 8);
            dst[0] = make_float4(f[0], f[1], f[2], f[3]);
            dst[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
        __syncthreads();
        for (int i = tid; i < k14N * k14; i += nt) {
            const int q = i / k14, k = i - q * k14, qh = q / k14, qw = q - qh * k14;
            const size_t o = (row0 + q) * k14 + k;
            sA[q * k14J + qh + k14 - 1 - k] = p.d_relh[o];
            sA[q * k14J + k14W + qw + k14 - 1 - k] = p.d_relw[o] + drw1[o];
        }
        __syncthreads();
        if (!act) continue;
        // rows whose spread can reach this thread's table rows: R_h rows need
        // qh in [4jg - 13, 4jg + 3]; R_w rows can be reached from every grid row
        int q0 = 0, q1 = k14N;
        if (4 * jg < 2 * k14 - 1) {
            q0 = k14 * max(0, 4 * jg - (k14 - 1));
            q1 = k14 * min(k14, 4 * jg + 4);
        }
#pragma unroll 4
        for (int q = q0; q < q1; ++q) {
            const float4 a = *reinterpret_cast<const float4*>(sA + q * k14J + 4 * jg);
            const float4 b = *reinterpret_cast<const float4*>(sQ + q * d + 4 * cg);
            fma4x4(y, a, b);
        }
    }
    if (!act || !any) return;
    const int nt_rows = 2 * k14 - 1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = 4 * jg + i;
        float* row = nullptr;
        if (j < nt_rows) row = p.d_bias + (size_t)j * d;
        else if (j >= k14W && j < k14W + nt_rows) row = p.d_bias + (size_t)(nt_rows + j - k14W) * d;
        if (row)
#pragma unroll
            for (int e = 0; e < 4; ++e) atomicAdd(row + 4 * cg + e, y[i][e]);
    }
}

// 14-wide grids: the block-wise dQ pass, then the per-slice table pass
template <bool BF>
cudaError_t launch_post14(const SamBwdParams& p, int nsm, cudaStream_t st) {
    using G = SamGeom<14>;
    const size_t smem_dq = (size_t)2 * G::NT * p.d * 2 + (size_t)(14 + G::JW) * kAP * 4;
    cudaError_t e = launch_k(bwd_sam_dq_kernel<14, BF>, p.BH * G::NBP, kDqThreads, smem_dq, nsm, st, p);
    if (e != cudaSuccess) return e;
    const size_t smem_t = (size_t)k14N * k14J * 4 + (size_t)k14N * p.d * 4;
    return launch_k(bwd_sam14_dtab_kernel<BF>, p.BH, 288, smem_t, nsm, st, p);
}

}  // namespace

int sam_bwd_groups(int S, int BH, int nsm) {
    const int nbp = S == 64 ? SamGeom<64>::NBP : (S == 48 ? SamGeom<48>::NBP : SamGeom<14>::NBP);
    return std::max(1, std::min(BH, 2 * nsm / nbp));
}

cudaError_t launch_bwd_sam_post(const SamBwdParams& p, int S, bool bf, int nsm, cudaStream_t st) {
    if (S == 64) return bf ? launch_post<64, true>(p, nsm, st) : launch_post<64, false>(p, nsm, st);
    if (S == 48) return bf ? launch_post<48, true>(p, nsm, st) : launch_post<48, false>(p, nsm, st);
    if (S == 14) return bf ? launch_post14<true>(p, nsm, st) : launch_post14<false>(p, nsm, st);
    return cudaErrorInvalidValue;
}

// ------------------------------------------------- resampled tables (rel_pos_resized)
// A table of lin rows used at lout = 2 S - 1 rows: row m is the linear
// interpolation, at half-pixel centres clamped to the table, of rows i0(m)
// and i1(m) with weights 1 - w(m) and w(m) -- the forward's resampling,
// rounded to the operand type as there.  The backward runs on the resampled
// rows and returns their fp32 gradients through the transposed map:
// dR[i] += sum over m with i0(m) = i of (1 - w(m)) dR'[m] + sum over m with
// i1(m) = i of w(m) dR'[m].
namespace {

__device__ __forceinline__ void resample_pos(int m, int lin, int lout, int& i0, int& i1, float& w1) {
    const float pos = fmaxf(__fmul_rn((float)lin / (float)lout, (float)m + 0.5f) - 0.5f, 0.f);
    i0 = min((int)pos, lin - 1);
    i1 = min(i0 + 1, lin - 1);
    w1 = pos - (float)i0;
}

// dst [lout][d] 16-bit from src [lin][d]; also clears dz (n floats)
template <bool BF>
__global__ void bwd_sam_resample_kernel(const uint16_t* src, uint16_t* dst, int lin, int lout, int d, float* dz, int n) {
    const int stride = gridDim.x * blockDim.x;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < lout * d; i += stride) {
        const int m = i / d, c = i - m * d;
        int i0, i1;
        float w1;
        resample_pos(m, lin, lout, i0, i1, w1);
        const uint16_t a = src[(size_t)i0 * d + c], b = src[(size_t)i1 * d + c];
        const float fa = BF ? __bfloat162float(__ushort_as_bfloat16(a)) : __half2float(__ushort_as_half(a));
        const float fb = BF ? __bfloat162float(__ushort_as_bfloat16(b)) : __half2float(__ushort_as_half(b));
        const float v = (1.f - w1) * fa + w1 * fb;
        dst[i] = BF ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dz[i] = 0.f;
}

// dR [lin][d] += the transposed resampling of dRr [lout][d]
__global__ void bwd_sam_unresample_kernel(const float* dRr, float* dR, int lin, int lout, int d) {
    const int stride = gridDim.x * blockDim.x;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < lin * d; i += stride) {
        const int r = i / d, c = i - r * d;
        float acc = 0.f;
        for (int m = 0; m < lout; ++m) {
            int i0, i1;
            float w1;
            resample_pos(m, lin, lout, i0, i1, w1);
            if (i0 == r) acc += (1.f - w1) * dRr[(size_t)m * d + c];
            if (i1 == r) acc += w1 * dRr[(size_t)m * d + c];
        }
        dR[i] += acc;
    }
}

}  // namespace

cudaError_t launch_bwd_sam_resample(const void* src, void* dst, int lin, int lout, int d, bool bf, float* dz, int n,
                                    cudaStream_t st) {
    const int work = std::max(lout * d, n);
    const int blocks = std::max(1, std::min((work + 255) / 256, 1024));
    if (bf)
        bwd_sam_resample_kernel<true><<<blocks, 256, 0, st>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst),
                                                              lin, lout, d, dz, n);
    else
        bwd_sam_resample_kernel<false><<<blocks, 256, 0, st>>>(static_cast<const uint16_t*>(src),
                                                               static_cast<uint16_t*>(dst), lin, lout, d, dz, n);
    return cudaGetLastError();
}

cudaError_t launch_bwd_sam_unresample(const float* dRr, float* dR, int lin, int lout, int d, cudaStream_t st) {
    const int blocks = std::max(1, std::min((lin * d + 255) / 256, 1024));
    bwd_sam_unresample_kernel<<<blocks, 256, 0, st>>>(dRr, dR, lin, lout, d);
    return cudaGetLastError();
}

}  // namespace sdpa09
