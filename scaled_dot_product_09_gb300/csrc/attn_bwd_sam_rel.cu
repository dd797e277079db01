// attn_bwd_sam_rel.cu -- the rel pre-pass of the SAM backward on the tensor
// cores:
//
//   rel_h[q][kh] = Q_q . R_h[qh - kh + S - 1],  rel_w[q][kw] = Q_q . R_w[qw - kw + S - 1]
//
// (Segment Anything, image encoder: the decomposed relative position terms
// added to the attention logits), in log2 units, stored fp16 per query row
// for the two tensor-core passes to add to their scores.  The forward forms
// the same terms at the start of each job (G = Q.R^T by MMA, then a barrel
// shift of each row); this kernel does the same for the backward, one block
// of 128 consecutive query rows at a time:
//
//   G_w = Q_blk . R_w^T and G_h = Q_blk . R_h^T by tcgen05 (M = 128, N = the
//   table rows padded to 16, K = d) into tensor memory; thread r reads row r
//   of both, shifts them by its qw and qh, and writes its S + S terms.
//
// The tables stay in shared memory for the CTA's blocks.  Operands are
// staged by the threads in the 32-byte-swizzled K-major layout of the TMA
// path (16-byte loads; d is a multiple of 8); the accumulation is fp32 in
// tensor memory from the 16-bit inputs, as in the CUDA-core version.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "attn_bwd_sam.cuh"
#include "attn_fwd_kernel.cuh"

namespace sdpa09 {
namespace {

constexpr float kLog2eRel = 1.4426950408889634f;
constexpr int kRelTcThreads = 128;  // one thread per row of the block; warp 0 lane 0 issues

// Offset of 16-byte chunk c of row R in a swizzled K-major tile of `rows`
// rows (16-column blocks rows * 32 bytes apart, 32 bytes per row, the two
// 16-byte halves of a row swapped on every other group of four rows: the
// layout the TMA path lands).
__device__ __forceinline__ uint32_t swz_off(int R, int c, int rows) {
    return (uint32_t)((c >> 1) * (rows * 32) + R * 32 + ((((c & 1) ^ ((R >> 2) & 1))) << 4));
}

template <int S, int DPAD>
struct RelTc {
    static constexpr int NT = 2 * S - 1;               // table rows
    static constexpr int NP = (NT + 15) / 16 * 16;     // MMA N: table rows padded to 16
    static constexpr int kAlloc = 2 * NP <= 32 ? 32 : (2 * NP <= 64 ? 64 : (2 * NP <= 128 ? 128 : 256));
    static constexpr int kPitch = RelLayout<S>::kStride * 2 + 16;  // staged output row, bytes
    static constexpr int kTab = (DPAD / 16) * NP * 32;            // one table tile, bytes
    static constexpr size_t kSmem = 2 * (size_t)Tile<DPAD>::kBytes + 2 * (size_t)kTab + (size_t)kBlockM * kPitch + 1024;
};

// The threads copy row `tid` of block `blk` into a Q tile with 16-byte
// cp.async copies (zeros past d and past the last row).
template <int DPAD>
__device__ __forceinline__ void load_q_rows(unsigned char* sq, const uint4* q4, size_t rows, int nc, int blk, int tid) {
    const size_t grow = (size_t)blk * kBlockM + tid;
    const bool rv = grow < rows;
#pragma unroll
    for (int c = 0; c < DPAD / 8; ++c) {
        const bool on = rv && c < nc;
        cp_async16(smem_u32(sq + swz_off(tid, c, kBlockM)), on ? q4 + grow * nc + c : q4, on ? 16u : 0u);
    }
    cp_async_commit();
}

// One CTA loops over blocks of 128 rows; block i + 1's Q is copied in while
// block i's terms are formed and written (two Q buffers).
template <int S, int DPAD, bool BF>
__global__ void __launch_bounds__(kRelTcThreads, 1) bwd_sam_rel_tc_kernel(const SamBwdParams p) {
    using C = RelTc<S, DPAD>;
    constexpr int NT = C::NT, NP = C::NP, kPitch = C::kPitch;
    constexpr int kGB = S <= 16 ? 4 : (S <= 32 ? 5 : 6);  // shift bits (qw, qh < S)
    constexpr int kChunks = DPAD / 8;
    constexpr int RW0 = RelLayout<S>::kRw0, STRIDE = RelLayout<S>::kStride;
    using T = Tile<DPAD>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // the swizzle pattern is taken from address bits: tiles start 1 KB aligned
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* sQ = smem;                          // 2 x [128][DPAD] swizzled
    unsigned char* sRw = smem + 2 * T::kBytes;         // [NP][DPAD] swizzled, rows >= NT zero
    unsigned char* sRh = sRw + C::kTab;
    unsigned char* sO = sRh + C::kTab;                 // [128][kPitch] output rows
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int d = p.d, nc = d / 8;
    const size_t rows = (size_t)p.BH * p.Nq;
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    const uint4* q4 = static_cast<const uint4*>(p.q);
    const int nblk = (int)((rows + kBlockM - 1) / kBlockM);
    if ((int)blockIdx.x < nblk) load_q_rows<DPAD>(sQ, q4, rows, nc, blockIdx.x, tid);

    // tables, once per CTA
    const uint4* th = static_cast<const uint4*>(p.rel_h);
    const uint4* tw = static_cast<const uint4*>(p.rel_w);
    for (int i = tid; i < NP * kChunks; i += kRelTcThreads) {
        const int R = i / kChunks, c = i - R * kChunks;
        const bool on = R < NT && c < nc;
        *reinterpret_cast<uint4*>(sRh + swz_off(R, c, NP)) = on ? th[(size_t)R * nc + c] : z4;
        *reinterpret_cast<uint4*>(sRw + swz_off(R, c, NP)) = on ? tw[(size_t)R * nc + c] : z4;
    }
    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, C::kAlloc);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_sh;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    constexpr uint32_t idesc = make_idesc_f16(BF, kBlockM, NP, false);
    int it = 0;
    bool ok = true;
    for (int blk = blockIdx.x; ok && blk < nblk; blk += gridDim.x, ++it) {
        unsigned char* sq = sQ + (it & 1) * T::kBytes;
        cp_async_wait<0>();        // this block's Q rows (copied during the last block)
        fence_proxy_async_smem();  // written through the generic proxy, read by the tensor core
        tc_fence_before();
        __syncthreads();           // Q staged; the last block's reads of tensor memory and sO done
        tc_fence_after();
        if (warp == 0) {  // converged: the wrappers issue from lane 0
            issue_qk_rows<DPAD, NP>(tmem, kdesc(smem_u32(sq)), kdesc(smem_u32(sRw)), idesc);
            issue_qk_rows<DPAD, NP>(tmem + NP, kdesc(smem_u32(sq)), kdesc(smem_u32(sRh)), idesc);
            mma_commit(&bar_mma);
        }
        // the next block's Q into the other buffer (its last reader, the MMAs
        // of the block before, completed before that block's terms were read)
        if (blk + (int)gridDim.x < nblk)
            load_q_rows<DPAD>(sQ + ((it + 1) & 1) * T::kBytes, q4, rows, nc, blk + gridDim.x, tid);
        __syncwarp();
        if (!mbar_wait(&bar_mma, it & 1, &abort_sh, kStatusWaitG)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const size_t grow = (size_t)blk * kBlockM + tid;
        const int q = grow < rows ? (int)(grow % (size_t)p.Nq) : 0;
        const int qh = q / S, qw = q - (q / S) * S;
        unsigned char* orow = sO + tid * kPitch;
        // rel_w[kw] = G_w[qw + S - 1 - kw] and rel_h[kh] = G_h[qh + S - 1 - kh]:
        // after a shift by qw (qh), entry S - 1 - kw (kh); packed to fp16, and
        // the row written as 16-byte chunks: rel_h at [0, S), rel_w at
        // [RW0, RW0 + S), zeros between and after
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            uint32_t pk[RW0 / 2];
            {
                float g[NP];
                {
                    uint32_t v[NP];
                    tmem_ld_cols<NP>(tmem + lane_base + (part ? NP : 0), v);
#pragma unroll
                    for (int t = 0; t < NP; ++t) g[t] = __uint_as_float(v[t]) * kLog2eRel;
                }
                shift_down<NP, kGB>(g, part ? qh : qw);
#pragma unroll
                for (int u = 0; u < RW0 / 2; ++u) {
                    const float lo = 2 * u < S ? g[S - 1 - 2 * u] : 0.f;
                    const float hi = 2 * u + 1 < S ? g[S - 2 - 2 * u] : 0.f;
                    const __half2 h2 = __floats2half2_rn(lo, hi);
                    pk[u] = *reinterpret_cast<const uint32_t*>(&h2);
                }
            }
            unsigned char* dstp = orow + (part ? 0 : RW0 * 2);
#pragma unroll
            for (int c = 0; c < RW0 / 8; ++c)
                *reinterpret_cast<uint4*>(dstp + 16 * c) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        __syncthreads();  // output rows staged
        // coalesced copies of the block's rows (consecutive in the output)
        const size_t r0 = (size_t)blk * kBlockM;
        const int nrow = (int)min((size_t)kBlockM, rows - r0);
        constexpr int cpr = STRIDE / 8;  // 16-byte chunks per row
        uint4* dst = reinterpret_cast<uint4*>(p.rel + r0 * STRIDE);
        for (int i = tid; i < nrow * cpr; i += kRelTcThreads) {
            const int r = i / cpr, ch = i - r * cpr;
            dst[i] = *reinterpret_cast<const uint4*>(sO + r * kPitch + ch * 16);
        }
        if constexpr (S != 64) {
            // on 14-wide grids a key row can straddle the query pass's two column
            // halves, so it adds its dRelH sums into rows cleared here
            float4* dr = reinterpret_cast<float4*>(p.d_relh + r0 * S);
            for (int i = tid; i < nrow * S / 4; i += kRelTcThreads) dr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i = nrow * S / 4 * 4 + tid; i < nrow * S; i += kRelTcThreads) p.d_relh[r0 * S + i] = 0.f;
        }
    }
    cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kAlloc);
    }
    if (tid == 0 && abort_sh != 0 && p.status) atomicCAS(p.status, 0, abort_sh);
}

template <int S, int DPAD, bool BF>
cudaError_t launch_rel_tc(const SamBwdParams& p, int nsm, cudaStream_t st) {
    using C = RelTc<S, DPAD>;
    auto kern = bwd_sam_rel_tc_kernel<S, DPAD, BF>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRelTcThreads, C::kSmem);
    if (e != cudaSuccess) return e;
    // resident CTAs of an SM must fit its 512 tensor-memory columns together
    per_sm = std::max(1, std::min(per_sm, 512 / C::kAlloc));
    const int64_t nblk = ((int64_t)p.BH * p.Nq + kBlockM - 1) / kBlockM;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(nblk, (int64_t)per_sm * nsm));
    kern<<<grid, kRelTcThreads, C::kSmem, st>>>(p);
    return cudaGetLastError();
}

template <int S, bool BF>
cudaError_t launch_rel_tc_d(const SamBwdParams& p, int nsm, cudaStream_t st) {
    const int dpad = (p.d + 15) / 16 * 16;
    if (dpad == 64) return launch_rel_tc<S, 64, BF>(p, nsm, st);
    if (dpad == 80) return launch_rel_tc<S, 80, BF>(p, nsm, st);
    return cudaErrorInvalidValue;
}

}  // namespace

template <int S>
cudaError_t launch_rel_tc_s(const SamBwdParams& p, bool bf, int nsm, cudaStream_t st) {
    if (p.rel_stride != RelLayout<S>::kStride || p.rw0 != RelLayout<S>::kRw0) return cudaErrorInvalidValue;
    return bf ? launch_rel_tc_d<S, true>(p, nsm, st) : launch_rel_tc_d<S, false>(p, nsm, st);
}

cudaError_t launch_bwd_sam_rel_tc(const SamBwdParams& p, int S, bool bf, int nsm, cudaStream_t st) {
    if (S == 64) return launch_rel_tc_s<64>(p, bf, nsm, st);
    if (S == 48) return launch_rel_tc_s<48>(p, bf, nsm, st);
    if (S == 14) return launch_rel_tc_s<14>(p, bf, nsm, st);
    return cudaErrorInvalidValue;
}

}  // namespace sdpa09
