// attn_bwd_long.cuh -- tensor-core backward for sequences longer than one
// 128-key tile: two passes over the (query block, key block) pairs of each
// slice, so that no gradient is summed across CTAs.
//
//   key pass (MODE 0): a job is one key block j of a slice; for every query
//     block i it recomputes S = Q_i.K_j^T and dP = dO_i.V_j^T, forms
//     P = exp(scale*S + bias - lse_i) and dS = P * (dP - D_i), and adds
//     P^T.dO_i to dV_j and dS^T.Q_i to dK_j in tensor memory;
//   query pass (MODE 1): a job is one query block i; for every key block j it
//     recomputes S, dP, P, dS and adds dS.K_j to dQ_i (and, for SAM, dS.E to
//     the row sums of dS over key rows with the same column, see below).
//
// lse is the forward's row log-sum-exp (attn_fwd_train) and D = rowsum(dO*O)
// comes from a pre-pass; both are per query row, so no row statistics are
// exchanged between threads.  P and dS go through shared memory as 16-bit
// A operands ([key block of 16][query row][16], read MN-major for dV, dK and
// K-major for dQ), as in the windows kernel.
//
// SAM decomposed relative position: the bias of (q, k) is
// rel_h[q][kh] + rel_w[q][kw] (log2 units), read from the pre-pass's table of
// each query row.  Its gradient: dRelH[q][kh] = sum_kw dS[q][(kh,kw)] and
// dRelW[q][kw] = sum_kh dS[q][(kh,kw)], summed in fp32 by the softmax threads
// of the query pass (key tiles start on grid rows, so a column's kw is fixed
// at compile time); rows of dS sum to zero, so these partial sums cancel
// heavily and are kept out of 16-bit operands.  A post-pass turns them into
// dQ and table gradients.
//
// Warps: 0-7 softmax (thread = query row of lane (warp & 3) * 32 + lane;
// warps 0-3 take key columns [0,64), warps 4-7 [64,128)), 8 TMA producer,
// 9 MMA issue (+ TMEM allocation), 10-11 idle.
//
// Tensor memory: S [0,128) dP [128,256); key pass dV [256,256+DPAD) dK [..,
// +DPAD); query pass dQ [256,256+DPAD).
#pragma once
#include "attn_bwd_kernel.cuh"

namespace sdpa09 {

enum BwdLongMode { kBwdKeyPass = 0, kBwdQueryPass = 1 };

struct BwdPrepParams {
    const void *o, *dout;  // [BH][Nq][d] 16-bit
    float* Dws;            // [BH][Nq] rowsum(dO * O)
    int rows, d, is_bf16;
};
cudaError_t launch_bwd_prep(const BwdPrepParams& p, int nsm, cudaStream_t stream);

struct BwdLongParams {
    void *dq, *dk, *dv;     // 16-bit outputs [BH][N][d]
    float* dq32;            // SAM query pass: scale * dS.K in fp32 [BH][Nq][d] (the post-pass adds the rel terms)
    const float* lse;       // [BH][Nq] natural log
    const float* Dws;       // [BH][Nq] rowsum(dO * O)
    const __half* rel;      // SAM: [BH][Nq][rel_stride] fp16 log2 units: rel_h at 0, rel_w at rw0
    float* d_relh;          // SAM query pass: [BH][Nq][k_h] (64-wide grids: stored; 14-wide: added to rows the pre-pass cleared)
    float* d_relw;          // SAM query pass: [2][BH][Nq][k_w], one array per column half (stored)
    int* status;
    int BH, Nq, Nk, d;
    int n_qb, n_kb;         // query / key blocks per slice
    int n_jobs;
    int kv_w;               // keys per key block (128; 112 on 14-wide SAM grids, 96 on 48-wide ones)
    int k_h, k_w, rel_stride, rw0;
    int nst;
    int full_atoms, part;
    uint32_t off_res, off_ring, off_p, off_ds, stage_bytes;
    float scale, scale_log2;
    int is_bf16;
};

// halves 8j..8j+7 of a fp16 row as floats
__device__ __forceinline__ void half8(const __half* p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
        f[2 * e] = t.x;
        f[2 * e + 1] = t.y;
    }
}

template <int DPAD, int BIAS, int MODE, int SW>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_long_kernel(const __grid_constant__ BwdMaps tm, const BwdLongParams p) {
    using T = Tile<DPAD>;
    static_assert(BIAS == kBiasNone || (BIAS == kBiasSam && (SW == 14 || SW == 48 || SW == 64)), "bias kinds");
    static_assert(256 + 2 * DPAD <= 512 && 256 + DPAD + 64 <= 512, "tensor memory");
    constexpr bool kSam = BIAS == kBiasSam;
    constexpr bool kKey = MODE == kBwdKeyPass;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* sRes = smem + p.off_res;    // key pass: K_j, V_j; query pass: Q_i, dO_i
    unsigned char* sRing = smem + p.off_ring;  // key pass: (Q_i, dO_i); query pass: (K_j, V_j)
    unsigned char* sP = smem + p.off_p;        // key pass only
    unsigned char* sDS = smem + p.off_ds;

    __shared__ uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
    __shared__ uint64_t bar_res_full, bar_res_empty;
    __shared__ uint64_t bar_s, bar_sfree, bar_p, bar_pfree, bar_acc, bar_accfree, bar_final;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = &abort_sh;
    const int nst = p.nst;
    const bool bf = p.is_bf16 != 0;
    const int n_inner = kKey ? p.n_qb : p.n_kb;

    if (tid == 0) {
        abort_sh = 0;
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_res_full, 1);
        mbar_init(&bar_res_empty, 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_sfree, 8);
        mbar_init(&bar_p, 8);
        mbar_init(&bar_pfree, 1);
        mbar_init(&bar_acc, 1);
        mbar_init(&bar_accfree, 8);
        mbar_init(&bar_final, 1);
        fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tm.q);
        prefetch_tensormap(&tm.k);
        prefetch_tensormap(&tm.v);
        prefetch_tensormap(&tm.dout);
    }
    griddep_wait();
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t tS = tmem, tDP = tmem + 128, tA0 = tmem + 256, tA1 = tmem + 256 + DPAD;
    const int job0 = blockIdx.x, job_step = gridDim.x;

    if (warp >= 8) {
        regs_dec<kControlRegs>();
        if (warp == kProducerWarp && lane == 0) {
            // ============================================================ producer
            const uint32_t tx = 2u * (uint32_t)T::kBytes;
            int u = 0, jn = 0;
            bool ok = true;
            for (int job = job0; ok && job < p.n_jobs; job += job_step, ++jn) {
                const int slice = job / (kKey ? p.n_kb : p.n_qb);
                const int blk = job - slice * (kKey ? p.n_kb : p.n_qb);
                // the job's resident tiles: K_j, V_j (key pass) or Q_i, dO_i
                if (jn > 0 && !mbar_wait(&bar_res_empty, (jn - 1) & 1, abort_flag, kStatusWaitEmpty)) break;
                const int r0 = kKey ? blk * p.kv_w : blk * kBlockM;
                mbar_arrive_expect_tx(&bar_res_full, tx);
                tma_load_4d(sRes, kKey ? &tm.k : &tm.q, &bar_res_full, 0, r0, slice, 0);
                tma_load_4d(sRes + T::kBytes, kKey ? &tm.v : &tm.dout, &bar_res_full, 0, r0, slice, 0);
                if (p.part) {
                    const int po = p.full_atoms * kBlockM * 32;
                    tma_load_3d(sRes + po, kKey ? &tm.kp : &tm.qp, &bar_res_full, 0, r0, slice);
                    tma_load_3d(sRes + T::kBytes + po, kKey ? &tm.vp : &tm.dop, &bar_res_full, 0, r0, slice);
                }
                for (int it = 0; it < n_inner; ++it, ++u) {
                    const int st = u % nst;
                    if (u >= nst && !mbar_wait(&bar_empty[st], ((u / nst) + 1) & 1, abort_flag, kStatusWaitEmpty)) {
                        ok = false;
                        break;
                    }
                    unsigned char* b = sRing + st * p.stage_bytes;
                    const int rr = kKey ? it * kBlockM : it * p.kv_w;
                    mbar_arrive_expect_tx(&bar_full[st], tx);
                    tma_load_4d(b, kKey ? &tm.q : &tm.k, &bar_full[st], 0, rr, slice, 0);
                    tma_load_4d(b + T::kBytes, kKey ? &tm.dout : &tm.v, &bar_full[st], 0, rr, slice, 0);
                    if (p.part) {
                        const int po = p.full_atoms * kBlockM * 32;
                        tma_load_3d(b + po, kKey ? &tm.qp : &tm.kp, &bar_full[st], 0, rr, slice);
                        tma_load_3d(b + T::kBytes + po, kKey ? &tm.dop : &tm.vp, &bar_full[st], 0, rr, slice);
                    }
                }
            }
            if (*abort_flag) {
                for (int w = (u > nst ? u - nst : 0); w < u; ++w)
                    mbar_wait(&bar_full[w % nst], (w / nst) & 1, nullptr, 0);
                if (jn > 0) mbar_wait(&bar_res_full, (jn - 1) & 1, nullptr, 0);
            }
        } else if (warp == kMmaWarp) {
            // ================================================================ MMA
            // the whole warp runs the issue loop; lane 0 issues
            const uint32_t idesc_s = make_idesc_f16(bf, kBlockM, kBlockN, false);
            const uint32_t idesc_g = make_idesc_f16_mn(bf, kBlockM, DPAD, true, true);   // dV, dK: A MN-major
            const uint32_t idesc_q = make_idesc_f16_mn(bf, kBlockM, DPAD, false, true);  // dQ: A K-major
            const uint32_t aRes = smem_u32(sRes), aP = smem_u32(sP), aDS = smem_u32(sDS);
            // every lane waits (no warp vote: the lanes run in step)
            auto waitb = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
                if (!mbar_wait(bar, parity, abort_flag, code)) return false;
                tc_fence_after();
                return true;
            };
            int u = 0;  // ring uses (= inner iterations over all jobs)
            int jn = 0;
            bool ok = true;
            for (int job = job0; ok && job < p.n_jobs; job += job_step, ++jn) {
                if (!waitb(&bar_res_full, jn & 1, kStatusWaitQ)) break;
                // S = Q.K^T and dP = dO.V^T of ring use w
                auto issue_sdp = [&](int w) -> bool {
                    const int st = w % nst;
                    const uint32_t b = smem_u32(sRing + st * p.stage_bytes);
                    if (!waitb(&bar_full[st], (w / nst) & 1, kStatusWaitK)) return false;
                    if (w > 0 && !waitb(&bar_sfree, (w - 1) & 1, kStatusWaitS)) return false;
                    const uint32_t aQ = kKey ? b : aRes, aK = kKey ? aRes : b;
                    const uint32_t aDO = kKey ? b + T::kBytes : aRes + T::kBytes, aV = kKey ? aRes + T::kBytes : b + T::kBytes;
                    issue_qk<DPAD>(tS, kdesc(aQ), kdesc(aK), idesc_s);
                    issue_qk<DPAD>(tDP, kdesc(aDO), kdesc(aV), idesc_s);
                    mma_commit(&bar_s);
                    return true;
                };
                const int u0 = u;
                if (!issue_sdp(u0)) break;
                for (int it = 0; it < n_inner; ++it, ++u) {
                    const int st = u % nst;
                    const uint32_t b = smem_u32(sRing + st * p.stage_bytes);
                    // the next tile's S and dP as soon as the softmax has read this
                    // tile's (they compute while it forms P and dS), then this
                    // tile's gradient products once P and dS are in shared memory
                    if (it + 1 < n_inner && !issue_sdp(u + 1)) { ok = false; break; }
                    if (!waitb(&bar_p, u & 1, kStatusWaitP)) { ok = false; break; }
                    // the accumulators are rewritten once the last job's epilogue read them
                    if (it == 0 && jn > 0 && !waitb(&bar_accfree, (jn - 1) & 1, kStatusWaitO)) { ok = false; break; }
                    const uint32_t acc = it > 0 ? 1u : 0u;
                    // descriptors built once; a step only moves the start-address
                    // field (16-byte units): 512 B per 16 rows, kBlockM * 32 B per
                    // 16-column block
                    if constexpr (kKey) {
                        const uint64_t dP = vdesc(aP), dS = vdesc(aDS), dQ = vdesc(b), dDO = vdesc(b + T::kBytes);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)  // dV += P^T.dO over 16 query rows per step
                            mma_ss(tA0, dP + (uint64_t)(ks * 32), dDO + (uint64_t)(ks * 32), idesc_g, (acc || ks > 0) ? 1u : 0u);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)  // dK += dS^T.Q
                            mma_ss(tA1, dS + (uint64_t)(ks * 32), dQ + (uint64_t)(ks * 32), idesc_g, (acc || ks > 0) ? 1u : 0u);
                    } else {
                        const uint64_t dS = kdesc(aDS), dK = vdesc(b);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)  // dQ += dS.K over 16 keys per step
                            mma_ss(tA0, dS + (uint64_t)(ks * (kBlockM * 32 / 16)), dK + (uint64_t)(ks * 32), idesc_q,
                                   (acc || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(&bar_pfree);
                    mma_commit(&bar_empty[st]);
                }
                if (!ok) break;
                mma_commit(&bar_acc);
                mma_commit(&bar_res_empty);
            }
            // every MMA issued has retired before tensor memory is released
            mma_commit(&bar_final);
            mbar_wait(&bar_final, 0, nullptr, 0);
        }
    } else {
        regs_inc<kSoftmaxRegs>();
        // ============================================================== softmax
        const int r = (warp & 3) * 32 + lane;  // row in the query block == TMEM lane
        const int half = warp >> 2;            // key columns [64 half, 64 half + 64)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t c0 = (uint32_t)(64 * half);
        int u = 0, jn = 0;
        bool ok = true;
        for (int job = job0; ok && job < p.n_jobs; job += job_step, ++jn) {
            const int slice = job / (kKey ? p.n_kb : p.n_qb);
            const int blk = job - slice * (kKey ? p.n_kb : p.n_qb);
            // query pass: the row and its statistics are fixed for the job
            float lse2 = 0.f, Dq = 0.f;
            int q = 0;
            bool q_ok = false;
            auto row_stats = [&](int qq) {
                q = qq;
                q_ok = qq < p.Nq;
                const size_t ri = (size_t)slice * p.Nq + (q_ok ? qq : 0);
                lse2 = q_ok ? p.lse[ri] * kLog2e : 0.f;
                Dq = q_ok ? p.Dws[ri] : 0.f;
            };
            if (!kKey) row_stats(blk * kBlockM + r);
            // SAM query pass: the row's dRelW partial sums (this thread's columns)
            float dw[kSam && !kKey ? (SW > 0 ? SW : 1) : 1];
#pragma unroll
            for (int c = 0; c < (int)(sizeof(dw) / sizeof(float)); ++c) dw[c] = 0.f;
            for (int it = 0; it < n_inner; ++it, ++u) {
                if (kKey) row_stats(it * kBlockM + r);
                const int key0 = kKey ? blk * p.kv_w : it * p.kv_w;
                const int nvalid = min(p.kv_w, p.Nk - key0);  // key columns of this tile
                // SAM bias terms of the row for this tile's keys (log2 units):
                // rel_w of every key column as fp16 pairs, rel_h of the key rows
                constexpr int kRW = SW > 0 ? (SW + 1) / 2 : 1;
                __half2 rw2[kRW];
                // key rows per key tile: 2 on 64- and 48-wide grids, 8 on 14-wide ones
                constexpr int kKR = SW == 14 ? 8 : 2;
                float rh[SW > 0 ? (SW == 64 ? 1 : kKR) : 1];
                if constexpr (kSam) {
                    const __half* rel = p.rel + ((size_t)slice * p.Nq + (q_ok ? q : 0)) * p.rel_stride;
                    const int kh0 = key0 / SW;
#pragma unroll
                    for (int j8 = 0; j8 < (SW + 7) / 8; ++j8) {
                        const uint4 u4 = *reinterpret_cast<const uint4*>(rel + p.rw0 + 8 * j8);
                        const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * j8 + e < kRW) rw2[4 * j8 + e] = *reinterpret_cast<const __half2*>(&w4[e]);
                    }
                    if constexpr (SW == 64) {
                        rh[0] = __half2float(rel[min(kh0 + half, p.k_h - 1)]);
                    } else if constexpr (SW == 48) {
                        // key rows kh0, kh0 + 1 (kh0 is even)
                        const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(rel + kh0));
                        rh[0] = f2.x;
                        rh[1] = f2.y;
                    } else {
                        float f[8];
                        half8(rel + kh0, f);  // key rows kh0..kh0+7 (kh0 is a multiple of 8)
#pragma unroll
                        for (int e = 0; e < 8; ++e) rh[e] = f[e];
                    }
                }
                __syncwarp();
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_s, u & 1, abort_flag, kStatusWaitS))) { ok = false; break; }
                tc_fence_after();
                float xs[64];
                {
                    uint32_t v[64];
                    tmem_ld64(tS + lane_base + c0, v);
#pragma unroll
                    for (int c = 0; c < 64; ++c) xs[c] = __uint_as_float(v[c]);
                }
                // P = 2^(s scale log2e + bias - lse), zero outside the tile; then
                // dS = P (dP - D), with dP read once P is done
                float dp[64];
                auto body = [&](auto hc) {
                    constexpr int H0 = decltype(hc)::value;  // this thread's column half
                    // column pairs through the packed FP32 ops (the same roundings
                    // as one column at a time)
                    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                    const float2 nl2 = make_float2(-lse2, -lse2);
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        const int col = 64 * H0 + c;
                        float2 b2 = make_float2(0.f, 0.f);
                        if constexpr (kSam) {
                            // grid widths are even: both columns share a key row
                            const float2 rwf = __half22float2(rw2[(col % SW) / 2]);
                            const float rhv = SW == 64 ? rh[0] : rh[col / SW < kKR ? col / SW : kKR - 1];
                            b2 = make_float2(rhv + rwf.x, rhv + rwf.y);
                        }
                        const float2 a = __ffma2_rn(make_float2(xs[c], xs[c + 1]), sc2, __fadd2_rn(b2, nl2));
                        xs[c] = (q_ok && col < nvalid) ? ex2_approx(a.x) : 0.f;
                        xs[c + 1] = (q_ok && col + 1 < nvalid) ? ex2_approx(a.y) : 0.f;
                    }
                    {
                        uint32_t v[64];
                        tmem_ld64(tDP + lane_base + c0, v);
                        const float2 nd2 = make_float2(-Dq, -Dq);
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            const float2 t = __fadd2_rn(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), nd2);
                            const float2 y = __fmul2_rn(make_float2(xs[c], xs[c + 1]), t);
                            dp[c] = y.x;
                            dp[c + 1] = y.y;
                        }
                    }
                    tc_fence_before();
                    warp_arrive(&bar_sfree);
                    if constexpr (kSam && !kKey) {
                        // dRelH: the row's dS summed over each key row of its columns
                        // (64-wide grids: one key row per column half, stored; on 14- and
                        // 48-wide grids a key row can straddle the halves: atomic adds);
                        // dRelW: summed per key column over the job's key rows
                        if (q_ok) {
                            const int kh0 = key0 / SW;
                            float* dst = p.d_relh + ((size_t)slice * p.Nq + q) * p.k_h;
                            constexpr int kr0 = (64 * H0) / SW, kr1 = (64 * H0 + 63) / SW;
#pragma unroll
                            for (int kr = kr0; kr <= kr1; ++kr) {
                                if (kr < kKR) {
                                    // column pairs (grid widths are even: a pair never
                                    // straddles two key rows), four partial sums
                                    float2 a2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                                    for (int c = 0; c < 64; c += 2)
                                        if ((64 * H0 + c) / SW == kr)
                                            a2[(c >> 1) & 1] = __fadd2_rn(a2[(c >> 1) & 1], make_float2(dp[c], dp[c + 1]));
                                    const float2 s2 = __fadd2_rn(a2[0], a2[1]);
                                    const float a = s2.x + s2.y;
                                    if constexpr (SW == 64) dst[kh0 + kr] = a;
                                    else if (kh0 + kr < p.k_h) atomicAdd(dst + kh0 + kr, a);
                                }
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            const int i = (64 * H0 + c) % SW;
                            const float2 y = __fadd2_rn(make_float2(dw[i], dw[i + 1]), make_float2(dp[c], dp[c + 1]));
                            dw[i] = y.x;
                            dw[i + 1] = y.y;
                        }
                    }
                };
                if (half == 0) body(std::integral_constant<int, 0>{});
                else body(std::integral_constant<int, 1>{});
                // the last tile's gradient products must be done with P and dS
                __syncwarp();
                if (u > 0 && !__all_sync(0xffffffffu, mbar_wait(&bar_pfree, (u - 1) & 1, abort_flag, kStatusWaitP))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // one packing loop per operand type, chosen once per tile
                auto pack_rows = [&](auto b16) {
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 8) {
                        uint32_t wp[4], wd[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float p0 = xs[cc + 2 * e], p1 = xs[cc + 2 * e + 1];
                            const float d0 = dp[cc + 2 * e], d1 = dp[cc + 2 * e + 1];
                            wp[e] = decltype(b16)::value ? pack_bf16(p0, p1) : pack_f16(p0, p1);
                            wd[e] = decltype(b16)::value ? pack_bf16(d0, d1) : pack_f16(d0, d1);
                        }
                        const int col = (int)c0 + cc;
                        const uint32_t off = (uint32_t)((col >> 4) * (kBlockM * 32)) + half_off(r, (col >> 3) & 1);
                        if constexpr (kKey) *reinterpret_cast<uint4*>(sP + off) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
                        *reinterpret_cast<uint4*>(sDS + off) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    }
                };
                if (bf) pack_rows(std::true_type{});
                else pack_rows(std::false_type{});
                fence_proxy_async_smem();  // read by the tensor core
                warp_arrive(&bar_p);
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_acc, jn & 1, abort_flag, kStatusWaitO))) break;
            tc_fence_after();
            if constexpr (kKey) {
                // key row r of the block: dV (half 0, x 1) or dK (half 1, x scale)
                const int key = blk * p.kv_w + r;
                uint32_t v[DPAD];
                tmem_ld_cols<DPAD>((half ? tA1 : tA0) + lane_base, v);
                if (r < p.kv_w && key < p.Nk) {
                    const float f = half ? p.scale : 1.0f;
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(half ? p.dk : p.dv) +
                                                          ((size_t)slice * p.Nk + key) * (size_t)p.d * 2);
#pragma unroll
                    for (int c8 = 0; c8 < DPAD / 8; ++c8) {
                        if (c8 * 8 < p.d) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float a = __uint_as_float(v[c8 * 8 + 2 * e]) * f;
                                const float b2 = __uint_as_float(v[c8 * 8 + 2 * e + 1]) * f;
                                w[e] = bf ? pack_bf16(a, b2) : pack_f16(a, b2);
                            }
                            dst[c8] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            } else {
                if (half == 0) {
                    // dQ row: scale dS.K, to 16 bits (or fp32 for the SAM post-pass)
                    uint32_t v[DPAD];
                    tmem_ld_cols<DPAD>(tA0 + lane_base, v);
                    if (q_ok) {
                        if (kSam) {
                            float4* dst = reinterpret_cast<float4*>(p.dq32 + ((size_t)slice * p.Nq + q) * (size_t)p.d);
#pragma unroll
                            for (int c4 = 0; c4 < DPAD / 4; ++c4)
                                if (c4 * 4 < p.d)
                                    dst[c4] = make_float4(__uint_as_float(v[4 * c4]) * p.scale, __uint_as_float(v[4 * c4 + 1]) * p.scale,
                                                          __uint_as_float(v[4 * c4 + 2]) * p.scale, __uint_as_float(v[4 * c4 + 3]) * p.scale);
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.dq) +
                                                                  ((size_t)slice * p.Nq + q) * (size_t)p.d * 2);
#pragma unroll
                            for (int c8 = 0; c8 < DPAD / 8; ++c8) {
                                if (c8 * 8 < p.d) {
                                    uint32_t w[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float a = __uint_as_float(v[c8 * 8 + 2 * e]) * p.scale;
                                        const float b2 = __uint_as_float(v[c8 * 8 + 2 * e + 1]) * p.scale;
                                        w[e] = bf ? pack_bf16(a, b2) : pack_f16(a, b2);
                                    }
                                    dst[c8] = make_uint4(w[0], w[1], w[2], w[3]);
                                }
                            }
                        }
                    }
                }
                if constexpr (kSam) {
                    // dRelW row: each column half stores its sums in its own array
                    if (q_ok) {
                        float* dst = p.d_relw + (((size_t)half * p.BH + slice) * p.Nq + q) * p.k_w;
                        if constexpr (SW % 4 == 0) {
#pragma unroll
                            for (int c = 0; c < SW; c += 4)
                                *reinterpret_cast<float4*>(dst + c) = make_float4(dw[c], dw[c + 1], dw[c + 2], dw[c + 3]);
                        } else {
#pragma unroll
                            for (int c = 0; c < SW; c += 2) *reinterpret_cast<float2*>(dst + c) = make_float2(dw[c], dw[c + 1]);
                        }
                    }
                }
            }
            tc_fence_before();
            warp_arrive(&bar_accfree);
        }
    }

    // ============================================================== teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && abort_sh != 0 && p.status) atomicCAS(p.status, 0, abort_sh);
}

}  // namespace sdpa09
