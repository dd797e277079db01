// attn_bwd_kernel.cuh -- tensor-core backward of the fused attention for
// GB300 (sm_103a): dQ, dK, dV (and the bias gradients) of
// O = softmax(scale * Q.K^T + bias) . V.
//
// "视觉大模型训练和推理加速" section 二: the window operators are written with
// their forward and their backward computation, for training.  With
// P = softmax(S), dO the gradient of the loss with respect to O and
// D_i = sum_c dO[i,c] O[i,c] (= sum_j P_ij dP_ij):
//     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//     dQ = scale dS K,  dK = scale dS^T Q,
// and every additive bias entry receives dS.
//
// Packed windows (this file's first kernel): every slice has at most 128
// queries and 128 keys, and g = 128 / SL whole slices share one 128-row tile
// (SL-row slots, block-diagonal validity), as in the forward's packed tiling.
// A tile is at once the query block and the key block, so the CTA computes
// the exact softmax of each row itself and all five products of the tile:
//     S  = Q.K^T, dP = dO.V^T              (TMEM, lanes = query rows)
//     P, dS                                (softmax warps -> shared memory,
//                                           16-bit, [key block][query row][16])
//     dV = P^T.dO, dK = dS^T.Q             (A operand read MN-major: M = keys)
//     dQ = dS.K                            (A operand read K-major: M = queries)
// The same shared-memory P / dS tile is the A operand of both orientations:
// blocks of 16 keys, each holding every query row's 32 bytes, is the K-major
// layout of dS (M = query) and the MN-major layout of dS^T (M = key), as the
// forward reads one K tile K-major and one V tile MN-major.
//
// Warps: 0-3 softmax (thread t = tile row t), 4-7 epilogue (read dV, dK, dQ
// out of tensor memory and store them while the next tile runs), 8 TMA
// producer, 9 MMA issue (+ TMEM allocation), 10-11 idle.
//
// Tensor memory: S [0,128) dP [128,256) dV [256,256+DPAD) dK [.., +DPAD)
// dQ [.., +DPAD).
#pragma once
#include "attn_fwd_kernel.cuh"

namespace sdpa09 {

constexpr int kBwdThreads = 384;
constexpr int kBwdSoftRegs = 232;
constexpr int kBwdEpiRegs = 184;
constexpr int kBwdCtlRegs = 88;
static_assert(128 * (kBwdSoftRegs + kBwdEpiRegs + kBwdCtlRegs) == kBwdThreads * kLaunchRegs,
              "register split must add up to the launch allocation");

struct BwdMaps {
    CUtensorMap q, k, v, dout, qp, kp, vp, dop;
};

struct BwdTcParams {
    void *dq, *dk, *dv;  // outputs [BH][N][d] 16-bit
    const void* o;       // the forward output [BH][Nq][d] (for D = rowsum(dO * O))
    int* status;         // device status word
    int BH, H, Nq, Nk, d;
    int n_jobs;          // packed tiles
    int g, sl;           // slices per tile, rows per slot
    int nst;             // ring stages
    int full_atoms, part;
    uint32_t off_ring, off_p, off_ds, off_extra, off_rows, stage_bytes;
    float scale, scale_log2;
    int is_bf16;
    // Swin (windows layout)
    const float* table;  // [(2M-1)^2][H]
    float* d_table;      // its gradient, added to
    int win, grid_h, grid_w, shift, n_w, n_ww, n_wh;
    uint32_t fd_h[2], fd_w[2], fd_ww[2];
    int swin_rows;  // 1: per-CTA bias rows (fp16, log2 units) and region bits in shared memory
    int swin_acc;       // 1: dS summed per (head, key token, query token) in shared memory
    int swin_acc_atomic;  // 1: two slots of a tile may share a head (g > H): atomic adds there
    uint32_t off_acc;   // that sum, fp32 [H][N keys][N queries]
    // Swin image layout: q/k/v/out/dout/dq/dk/dv are [images][grid_h][grid_w][H][d];
    // the producer warp gathers each window's rows (shift and partition folded
    // into the addresses) and the epilogue writes the gradients back the same way
    int swin_image;
    uint32_t fd_m[2];
    const void *q, *k, *v, *dout;
};

// Byte offset of the 16-byte half `hh` (columns 8hh..8hh+7) of row r in a
// 16-column block of a 128-row operand tile (32-byte swizzle).
__device__ __forceinline__ uint32_t half_off(int r, int hh) {
    return (uint32_t)(r * 32 + ((hh ^ ((r >> 2) & 1)) << 4));
}

template <int DPAD, int BIAS, int SL, bool IMG, bool FAST>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_win_kernel(const __grid_constant__ BwdMaps tm, const BwdTcParams p) {
    using T = Tile<DPAD>;
    // Swin image token layout (p.swin_image) as a compile-time choice: the
    // windows-layout kernel carries none of its gather and scatter code.
    // FAST: the Swin case of bias rows and a shared, non-atomic table-gradient
    // area (p.swin_rows, p.swin_acc, !p.swin_acc_atomic), fixed at compile
    // time so that the kernel carries only that path
    constexpr bool kImg = IMG && BIAS == kBiasSwin;
    static_assert(SL == 32 || SL == 64 || SL == 128, "slot rows");
    static_assert(256 + 3 * DPAD <= 512, "tensor memory: S, dP and three accumulators");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* sRing = smem + p.off_ring;  // stages: Q, K, V, dO tiles
    unsigned char* sP = smem + p.off_p;        // P  [8 key blocks][128 rows][32 B]
    unsigned char* sDS = smem + p.off_ds;      // dS, same layout
    float* sTab = reinterpret_cast<float*>(smem + p.off_extra);  // Swin table [(2M-1)^2][H]
    const int n_tab = (2 * p.win - 1) * (2 * p.win - 1) * p.H;
    float* sDTab = sTab + n_tab;  // its gradient, summed per CTA
    // Swin rows variant (when the host found room): per head an fp16 bias
    // matrix [SL query tokens][SL key tokens] in log2 units (the SL / 8
    // 16-byte chunks of a row XOR-swizzled by the row's low bits), then the
    // region-difference
    // bits [3 window kinds][SL][SL / 32]
    unsigned char* sRows = smem + p.off_rows;
    const uint32_t* sBits = reinterpret_cast<const uint32_t*>(sRows + p.H * SL * SL * 2);
    float* sAcc = reinterpret_cast<float*>(smem + p.off_acc);

    __shared__ uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
    __shared__ uint64_t bar_s, bar_sfree, bar_p, bar_pfree, bar_acc, bar_accfree, bar_final;
    __shared__ uint64_t bar_d[2];  // D of a tile is in sD[t & 1]
    __shared__ uint64_t bar_accsync;  // Swin: every softmax warp added this tile's dS
    __shared__ float sD[2][128];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    __shared__ int s_tok[128];  // Swin: per-token position and region labels

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = &abort_sh;
    const int nst = p.nst;
    const bool bf = p.is_bf16 != 0;

    if (tid == 0) {
        abort_sh = 0;
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&bar_full[i], kImg ? 32 : 1);  // image layout: one per gathering lane
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_s, 1);
        mbar_init(&bar_sfree, 4);
        mbar_init(&bar_p, 4);
        // P / dS are free once the products are done with them
        mbar_init(&bar_pfree, 1);
        mbar_init(&bar_acc, 1);
        mbar_init(&bar_accfree, 4);
        mbar_init(&bar_final, 1);
        mbar_init(&bar_accsync, 4);
        mbar_init(&bar_d[0], 4);
        mbar_init(&bar_d[1], 4);
        fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tm.q);
        prefetch_tensormap(&tm.k);
        prefetch_tensormap(&tm.v);
        prefetch_tensormap(&tm.dout);
    }
    griddep_wait();
    // P and dS start as zeros: a row's columns outside its own slot are never
    // written again, so the block-diagonal products see exact zeros there
    for (int i = tid; i < 2 * 8 * 128 * 32 / 16; i += kBwdThreads)
        reinterpret_cast<uint4*>(i < 8 * 128 * 2 ? sP : sDS)[i % (8 * 128 * 2)] = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (BIAS == kBiasSwin) {
        const int M = p.win, TT = 2 * M - 1;
        const int yb = (p.n_wh - 1) * M, xb = (p.n_ww - 1) * M;  // last window row / column origin
        for (int t = tid; t < 128; t += kBwdThreads) {
            const int tt = t < M * M ? t : 0;
            const int rt = tt / M, ct = tt - (tt / M) * M;
            const int lab = swin_strip(xb + ct, p.grid_w, M, p.shift) | (swin_strip(yb + rt, p.grid_h, M, p.shift) << 2);
            s_tok[t] = (rt * TT + ct) | (lab << 16);
        }
        for (int i = tid; i < n_tab; i += kBwdThreads) {
            sTab[i] = p.table[i];
            sDTab[i] = 0.f;
        }
        if ((FAST || p.swin_acc))
            for (int i = tid; i < p.H * p.Nq * p.Nk; i += kBwdThreads) sAcc[i] = 0.f;
        if ((FAST || p.swin_rows)) {
            __syncthreads();
            const int N = p.Nk, c0 = 2 * M * (M - 1);
            for (int w = tid; w < p.H * SL * (SL / 8); w += kBwdThreads) {
                const int q = w % (SL / 8), i = (w / (SL / 8)) % SL, hh = w / (SL * (SL / 8));
                const int pi = s_tok[i] & 0xFFFF;
                uint32_t v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float b2[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int j = 8 * q + 2 * e + z;
                        const bool ok = i < N && j < N;
                        // keys past the window get -inf: their score needs no mask
                        b2[z] = ok ? sTab[(pi - (s_tok[j] & 0xFFFF) + c0) * p.H + hh] * kLog2e
                                   : (j >= N ? -INFINITY : 0.f);
                    }
                    v[e] = pack_f16(b2[0], b2[1]);
                }
                *reinterpret_cast<uint4*>(sRows + (hh * SL + i) * SL * 2 + ((q ^ (i & (SL / 8 - 1) & 7)) << 4)) =
                    make_uint4(v[0], v[1], v[2], v[3]);
            }
            uint32_t* bits = reinterpret_cast<uint32_t*>(sRows + p.H * SL * SL * 2);
            for (int w = tid; w < 3 * SL * (SL / 32); w += kBwdThreads) {
                const int wd = w % (SL / 32), i = (w / (SL / 32)) % SL, kd = w / (SL * (SL / 32)) + 1;
                const int sl = ((kd & 1) ? 0x3 : 0) | ((kd & 2) ? 0xC : 0);
                const int li = s_tok[i] >> 16;
                uint32_t b = 0;
                if (i < N && p.shift) {
                    for (int e = 0; e < 32; ++e) {
                        const int j = wd * 32 + e;
                        if (j < N && (((s_tok[j] >> 16) ^ li) & sl)) b |= 1u << e;
                    }
                }
                bits[w] = b;
            }
        }
    }
    fence_proxy_async_smem();  // the zeros above are read by the tensor core
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tDV + DPAD, tDQ = tDK + DPAD;
    const int job0 = blockIdx.x, job_step = gridDim.x;

    if (warp >= 8) {
        regs_dec<kBwdCtlRegs>();
        if (kImg && warp == kProducerWarp) {
            // ============================================ producer, image layout
            // The whole warp copies each window's token rows of Q, K, V and dO
            // with 16-byte cp.async copies into the same swizzled tiles the TMA
            // path lands; token (r, c) of window (wr, wc) comes from image
            // position ((wr*win + r + shift) mod grid_h, (wc*win + c + shift)
            // mod grid_w) ("视觉大模型训练和推理加速" sections 一 and 二: the
            // shift and the partition are index mappings).  Padding rows and
            // columns are written as zeros.  Each lane's arrival on the stage
            // barrier is made by the copy hardware once that lane's copies
            // have landed, so the warp runs ahead to the next stage; the MMA
            // warp fences the proxies after its wait.
            constexpr int kChunks = DPAD / 8;
            constexpr int kLanesRow = kChunks <= 2 ? 2 : (kChunks <= 4 ? 4 : 8);
            constexpr int kRowsIt = 32 / kLanesRow;
            static_assert(SL % kRowsIt == 0, "a warp instruction stays inside one slice");
            const int c = lane % kLanesRow, rsub = lane / kLanesRow;
            const bool lane_on = c < kChunks, c_data = c * 8 < p.d;
            const uint32_t dchunk = (uint32_t)((c >> 1) * (kBlockM * 32));
            const size_t rowb = (size_t)p.d * 2;
            int u = 0;
            for (int job = job0; job < p.n_jobs; job += job_step, ++u) {
                const int st = u % nst;
                __syncwarp();
                if (u >= nst &&
                    !__all_sync(0xffffffffu, mbar_wait(&bar_empty[st], ((u / nst) + 1) & 1, abort_flag, kStatusWaitEmpty)))
                    break;
                unsigned char* b = sRing + st * p.stage_bytes;
                if (lane_on) {
#pragma unroll 1
                    for (int g = 0; g < p.g; ++g) {
                        const uint32_t slice = (uint32_t)(job * p.g + g);
                        const bool sv = (int)slice < p.BH;
#pragma unroll 4
                        for (int it = 0; it < SL / kRowsIt; ++it) {
                            const uint32_t t = (uint32_t)(it * kRowsIt + rsub);
                            const int R = g * SL + (int)t;
                            const bool on = c_data && sv && (int)t < p.Nq;
                            const size_t row = on ? swin_image_row(slice, t, p.H, p.n_w, p.n_ww, p.win, p.grid_h, p.grid_w,
                                                                   p.shift, p.fd_h, p.fd_w, p.fd_ww, p.fd_m)
                                                  : 0;
                            const size_t off = on ? row * rowb + (size_t)c * 16 : 0;
                            const uint32_t dst = smem_u32(b + R * 32) + dchunk +
                                                 ((((uint32_t)c & 1u) ^ (((uint32_t)R >> 2) & 1u)) << 4);
                            const uint32_t nb = on ? 16u : 0u;
                            cp_async16(dst, static_cast<const unsigned char*>(p.q) + off, nb);
                            cp_async16(dst + T::kBytes, static_cast<const unsigned char*>(p.k) + off, nb);
                            cp_async16(dst + 2 * T::kBytes, static_cast<const unsigned char*>(p.v) + off, nb);
                            cp_async16(dst + 3 * T::kBytes, static_cast<const unsigned char*>(p.dout) + off, nb);
                        }
                    }
                }
                cp_async_arrive_noinc(&bar_full[st]);
            }
            cp_async_wait<0>();
        } else if (warp == kProducerWarp && lane == 0) {
            // ============================================================ producer
            const uint32_t tx = 4u * (uint32_t)T::kBytes;
            int u = 0;
            for (int job = job0; job < p.n_jobs; job += job_step, ++u) {
                const int st = u % nst;
                if (u >= nst && !mbar_wait(&bar_empty[st], ((u / nst) + 1) & 1, abort_flag, kStatusWaitEmpty)) break;
                unsigned char* b = sRing + st * p.stage_bytes;
                const int s0 = job * p.g;
                mbar_arrive_expect_tx(&bar_full[st], tx);
                tma_load_4d(b, &tm.q, &bar_full[st], 0, 0, s0, 0);
                tma_load_4d(b + T::kBytes, &tm.k, &bar_full[st], 0, 0, s0, 0);
                tma_load_4d(b + 2 * T::kBytes, &tm.v, &bar_full[st], 0, 0, s0, 0);
                tma_load_4d(b + 3 * T::kBytes, &tm.dout, &bar_full[st], 0, 0, s0, 0);
                if (p.part) {
                    const int po = p.full_atoms * kBlockM * 32;
                    tma_load_3d(b + po, &tm.qp, &bar_full[st], 0, 0, s0);
                    tma_load_3d(b + T::kBytes + po, &tm.kp, &bar_full[st], 0, 0, s0);
                    tma_load_3d(b + 2 * T::kBytes + po, &tm.vp, &bar_full[st], 0, 0, s0);
                    tma_load_3d(b + 3 * T::kBytes + po, &tm.dop, &bar_full[st], 0, 0, s0);
                }
            }
            if (*abort_flag) {
                // let copies still in flight land before the CTA retires
                for (int w = (u > nst ? u - nst : 0); w < u; ++w)
                    mbar_wait(&bar_full[w % nst], (w / nst) & 1, nullptr, 0);
            }
        } else if (warp == kMmaWarp) {
            // ================================================================ MMA
            // the whole warp runs the issue loop; lane 0 issues
            const uint32_t idesc_s = make_idesc_f16(bf, kBlockM, kBlockN, false);
            const uint32_t idesc_g = make_idesc_f16_mn(bf, kBlockM, DPAD, true, true);
            const uint32_t idesc_q = make_idesc_f16_mn(bf, kBlockM, DPAD, false, true);
            const uint32_t aP = smem_u32(sP), aDS = smem_u32(sDS);
            // every lane waits (no warp vote: the lanes run in step)
            auto waitb = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
                if (!mbar_wait(bar, parity, abort_flag, code)) return false;
                tc_fence_after();
                return true;
            };
            // S and dP of tile u (scores, and dO.V^T), once its stage has landed
            // and the softmax has read the last tile's
            auto issue_sdp = [&](int u) -> bool {
                const int st = u % nst;
                const uint32_t b = smem_u32(sRing + st * p.stage_bytes);
                if (!waitb(&bar_full[st], (u / nst) & 1, kStatusWaitK)) return false;
                // image layout: the tiles were written by cp.async (generic proxy)
                if constexpr (kImg) fence_proxy_async_smem();
                if (u > 0 && !waitb(&bar_sfree, (u - 1) & 1, kStatusWaitS)) return false;
                issue_qk<DPAD>(tS, kdesc(b), kdesc(b + T::kBytes), idesc_s);
                issue_qk<DPAD>(tDP, kdesc(b + 3 * T::kBytes), kdesc(b + 2 * T::kBytes), idesc_s);
                mma_commit(&bar_s);
                return true;
            };
            const int n_tiles = job0 < p.n_jobs ? (p.n_jobs - job0 + job_step - 1) / job_step : 0;
            bool ok = n_tiles == 0 || issue_sdp(0);
            for (int t = 0; ok && t < n_tiles; ++t) {
                const int st = t % nst;
                const uint32_t b = smem_u32(sRing + st * p.stage_bytes);
                const uint32_t aQ = b, aK = b + T::kBytes, aDO = b + 3 * T::kBytes;
                // the next tile's S and dP go first, as soon as the softmax has
                // read this tile's: they compute while it forms P and dS, and it
                // works on them while the tensor core runs this tile's gradient
                // products
                if (t + 1 < n_tiles && !issue_sdp(t + 1)) break;
                if (!waitb(&bar_p, t & 1, kStatusWaitP)) break;
                // the accumulators are rewritten once the epilogue has read the last tile's
                if (t > 0 && !waitb(&bar_accfree, (t - 1) & 1, kStatusWaitO)) break;
                // descriptors built once; a step only moves the start-address
                // field (16-byte units): 512 B per 16 rows, kBlockM * 32 B per
                // 16-column block
                const uint64_t dP = vdesc(aP), dSm = vdesc(aDS), dSk = kdesc(aDS);
                const uint64_t dDO = vdesc(aDO), dQm = vdesc(aQ), dKm = vdesc(aK);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)  // dV = P^T.dO over 16 query rows per step
                    mma_ss(tDV, dP + (uint64_t)(ks * 32), dDO + (uint64_t)(ks * 32), idesc_g, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)  // dK = dS^T.Q
                    mma_ss(tDK, dSm + (uint64_t)(ks * 32), dQm + (uint64_t)(ks * 32), idesc_g, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)  // dQ = dS.K over 16 keys per step
                    mma_ss(tDQ, dSk + (uint64_t)(ks * (kBlockM * 32 / 16)), dKm + (uint64_t)(ks * 32), idesc_q,
                           ks > 0 ? 1u : 0u);
                mma_commit(&bar_pfree);
                mma_commit(&bar_acc);
                mma_commit(&bar_empty[st]);
            }
            // every MMA issued has retired before tensor memory is released
            mma_commit(&bar_final);
            mbar_wait(&bar_final, 0, nullptr, 0);
        }
    } else if (warp < 4) {
        regs_inc<kBwdSoftRegs>();
        // ============================================================== softmax
        const int r = tid;                 // tile row == TMEM lane
        const int slot = r / SL, tok = r - slot * SL;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t col0 = (uint32_t)(slot * SL);  // the row's own key columns (uniform per warp)
        int t = 0;
        bool ok = true;
        for (int job = job0; ok && job < p.n_jobs; job += job_step, ++t) {
            const int slice = job * p.g + slot;
            const bool row_ok = tok < p.Nq && slice < p.BH;
            int h = 0, kind = 0;
            if constexpr (BIAS == kBiasSwin)
                swin_slice_info((uint32_t)min(slice, p.BH - 1), p.H, p.n_w, p.n_ww, p.n_wh, p.shift, p.fd_h, p.fd_w,
                                p.fd_ww, h, kind);
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_s, t & 1, abort_flag, kStatusWaitS))) { ok = false; break; }
            tc_fence_after();
            // the row's SL score columns (its own slot); its dP columns are read
            // once P is done, after which S / dP are free for the next tile
            float xs[SL];
            {
                uint32_t v[SL];
                tmem_ld_cols<SL>(tS + lane_base + col0, v);
#pragma unroll
                for (int c = 0; c < SL; ++c) xs[c] = __uint_as_float(v[c]);
            }
            // D = rowsum(dO * O) of the row, from the epilogue warps
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_d[t & 1], (t >> 1) & 1, abort_flag, kStatusWaitV))) {
                ok = false;
                break;
            }
            const float D = sD[t & 1][r];
            // x = scale * s + bias (log2 units); keys past the slice get -inf
            const int nk = p.Nk;
            int pos_q = 0, lab_q = 0, sel = 0;
            if constexpr (BIAS == kBiasSwin) {
                const int tq = s_tok[tok];
                pos_q = (tq & 0xFFFF) + 2 * p.win * (p.win - 1);
                lab_q = tq >> 16;
                sel = ((kind & 1) ? 0x3 : 0) | ((kind & 2) ? 0xC : 0);
            }
            float m = -INFINITY;
            if (BIAS == kBiasSwin && (FAST || p.swin_rows)) {
                // x = s * scale * log2(e) + bias row (-inf past the window; and
                // -100 log2(e) across regions in edge windows)
                const unsigned char* rowp = sRows + (h * SL + tok) * SL * 2;
                const float2 s2 = make_float2(p.scale_log2, p.scale_log2);
                uint4 b4[SL / 8];
#pragma unroll
                for (int q8 = 0; q8 < SL / 8; ++q8)
                    b4[q8] = *reinterpret_cast<const uint4*>(rowp + ((q8 ^ (tok & (SL / 8 - 1) & 7)) << 4));
#pragma unroll
                for (int q8 = 0; q8 < SL / 8; ++q8) {
                    const uint32_t bw[4] = {b4[q8].x, b4[q8].y, b4[q8].z, b4[q8].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = q8 * 8 + 2 * e;
                        const float2 y = __ffma2_rn(make_float2(xs[c], xs[c + 1]), s2,
                                                    __half22float2(*reinterpret_cast<const __half2*>(&bw[e])));
                        xs[c] = y.x;
                        xs[c + 1] = y.y;
                    }
                }
                if (kind) {
                    const uint32_t* mrow = sBits + (kind - 1) * SL * (SL / 32) + tok * (SL / 32);
                    const float mneg = -100.0f * kLog2e;
#pragma unroll
                    for (int wd = 0; wd < SL / 32; ++wd) {
                        const uint32_t mb = mrow[wd];
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if ((mb >> e) & 1u) xs[wd * 32 + e] += mneg;
                    }
                }
#pragma unroll
                for (int c = 0; c < SL; ++c) m = fmaxf(m, xs[c]);
            } else {
#pragma unroll
                for (int c = 0; c < SL; ++c) {
                    float xv = -INFINITY;
                    if (c < nk) {
                        xv = xs[c] * p.scale_log2;
                        if constexpr (BIAS == kBiasSwin) {
                            const int tk = s_tok[c];
                            float bv = sTab[(pos_q - (tk & 0xFFFF)) * p.H + h];
                            if (((tk >> 16) ^ lab_q) & sel) bv -= 100.0f;
                            xv = fmaf(bv, kLog2e, xv);
                        }
                    }
                    xs[c] = xv;
                    m = fmaxf(m, xv);
                }
            }
            const float m_use = m == -INFINITY ? 0.f : m;
            // column pairs through the packed FP32 ops, the row sum in four
            // independent partial sums (128-token slots: one column at a time,
            // which needs fewer registers)
            float l = 0.f;
            if constexpr (SL <= 64) {
                float2 l2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                const float2 nm2 = make_float2(-m_use, -m_use);
#pragma unroll
                for (int c = 0; c < SL; c += 2) {
                    const float2 a = __fadd2_rn(make_float2(xs[c], xs[c + 1]), nm2);
                    xs[c] = ex2_approx(a.x);
                    xs[c + 1] = ex2_approx(a.y);
                    l2[(c >> 1) & 3] = __fadd2_rn(l2[(c >> 1) & 3], make_float2(xs[c], xs[c + 1]));
                }
                const float2 l2s = __fadd2_rn(__fadd2_rn(l2[0], l2[1]), __fadd2_rn(l2[2], l2[3]));
                l = l2s.x + l2s.y;
            } else {
#pragma unroll
                for (int c = 0; c < SL; ++c) {
                    xs[c] = ex2_approx(xs[c] - m_use);
                    l += xs[c];
                }
            }
            // P of the row (zero for rows past the slice or missing slices)
            const float inv_l = (row_ok && l > 0.f) ? 1.0f / l : 0.f;
            if constexpr (SL <= 64) {
                const float2 il2 = make_float2(inv_l, inv_l);
#pragma unroll
                for (int c = 0; c < SL; c += 2) {
                    const float2 y = __fmul2_rn(make_float2(xs[c], xs[c + 1]), il2);
                    xs[c] = y.x;
                    xs[c + 1] = y.y;
                }
            } else {
#pragma unroll
                for (int c = 0; c < SL; ++c) xs[c] *= inv_l;
            }
            constexpr int kDp = SL <= 64 ? SL : 1;
            float dp[kDp];
            if constexpr (SL <= 64) {
                uint32_t v[SL];
                tmem_ld_cols<SL>(tDP + lane_base + col0, v);
#pragma unroll
                for (int c = 0; c < SL; ++c) dp[c] = __uint_as_float(v[c]);
                tc_fence_before();
                warp_arrive(&bar_sfree);
            }
            // the last tile's dV, dK, dQ products must be done with P and dS
            __syncwarp();
            if (t > 0 && !__all_sync(0xffffffffu, mbar_wait(&bar_pfree, (t - 1) & 1, abort_flag, kStatusWaitP))) {
                ok = false;
                break;
            }
            if (BIAS == kBiasSwin && (FAST || p.swin_acc) && t > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(&bar_accsync, (t - 1) & 1, abort_flag, kStatusWaitP))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // dS = P (dP - D) in chunks of up to 64 columns; P and dS go to shared
            // memory as 16-bit A-operand rows, the Swin table gradient collects dS
            constexpr int kCh = SL <= 64 ? SL : 64;
            // one chunk of kCh columns from column ch: dq holds dP on entry
            auto do_chunk = [&](float (&dq)[kCh], int ch) {
                if constexpr (SL <= 64) {
                    const float2 nd2 = make_float2(-D, -D);
#pragma unroll
                    for (int c = 0; c < kCh; c += 2) {
                        const float2 t = __fadd2_rn(make_float2(dq[c], dq[c + 1]), nd2);
                        const float2 y = __fmul2_rn(make_float2(xs[ch + c], xs[ch + c + 1]), t);
                        dq[c] = y.x;
                        dq[c + 1] = y.y;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kCh; ++c) dq[c] = xs[ch + c] * (dq[c] - D);
                }
                if constexpr (BIAS == kBiasSwin) {
                    if ((FAST || p.swin_acc)) {
                        // dS summed per (head, key token, query token): the query
                        // token's own entries, consecutive across the warp's lanes
                        if (row_ok) {
                            float* a = sAcc + (size_t)h * p.Nk * p.Nq + tok;
                            if (!(!FAST && p.swin_acc_atomic)) {
                                // 16 loads, then 16 stores: the entries are distinct
#pragma unroll
                                for (int c0 = 0; c0 < kCh; c0 += 16) {
                                    float o[16];
#pragma unroll
                                    for (int c = 0; c < 16; ++c)
                                        o[c] = (ch + c0 + c < nk) ? a[(ch + c0 + c) * p.Nq] : 0.f;
#pragma unroll
                                    for (int c = 0; c < 16; ++c)
                                        if (ch + c0 + c < nk) a[(ch + c0 + c) * p.Nq] = o[c] + dq[c0 + c];
                                }
                            } else {
#pragma unroll
                                for (int c = 0; c < kCh; ++c)
                                    if (ch + c < nk) atomicAdd(&a[(ch + c) * p.Nq], dq[c]);
                            }
                        }
                    } else if (row_ok) {
                        const int tq = s_tok[tok];
                        const int pq = (tq & 0xFFFF) + 2 * p.win * (p.win - 1);
#pragma unroll
                        for (int c = 0; c < kCh; ++c)
                            if (ch + c < nk) atomicAdd(&sDTab[(pq - (s_tok[ch + c] & 0xFFFF)) * p.H + h], dq[c]);
                    }
                }
                // one loop per operand type, chosen once per chunk (not per pair)
                auto pack_rows = [&](auto b16) {
#pragma unroll
                    for (int c0 = 0; c0 < kCh; c0 += 8) {
                        uint32_t wp[4], wd[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float p0 = xs[ch + c0 + 2 * e], p1 = xs[ch + c0 + 2 * e + 1];
                            const float d0 = dq[c0 + 2 * e], d1 = dq[c0 + 2 * e + 1];
                            wp[e] = decltype(b16)::value ? pack_bf16(p0, p1) : pack_f16(p0, p1);
                            wd[e] = decltype(b16)::value ? pack_bf16(d0, d1) : pack_f16(d0, d1);
                        }
                        const int col = (int)col0 + ch + c0;
                        const uint32_t off = (uint32_t)((col >> 4) * (kBlockM * 32)) + half_off(r, (col >> 3) & 1);
                        *reinterpret_cast<uint4*>(sP + off) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
                        *reinterpret_cast<uint4*>(sDS + off) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    }
                };
                if (bf) pack_rows(std::true_type{});
                else pack_rows(std::false_type{});
            };
            if constexpr (SL <= 64) {
                do_chunk(dp, 0);
            } else {
#pragma unroll
                for (int ch = 0; ch < SL; ch += kCh) {
                    float dq[kCh];
                    uint32_t v[kCh];
                    tmem_ld_cols<kCh>(tDP + lane_base + col0 + (uint32_t)ch, v);
#pragma unroll
                    for (int c = 0; c < kCh; ++c) dq[c] = __uint_as_float(v[c]);
                    do_chunk(dq, ch);
                }
            }
            if constexpr (SL > 64) {
                tc_fence_before();
                warp_arrive(&bar_sfree);
            }
            fence_proxy_async_smem();  // read by the tensor core
            warp_arrive(&bar_p);
            // the next tile may add to the same (head, token) sums from another
            // warp: every warp's additions of this tile come first
            if (BIAS == kBiasSwin && (FAST || p.swin_acc)) warp_arrive(&bar_accsync);
        }
    } else {
        regs_inc<kBwdEpiRegs>();
        // ============================================================= epilogue
        const int r = tid - 128;  // tile row == TMEM lane
        const int slot = r / SL, tok = r - slot * SL;
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        // D = rowsum(dO * O) of tile u's row r (dO from the landed stage, O
        // from global memory) into sD[u & 1], computed two tiles ahead of the
        // softmax that reads it; its buffer was last read by tile u - 2,
        // which finished before that tile's products (waited below) did.
        auto row_d = [&](int u) -> bool {
            const int jb = job0 + u * job_step;
            if (jb >= p.n_jobs) return true;
            const int st = u % nst;
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_full[st], (u / nst) & 1, abort_flag, kStatusWaitK))) return false;
            const unsigned char* sDO = sRing + st * p.stage_bytes + 3 * T::kBytes;
            const int slice = jb * p.g + slot;
            float D = 0.f;
            // one loop per input type
            auto dot_row = [&](auto b16, const uint4* orow) {
#pragma unroll
                for (int c8 = 0; c8 < DPAD / 8; ++c8) {
                    if (c8 * 8 < p.d) {
                        const uint4 ov = orow[c8];
                        const uint4 dv = *reinterpret_cast<const uint4*>(sDO + (c8 >> 1) * (kBlockM * 32) + half_off(r, c8 & 1));
                        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float2 a, c;
                            if constexpr (decltype(b16)::value) {
                                a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
                                c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[e]));
                            } else {
                                a = __half22float2(*reinterpret_cast<const __half2*>(&ow[e]));
                                c = __half22float2(*reinterpret_cast<const __half2*>(&dw[e]));
                            }
                            D = fmaf(a.x, c.x, fmaf(a.y, c.y, D));
                        }
                    }
                }
            };
            if (tok < p.Nq && slice < p.BH) {
                const size_t orow_i = kImg
                                          ? swin_image_row((uint32_t)slice, (uint32_t)tok, p.H, p.n_w, p.n_ww, p.win,
                                                           p.grid_h, p.grid_w, p.shift, p.fd_h, p.fd_w, p.fd_ww, p.fd_m)
                                          : (size_t)slice * p.Nq + tok;
                const uint4* orow = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.o) +
                                                                   orow_i * (size_t)p.d * 2);
                if (bf) dot_row(std::true_type{}, orow);
                else dot_row(std::false_type{}, orow);
            }
            sD[u & 1][r] = D;
            warp_arrive(&bar_d[u & 1]);
            return true;
        };
        bool ok = row_d(0) && row_d(1);
        int t = 0;
        for (int job = job0; ok && job < p.n_jobs; job += job_step, ++t) {
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(&bar_acc, t & 1, abort_flag, kStatusWaitO))) break;
            tc_fence_after();
            const int slice = job * p.g + slot;
            const bool key_ok = tok < p.Nk && slice < p.BH, q_ok = tok < p.Nq && slice < p.BH;
            // dV (x 1), dK (x scale) for key row `tok`, dQ (x scale) for query row `tok`
#pragma unroll 1
            for (int which = 0; which < 3; ++which) {
                uint32_t v[DPAD];
                tmem_ld_cols<DPAD>(lane_base + (which == 0 ? tDV : which == 1 ? tDK : tDQ), v);
                const bool ok_row = which == 2 ? q_ok : key_ok;
                const float f = which == 0 ? 1.0f : p.scale;
                void* base = which == 0 ? p.dv : which == 1 ? p.dk : p.dq;
                const int n = which == 2 ? p.Nq : p.Nk;
                if (ok_row) {
                    const size_t grow = kImg
                                            ? swin_image_row((uint32_t)slice, (uint32_t)tok, p.H, p.n_w, p.n_ww, p.win,
                                                             p.grid_h, p.grid_w, p.shift, p.fd_h, p.fd_w, p.fd_ww, p.fd_m)
                                            : (size_t)slice * n + tok;
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(base) + grow * (size_t)p.d * 2);
                    auto store_row = [&](auto b16) {
#pragma unroll
                        for (int c8 = 0; c8 < DPAD / 8; ++c8) {
                            if (c8 * 8 < p.d) {
                                uint32_t w[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float a = __uint_as_float(v[c8 * 8 + 2 * e]) * f;
                                    const float b = __uint_as_float(v[c8 * 8 + 2 * e + 1]) * f;
                                    w[e] = decltype(b16)::value ? pack_bf16(a, b) : pack_f16(a, b);
                                }
                                dst[c8] = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    };
                    if (bf) store_row(std::true_type{});
                    else store_row(std::false_type{});
                }
            }
            tc_fence_before();
            warp_arrive(&bar_accfree);
            ok = row_d(t + 2);
        }
    }

    // ============================================================== teardown
    tc_fence_before();
    __syncthreads();
    if constexpr (BIAS == kBiasSwin) {
        if (abort_sh == 0) {
            if ((FAST || p.swin_acc)) {
                // each table entry (head, offset (dr, dc)) sums the (key, query)
                // sums of its pairs q = (rq, cq), k = (rq - dr, cq - dc)
                const int M = p.win, N = p.Nq, TT = 2 * M - 1;
                for (int i = tid; i < p.H * TT * TT; i += kBwdThreads) {
                    const int hh = i / (TT * TT), idx = i - hh * (TT * TT);
                    const int dr = idx / TT - (M - 1), dc = idx % TT - (M - 1);
                    const float* a = sAcc + (size_t)hh * N * N;
                    float v = 0.f;
                    for (int rq = max(0, dr); rq < min(M, M + dr); ++rq)
                        for (int cq = max(0, dc); cq < min(M, M + dc); ++cq)
                            v += a[((rq - dr) * M + (cq - dc)) * N + rq * M + cq];
                    sDTab[idx * p.H + hh] += v;
                }
                __syncthreads();
            }
            for (int i = tid; i < n_tab; i += kBwdThreads)
                if (sDTab[i] != 0.f) atomicAdd(&p.d_table[i], sDTab[i]);
        }
    }
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && abort_sh != 0 && p.status) atomicCAS(p.status, 0, abort_sh);
}

}  // namespace sdpa09
