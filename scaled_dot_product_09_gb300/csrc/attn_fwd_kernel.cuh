// attn_fwd_kernel.cuh -- fused scaled-dot-product attention forward for
// GB300 (sm_103a): O = softmax(scale * Q.K^T + bias) . V.
//
// Method: "视觉大模型训练和推理加速" section 一 (attention map from query and
// key through a softmax, weighting the values) computed the memory-efficient
// way the SAM and diffusers pages describe ("PyTorch团队重写「分割一切」模型，
// 比原始实现快8倍", section SDPA: scaled_dot_product_attention; "Accelerated
// Diffusers with PyTorch 2.0", section 加速 Transformer 块): the score matrix
// never leaves the chip; an online softmax (running max and sum) carries the
// row statistics across key tiles.
//
// One CTA owns one 128-row query tile.  Eight warps, specialised:
//   warp 0      TMA producer: Q once, then a ring of K/V stages.
//   warp 1      allocates tensor memory; lane 0 issues every tcgen05.mma.
//   warps 2-3   bias helpers (SAM relative-position prologue).
//   warps 4-7   softmax: thread t owns query row t = TMEM lane t.  They
//               read S from TMEM, add scale and bias, keep the running max
//               and sum, write P (16-bit) back into TMEM over S, rescale O
//               when the max grows by more than 2^8, and run the epilogue.
// Tensor memory (512 columns): S double buffer at columns [0,128) and
// [128,256) (P aliases the first 64 columns of its S buffer), O at
// [256, 256+DPAD).
// Shared memory holds Q, K and V in the 32-byte-swizzled K-major layout the
// TMA writes: DPAD/16 column blocks of 128 rows x 32 bytes.  S = Q.K^T is an
// SS MMA with both operands K-major; O += P.V is a TS MMA with P from TMEM
// and V read MN-major from shared memory.
//
// Two tilings:
//   long   : one slice per CTA, 128 query rows, key loop over 128-key tiles.
//   packed : g whole slices per CTA (g*Nq <= 128, g*Nk <= 128), one key
//            tile, block-diagonal validity (window attention with short
//            windows: Swin's 49-token windows, two per tile).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "sm103_ptx.cuh"

namespace sdpa09 {

constexpr int kThreads = 256;
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr int kTmemO = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow to 2^8 before O is rescaled

enum BiasKind { kBiasNone = 0, kBiasSwin = 1, kBiasSam = 2 };

// Error codes left in the device status word.
enum DevStatus {
    kStatusOk = 0,
    kStatusWaitQ = 1,
    kStatusWaitK = 2,
    kStatusWaitV = 3,
    kStatusWaitS = 4,
    kStatusWaitP = 5,
    kStatusWaitO = 6,
    kStatusWaitEmpty = 7,
    kStatusWaitFinal = 8,
};

struct AttnParams {
    void* out;         // [BH][Nq][d]
    float* dbg;        // debug bias [BH][Nq][Nk] or null
    int* status;       // device status word
    int BH, H, Nq, Nk, d;
    int g;             // slices per tile (packed) or 1 (long)
    int packed;        // 1 = packed tiling
    int n_q_tiles;     // query tiles per slice (long)
    int n_kv_tiles;    // key tiles (long) or 1 (packed)
    int kv_cols;       // N of the S MMA (multiple of 16)
    int box_rows_q;    // rows per Q TMA box
    int box_rows_kv;   // rows per K/V TMA box
    float scale_log2;  // scale * log2(e)
    int is_bf16;
    // Swin
    const float* table;  // [(2M-1)^2][H]
    int win, grid_h, grid_w, shift, n_w, n_ww;
    // SAM
    const void* rel_h;   // [2*s_h-1][d]
    const void* rel_w;   // [2*s_w-1][d]
    const void* q;       // Q again, read by the SAM prologue
    int s_h, s_w;
};

template <int DPAD>
struct KernelCfg {
    static constexpr int kAtoms = DPAD / 16;                 // 16-element column blocks
    static constexpr int kTileBytes = kAtoms * kBlockM * 32; // 128 rows x DPAD x 2 B
    static constexpr int kStages = DPAD <= 64 ? 4 : (DPAD <= 96 ? 3 : 2);
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffExtra = kOffV + kStages * kTileBytes;  // bias scratch
    static_assert(DPAD % 16 == 0 && DPAD >= 16 && DPAD <= 128, "head dim block");
};

// Bias scratch in shared memory (after the tiles).
//   Swin: table for the heads present [(2M-1)^2 * H] (log2 units unless
//         debugging), then per-column info for the key tile [128].
//   SAM : per-row relative terms [128][s_h + s_w + 1] fp32 (natural units),
//         then (kh, kw) of every key [Nk].
__host__ __device__ constexpr int swin_extra_bytes(int table_len) {
    return (table_len + kBlockN) * 4;
}
__host__ __device__ constexpr int sam_extra_bytes(int s_h, int s_w, int n_keys) {
    return (kBlockM * (s_h + s_w + 1) + n_keys) * 4;
}

__device__ __forceinline__ int swin_strip(int pos, int G, int M, int s) {
    return pos < G - M ? 0 : (pos < G - s ? 1 : 2);
}

__device__ __forceinline__ float to_float(const void* base, size_t idx, int is_bf16) {
    if (is_bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return __half2float(reinterpret_cast<const __half*>(base)[idx]);
}

template <int DPAD, int BIAS, bool DBG>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
    using Cfg = KernelCfg<DPAD>;
    constexpr int NST = Cfg::kStages;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sQ = smem + Cfg::kOffQ;
    unsigned char* sK = smem + Cfg::kOffK;
    unsigned char* sV = smem + Cfg::kOffV;
    float* sExtra = reinterpret_cast<float*>(smem + Cfg::kOffExtra);

    __shared__ uint64_t bar_q, bar_o, bar_o_final, bar_mma_final;
    __shared__ uint64_t bar_k[NST], bar_v[NST], bar_empty[NST];
    __shared__ uint64_t bar_s[2], bar_p[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int* abort_flag = &abort_sh;

    // ------------------------------------------------------------ tile --
    const int tile = blockIdx.x;
    int slice0, q_row0, rows_valid;
    if (p.packed) {
        slice0 = tile * p.g;
        q_row0 = 0;
        const int ns = min(p.g, p.BH - slice0);
        rows_valid = ns * p.Nq;
    } else {
        slice0 = tile / p.n_q_tiles;
        q_row0 = (tile % p.n_q_tiles) * kBlockM;
        rows_valid = min(kBlockM, p.Nq - q_row0);
    }
    const int n_kv = p.n_kv_tiles;

    // ------------------------------------------------------------ setup --
    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_q, 1);
        mbar_init(&bar_o, 1);
        mbar_init(&bar_o_final, 1);
        mbar_init(&bar_mma_final, 1);
        for (int i = 0; i < NST; ++i) {
            mbar_init(&bar_k[i], 1);
            mbar_init(&bar_v[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_s[i], 1);
            mbar_init(&bar_p[i], kBlockM);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (p.packed) {
        // Boxes shorter than 128 rows leave the tail rows of each block
        // untouched; zero them once so the MMAs read finite values there.
        const int total = Cfg::kOffExtra / 16;
        uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = tid; i < total; i += kThreads) reinterpret_cast<uint4*>(smem)[i] = z;
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    // Bias tables into shared memory.
    if constexpr (BIAS == kBiasSwin) {
        const int tl = (2 * p.win - 1) * (2 * p.win - 1);
        const float f = DBG ? 1.0f : kLog2e;
        // stored head-major: [h][idx]
        for (int i = tid; i < tl * p.H; i += kThreads) {
            const int idx = i / p.H, h = i % p.H;
            sExtra[h * tl + idx] = p.table[i] * f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    const int q_atom_bytes = p.box_rows_q * 32;
    const int kv_atom_bytes = p.box_rows_kv * 32;

    if (warp == 0) {
        // ====================================================== producer ==
        if (lane == 0) {
            int z_q = slice0;
            mbar_arrive_expect_tx(&bar_q, Cfg::kAtoms * q_atom_bytes);
            for (int a = 0; a < Cfg::kAtoms; ++a) {
                if (p.packed)
                    tma_load_2d(sQ + a * kBlockM * 32, &tm_q, &bar_q, a * 16, slice0 * p.Nq);
                else
                    tma_load_3d(sQ + a * kBlockM * 32, &tm_q, &bar_q, a * 16, q_row0, z_q);
            }
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % NST;
                if (j >= NST) {
                    if (!mbar_wait(&bar_empty[st], ((j / NST) + 1) & 1, abort_flag, kStatusWaitEmpty)) break;
                }
                unsigned char* dk = sK + st * Cfg::kTileBytes;
                unsigned char* dv = sV + st * Cfg::kTileBytes;
                mbar_arrive_expect_tx(&bar_k[st], Cfg::kAtoms * kv_atom_bytes);
                for (int a = 0; a < Cfg::kAtoms; ++a) {
                    if (p.packed)
                        tma_load_2d(dk + a * kBlockN * 32, &tm_k, &bar_k[st], a * 16, slice0 * p.Nk);
                    else
                        tma_load_3d(dk + a * kBlockN * 32, &tm_k, &bar_k[st], a * 16, j * kBlockN, slice0);
                }
                mbar_arrive_expect_tx(&bar_v[st], Cfg::kAtoms * kv_atom_bytes);
                for (int a = 0; a < Cfg::kAtoms; ++a) {
                    if (p.packed)
                        tma_load_2d(dv + a * kBlockN * 32, &tm_v, &bar_v[st], a * 16, slice0 * p.Nk);
                    else
                        tma_load_3d(dv + a * kBlockN * 32, &tm_v, &bar_v[st], a * 16, j * kBlockN, slice0);
                }
                issued = j + 1;
            }
            if (*abort_flag) {
                // Let copies still in flight land before the CTA retires.
                mbar_wait(&bar_q, 0, nullptr, 0);
                for (int j = max(0, issued - NST); j < issued; ++j) {
                    const int st = j % NST;
                    mbar_wait(&bar_k[st], (j / NST) & 1, nullptr, 0);
                    mbar_wait(&bar_v[st], (j / NST) & 1, nullptr, 0);
                }
            }
        }
    } else if (warp == 1) {
        // ========================================================= MMA ==
        if (lane == 0) {
            const bool bf = p.is_bf16 != 0;
            const uint32_t idesc_s = make_idesc_f16(bf, kBlockM, p.kv_cols, false);
            const uint32_t idesc_o = make_idesc_f16(bf, kBlockM, DPAD, true);
            const int kv_steps = p.kv_cols / 16;
            bool ok = mbar_wait(&bar_q, 0, abort_flag, kStatusWaitQ);
            auto issue_s = [&](int j) -> bool {
                const int st = j % NST;
                if (!mbar_wait(&bar_k[st], (j / NST) & 1, abort_flag, kStatusWaitK)) return false;
                tc_fence_after();
                const uint32_t qa = smem_u32(sQ);
                const uint32_t ka = smem_u32(sK + st * Cfg::kTileBytes);
                const uint32_t d_tmem = tmem + (j & 1) * kBlockN;
#pragma unroll
                for (int ks = 0; ks < Cfg::kAtoms; ++ks) {
                    const uint64_t da = make_sdesc(qa + ks * kBlockM * 32, 16, 256, kSwizzle32B);
                    const uint64_t db = make_sdesc(ka + ks * kBlockN * 32, 16, 256, kSwizzle32B);
                    mma_ss(d_tmem, da, db, idesc_s, ks > 0 ? 1u : 0u);
                }
                mma_commit(&bar_s[j & 1]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) {
                    if (!issue_s(j + 1)) break;
                }
                if (!mbar_wait(&bar_p[j & 1], (j >> 1) & 1, abort_flag, kStatusWaitP)) break;
                const int st = j % NST;
                if (!mbar_wait(&bar_v[st], (j / NST) & 1, abort_flag, kStatusWaitV)) break;
                tc_fence_after();
                const uint32_t va = smem_u32(sV + st * Cfg::kTileBytes);
                const uint32_t p_tmem = tmem + (j & 1) * kBlockN;
                for (int ks = 0; ks < kv_steps; ++ks) {
                    // V: MN-major, 32-byte swizzle; 16 keys = 512 bytes per step,
                    // column blocks of 16 dims are kBlockN*32 bytes apart.
                    const uint64_t db = make_sdesc(va + ks * 512, kBlockN * 32, 256, kSwizzle32B);
                    mma_ts(tmem + kTmemO, p_tmem + ks * 8, db, idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(&bar_empty[st]);
                mma_commit(&bar_o);
                if (j == n_kv - 1) mma_commit(&bar_o_final);
            }
            // Every MMA this thread issued has retired before TMEM is freed.
            mma_commit(&bar_mma_final);
            mbar_wait(&bar_mma_final, 0, nullptr, 0);
        }
    } else if (warp >= kSoftmaxWarp0) {
        // ===================================================== softmax ==
        const int r = tid - kSoftmaxWarp0 * 32;              // row in tile == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const bool row_ok = r < rows_valid;
        int my_slice, my_tok, my_sl;
        if (p.packed) {
            my_sl = r / p.Nq;
            my_slice = slice0 + my_sl;
            my_tok = r - my_sl * p.Nq;
        } else {
            my_sl = 0;
            my_slice = slice0;
            my_tok = q_row0 + r;
        }
        // ---- bias row setup
        const float* swin_tab = nullptr;
        int swin_row_base = 0, swin_lab = 0;
        int* col_info = nullptr;
        float mask_val = DBG ? -100.0f : -100.0f * kLog2e;
        if constexpr (BIAS == kBiasSwin) {
            const int M = p.win, tl = (2 * M - 1) * (2 * M - 1);
            col_info = reinterpret_cast<int*>(sExtra + tl * p.H);
            const int h = my_slice % p.H;
            swin_tab = sExtra + h * tl;
            const int ri = my_tok / M, ci = my_tok % M;
            swin_row_base = (ri + M - 1) * (2 * M - 1) + (ci + M - 1);
            const int w = (my_slice / p.H) % p.n_w;
            const int y = (w / p.n_ww) * M + ri, x = (w % p.n_ww) * M + ci;
            swin_lab = p.shift ? swin_strip(y, p.grid_h, M, p.shift) * 3 + swin_strip(x, p.grid_w, M, p.shift) : 0;
            // column info of the (single) key tile: key offset, region, slice
            {
                const int c = r;
                const int sl = c / p.Nk;
                const int slice = slice0 + sl;
                const int t = c - sl * p.Nk;
                const int rj = t / M, cj = t % M;
                const int wk = (slice / p.H) % p.n_w;
                const int yk = (wk / p.n_ww) * M + rj, xk = (wk % p.n_ww) * M + cj;
                const int lab = p.shift ? swin_strip(yk, p.grid_h, M, p.shift) * 3 + swin_strip(xk, p.grid_w, M, p.shift) : 0;
                const int valid = (sl < p.g) ? 1 : 0;
                col_info[c] = (rj * (2 * M - 1) + cj) | (lab << 16) | ((valid ? sl : 255) << 20);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        float* sam_rel = nullptr;
        int* sam_col = nullptr;
        int sam_qh = 0, sam_qw = 0;
        if constexpr (BIAS == kBiasSam) {
            const int sh = p.s_h, sw = p.s_w, rs = sh + sw + 1;
            sam_rel = sExtra + r * rs;
            sam_col = reinterpret_cast<int*>(sExtra + kBlockM * rs);
            // (kh, kw) of every key, shared by all rows
            for (int key = r; key < p.Nk; key += kBlockM) sam_col[key] = (key / sw) | ((key % sw) << 16);
            sam_qh = my_tok / sw;
            sam_qw = my_tok % sw;
            if (row_ok) {
                // rel_h[kh] = Q_i . R_h[qh-kh+sh-1], rel_w[kw] = Q_i . R_w[qw-kw+sw-1]
                const size_t qoff = ((size_t)my_slice * p.Nq + my_tok) * p.d;
                float qv[DPAD];
#pragma unroll
                for (int c = 0; c < DPAD; ++c) qv[c] = c < p.d ? to_float(p.q, qoff + c, p.is_bf16) : 0.f;
                for (int kh = 0; kh < sh; ++kh) {
                    const size_t ro = (size_t)(sam_qh - kh + sh - 1) * p.d;
                    float acc = 0.f;
#pragma unroll
                    for (int c = 0; c < DPAD; ++c) acc += c < p.d ? qv[c] * to_float(p.rel_h, ro + c, p.is_bf16) : 0.f;
                    sam_rel[kh] = acc;
                }
                for (int kw = 0; kw < sw; ++kw) {
                    const size_t ro = (size_t)(sam_qw - kw + sw - 1) * p.d;
                    float acc = 0.f;
#pragma unroll
                    for (int c = 0; c < DPAD; ++c) acc += c < p.d ? qv[c] * to_float(p.rel_w, ro + c, p.is_bf16) : 0.f;
                    sam_rel[sh + kw] = acc;
                }
            } else {
                for (int t = 0; t < sh + sw; ++t) sam_rel[t] = 0.f;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }

        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            __syncwarp();
            if (!mbar_wait(&bar_s[j & 1], (j >> 1) & 1, abort_flag, kStatusWaitS)) { ok = false; break; }
            tc_fence_after();
            const uint32_t s_tmem = tmem + lane_base + (j & 1) * kBlockN;
            float x[kBlockN];
#pragma unroll
            for (int c0 = 0; c0 < kBlockN; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(s_tmem + c0, v);
#pragma unroll
                for (int t = 0; t < 32; ++t) x[c0 + t] = __uint_as_float(v[t]);
            }
            const int key0 = j * kBlockN;
            float m_tile = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) {
                bool valid;
                float b = 0.f;
                if (p.packed) {
                    valid = c < p.kv_cols;
                } else {
                    valid = key0 + c < p.Nk;
                }
                if constexpr (BIAS == kBiasSwin) {
                    const int info = col_info[c];
                    valid = valid && ((info >> 20) == my_sl);
                    const int idx = swin_row_base - (info & 0xFFFF);
                    b = valid ? swin_tab[idx] + ((((info >> 16) & 15) == swin_lab) ? 0.f : mask_val) : 0.f;
                } else if constexpr (BIAS == kBiasSam) {
                    const int ci = sam_col[min(key0 + c, p.Nk - 1)];
                    b = valid ? (sam_rel[ci & 0xFFFF] + sam_rel[p.s_h + (ci >> 16)]) : 0.f;
                } else {
                    if (p.packed) valid = valid && (c / p.Nk == my_sl);
                }
                if constexpr (DBG) {
                    if (valid && row_ok) {
                        const int key = p.packed ? (c - my_sl * p.Nk) : (key0 + c);
                        p.dbg[((size_t)my_slice * p.Nq + my_tok) * p.Nk + key] = b;
                    }
                }
                float xv;
                if constexpr (BIAS == kBiasSam) {
                    xv = fmaf(x[c], p.scale_log2, b * kLog2e);
                } else if constexpr (BIAS == kBiasSwin && DBG) {
                    xv = fmaf(x[c], p.scale_log2, b * kLog2e);
                } else {
                    xv = fmaf(x[c], p.scale_log2, b);
                }
                x[c] = valid ? xv : -INFINITY;
                m_tile = fmaxf(m_tile, x[c]);
            }
            const float m_new = fmaxf(m_run, m_tile);
            const bool need = m_new > m_run + kRescaleThreshold;
            const bool warp_need = __any_sync(0xffffffffu, need && j > 0);
            if (warp_need) {
                // O must hold P_{j-1}.V_{j-1} before it is rescaled.
                if (!mbar_wait(&bar_o, (j - 1) & 1, abort_flag, kStatusWaitO)) { ok = false; break; }
                tc_fence_after();
                const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
#pragma unroll
                for (int c0 = 0; c0 < DPAD; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_base + kTmemO + c0, v);
#pragma unroll
                    for (int t = 0; t < 16; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
                    tmem_st16(tmem + lane_base + kTmemO + c0, v);
                }
            }
            if (need) {
                l_run *= ex2_approx(m_run - m_new);
                m_run = m_new;
            }
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            float lsum = 0.f;
            uint32_t pk[kBlockN / 2];
#pragma unroll
            for (int c = 0; c < kBlockN; c += 2) {
                const float p0 = ex2_approx(x[c] - m_use);
                const float p1 = ex2_approx(x[c + 1] - m_use);
                lsum += p0 + p1;
                pk[c / 2] = p.is_bf16 ? pack_bf16(p0, p1) : pack_f16(p0, p1);
            }
            l_run += lsum;
#pragma unroll
            for (int c0 = 0; c0 < kBlockN / 2; c0 += 16) {
                uint32_t v[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) v[t] = pk[c0 + t];
                tmem_st16(s_tmem + c0, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_p[j & 1]);
        }
        // ---------------------------------------------------- epilogue --
        if (ok && mbar_wait(&bar_o_final, 0, abort_flag, kStatusWaitO)) {
            tc_fence_after();
            const float inv_l = l_run > 0.f ? 1.0f / l_run : 0.f;
            uint32_t o[DPAD / 2];
#pragma unroll
            for (int c0 = 0; c0 < DPAD; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + lane_base + kTmemO + c0, v);
#pragma unroll
                for (int t = 0; t < 16; t += 2) {
                    const float a = __uint_as_float(v[t]) * inv_l;
                    const float b = __uint_as_float(v[t + 1]) * inv_l;
                    o[(c0 + t) / 2] = p.is_bf16 ? pack_bf16(a, b) : pack_f16(a, b);
                }
            }
            if (row_ok && !DBG) {
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(p.out) +
                                                      (((size_t)my_slice * p.Nq + my_tok) * p.d) * 2);
#pragma unroll
                for (int c = 0; c < DPAD / 8; ++c)
                    if (c * 8 < p.d) dst[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            }
        }
    }

    // ------------------------------------------------------------ teardown --
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && abort_sh != 0 && p.status) atomicCAS(p.status, 0, abort_sh);
}

}  // namespace sdpa09
