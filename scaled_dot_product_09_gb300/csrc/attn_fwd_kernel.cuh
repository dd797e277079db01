// attn_fwd_kernel.cuh -- fused scaled-dot-product attention forward for
// GB300 (sm_103a): O = softmax(scale * Q.K^T + bias) . V.
//
// Method: "视觉大模型训练和推理加速" section 一 (attention map from query and
// key through a softmax, weighting the values), computed the memory-efficient
// way the SAM and diffusers pages describe ("PyTorch团队重写「分割一切」模型，
// 比原始实现快8倍", section SDPA: scaled_dot_product_attention; "Accelerated
// Diffusers with PyTorch 2.0", section 加速 Transformer 块): the score matrix
// never leaves the chip; an online softmax (running max and sum) carries the
// row statistics across key tiles.
//
// Persistent kernel, one CTA per SM, twelve warps (three warpgroups):
//   warps 0-3   softmax slot A: thread t owns query row t of tile A (TMEM lane t)
//   warps 4-7   softmax slot B: the same for tile B
//   warp 8      TMA producer
//   warp 9      tensor-memory allocator; lane 0 issues slot A's tcgen05.mma
//   warp 10     lane 0 issues slot B's tcgen05.mma
//   warp 11     idle
// While one slot runs its softmax the tensor core works on the other slot's
// products.  After setup the softmax warpgroups grow to kSoftmaxRegs registers
// and the control warpgroup shrinks to kControlRegs; the split adds up exactly
// to the launch allocation.
//
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A [256,384),
// O_B [384,512).  P (16-bit) overwrites the first 64 columns of its S buffer
// and feeds the P.V MMA straight from TMEM.
//
// Shared-memory operand tiles are 32-byte-swizzled K-major blocks (16-column
// blocks of R rows x 32 bytes) as the TMA writes them.  S = Q.K^T: both
// operands K-major.  O += P.V: V read MN-major.
//
// Job modes:
//   shared   : a job is 256 query rows of one slice (A = first 128, B = next
//              128); both slots consume the same K/V ring (long sequences,
//              SAM windows of 196 tokens).  With the SAM bias each job first
//              passes the rel-pos tables R_w, R_h through the ring; the tensor
//              core forms G_w = Q.R_w^T and G_h = Q.R_h^T, from which every
//              row gathers its decomposed relative terms.
//   separate : a job is two packed tiles; a tile holds 128/SL whole slices,
//              one per SL-row slot (short windows: two 49-token Swin windows
//              in 64-row slots), and brings its own Q, K and V.  A warp's
//              rows all lie in one slot, so it only reads that slot's SL key
//              columns.  The Swin bias is added by the tensor core: with Qone
//              the one-hot code of each row's window token, Qone.E_h^T adds
//              the per-head relative-position block E_h[t_q][t_k] =
//              table[idx(t_q,t_k), h] / scale and Qone.M^T the shifted-window
//              mask block of the window's kind (interior, last row, last
//              column, corner), both built once per CTA in shared memory.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "sm103_ptx.cuh"

namespace sdpa09 {

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 208;
constexpr int kControlRegs = 88;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs == kThreads * kLaunchRegs,
              "register split must add up to the launch allocation");
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kGatherWarp = 11;  // second copy warp of the image-layout Swin gather, else idle
constexpr int kTmemCols = 512;
constexpr int kMaxStages = 8;
constexpr int kSamMaxSide = 64;  // rel-pos grids up to 64 x 64
constexpr float kLog2e = 1.4426950408889634f;
// SAM on the 64 x 64 grid: shared-memory extra area = rel_h rows (fp16,
// [2 slots][64][128])
constexpr uint32_t kSamDbsExtra = 2 * 64 * 128 * 2;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may reach 2^8 before O is rescaled

enum BiasKind { kBiasNone = 0, kBiasSwin = 1, kBiasSam = 2 };
enum JobMode { kModeShared = 0, kModeSeparate = 1 };

// Codes left in the device status word when a bounded wait runs out.
enum DevStatus {
    kStatusOk = 0,
    kStatusWaitQ = 1,
    kStatusWaitK = 2,
    kStatusWaitV = 3,
    kStatusWaitS = 4,
    kStatusWaitP = 5,
    kStatusWaitO = 6,
    kStatusWaitEmpty = 7,
    kStatusWaitG = 8,
    kStatusWaitSelfTest = 9,  // the bounded-wait self-test kernel
};

struct AttnParams {
    void* out;        // [BH][Nq][d]
    float* lse;       // [BH][Nq] natural-log row log-sum-exp, or null (not written)
    float* dbg;       // debug bias [BH][Nq][Nk] or null
    int* status;      // device status word
    int BH, H, Nq, Nk, d;
    int n_jobs;       // jobs of the grid-stride loop
    int n_kv;         // key tiles per job (shared mode)
    int kv_w;         // keys advanced per key tile (shared mode)
    int kv_cols;      // N of the S MMA, multiple of 16, <= 128
    int q_jobs;       // 256-row jobs per slice (shared mode)
    int g;            // slices per packed tile (separate mode)
    int nst;          // ring stages
    int nq;           // Q buffers per slot (shared mode): 1 or 2
    int box_q, box_kv;
    int full_atoms;   // 16-column blocks fully inside d
    int part;         // 1 when d is not a multiple of 16 (one partial block)
    uint32_t off_q, off_ring, off_extra;  // shared-memory offsets (bytes)
    uint32_t ring_stage_bytes;
    float scale;
    float scale_log2;
    int is_bf16;
    // Swin
    const float* table;  // [(2M-1)^2][H]
    int win, grid_h, grid_w, shift, n_w, n_ww, n_wh;
    uint32_t fd_h[2], fd_w[2], fd_ww[2];  // magic/shift pairs dividing by H, n_w, n_ww
    int swin_rows;  // 1: bias rows in shared memory, added by the softmax; 0: added by MMAs
    int swin_image;                 // 1: q/k/v/out in image layout [images][grid_h][grid_w][H][d]
    uint32_t fd_m[2];               // magic/shift pair dividing by win
    const void *q, *k, *v;          // operand bases (image layout gathers them directly)
    // SAM
    int s_h, s_w, n_rh, n_rw;  // query grid; MMA widths of the R_h / R_w tables as given
    int k_h, k_w;              // key grid (the query grid unless general)
    // General SAM (unequal query and key grids, which the host sends to the
    // generic kernel): per axis the float32 coordinate scalers of the query
    // and key coordinates and the offset, the table length as given and the
    // length the index addresses (2 * max(q, k) - 1)
    int sam_general;
    float sam_qs_h, sam_ks_h, sam_off_h, sam_qs_w, sam_ks_w, sam_off_w;
    int sam_lin_h, sam_lout_h, sam_lin_w, sam_lout_w;
    // Equal grids, tables of another length: each CTA resamples both tables
    // once into shared memory at off_rtab (R_w' then R_h', one K-major tile
    // each), and the G MMAs read them there instead of from the ring.
    int sam_resample;
    uint32_t off_rtab;
    const void *rel_h, *rel_w;
};

// Variable-length batches (no bias, shared tiling): Q/O are the concatenation
// over sequences s of [H][Lq_s][d] and K/V of [H][Lk_s][d] -- the buffer of a
// nested tensor of (B, H, N*, d) -- and each sequence attends to itself only
// ("PyTorch团队重写「分割一切」模型" on Nested Tensor: data of non-uniform
// size, e.g. images of different sizes, batched in one tensor).  The table
// travels by value with the launch.  Its entries are the sequences that have
// queries, longest key range first, so that the CTAs' round-robin share of
// the jobs comes out even (longest-processing-time order).
constexpr int kVarlenMaxSeq = 128;
struct VarlenTable {
    int n_seq;                      // entries
    int jobs_end[kVarlenMaxSeq];    // jobs of entries 0..s; an entry has H * ceil(Lq / 256)
    int q_off[kVarlenMaxSeq];       // first token of the entry's sequence in Q/O
    int q_len[kVarlenMaxSeq];       // and its query count (>= 1)
    int k_off[kVarlenMaxSeq];       // first token in K/V
    int k_len[kVarlenMaxSeq];       // key count (>= 1)
};
template <bool VL>
struct VarlenArg {
    int unused;
};
template <>
struct VarlenArg<true> : VarlenTable {};

// Rows of one shared-tiling job: TMA coordinates (row, slice) of its first
// query row (slot A) and of its key row 0, the row of its slice's token 0 in
// the output viewed as [rows][d], its query and key counts and key tiles.
struct JobRows {
    int q_row, q_slice, k_row, k_slice;
    int out_row0;  // output row of token 0 of the job's (sequence, head) slice
    int q0;        // token of the job's first query row within the slice
    int nq, nk, n_kv;
};
template <bool VL>
__device__ __forceinline__ JobRows shared_job(const AttnParams& p, const VarlenArg<VL>& vt, int job) {
    JobRows j;
    if constexpr (!VL) {
        const int slice = job / p.q_jobs;
        j.q0 = (job - slice * p.q_jobs) * 2 * kBlockM;
        j.q_row = j.q0;
        j.q_slice = slice;
        j.k_row = 0;
        j.k_slice = slice;
        j.out_row0 = slice * p.Nq;
        j.nq = p.Nq;
        j.nk = p.Nk;
        j.n_kv = p.n_kv;
    } else {
        // the entry: the first whose job range ends past `job`
        int lo = 0, hi = vt.n_seq - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (vt.jobs_end[mid] > job) hi = mid;
            else lo = mid + 1;
        }
        const int s = lo;
        const int local = job - (s > 0 ? vt.jobs_end[s - 1] : 0);
        const int lq = vt.q_len[s];
        const int lk = vt.k_len[s];
        const int nqb = (lq + 2 * kBlockM - 1) / (2 * kBlockM);
        const int h = local / nqb;
        j.q0 = (local - h * nqb) * 2 * kBlockM;
        j.out_row0 = p.H * vt.q_off[s] + h * lq;
        j.q_row = j.out_row0 + j.q0;
        j.q_slice = 0;
        j.k_row = p.H * vt.k_off[s] + h * lk;
        j.k_slice = 0;
        j.nq = lq;
        j.nk = lk;
        j.n_kv = (lk + p.kv_w - 1) / p.kv_w;
    }
    return j;
}

// Shared memory after the ring ("extra"):
//   Swin (separate mode, slot SL), rows variant: per head an fp32 bias matrix
//        [SL query tokens][SL key tokens] (16-byte chunks of a row XOR-swizzled
//        by the row's low 3 bits), then region-difference bits
//        [3 window kinds][SL query tokens][SL / 32 words]
//   Swin, MMA variant: Qone [128 rows][SL] then H + 3 bias blocks
//        [SL][SL] (per-head tables, then last-column / last-row / corner
//        masks), all 16-bit K-major 32B-swizzled
//   SAM : rel_h [2 slots][k_h][128] fp32, then for generic grids rel_w
//        [2][k_w][128] and a key table [Nk] (k_h x k_w: the key grid)
__host__ __device__ constexpr uint32_t swin_rows_extra_bytes(int sl, int H) {
    return (uint32_t)(H * sl * sl * 4 + 3 * sl * (sl / 32) * 4);
}
__host__ __device__ constexpr uint32_t swin_extra_bytes(int sl, int H) {
    return (uint32_t)(128 * sl * 2 + (H + 3) * sl * sl * 2);
}
__host__ __device__ constexpr uint32_t sam_extra_floats(bool generic, int s_h, int s_w, int nk) {
    return 2u * (uint32_t)s_h * kBlockM + (generic ? 2u * (uint32_t)s_w * kBlockM + (uint32_t)nk : 0u);
}

// TMA descriptors.  Data maps view a [slices][rows][d] tensor as
// (16 elements, row, slice, column block) so that one copy brings every full
// 16-column block of a tile, landing as [block][row][16] (the 32B-swizzled
// K-major layout); the *p maps cover a last partial block when d is not a
// multiple of 16.  Rel-pos maps view [rows][d] as (16, row, block).
struct TmaMaps {
    CUtensorMap q, k, v, qp, kp, vp, rh, rw, rhp, rwp;
};

template <int DPAD>
struct Tile {
    static constexpr int kAtoms = DPAD / 16;
    static constexpr int kBytes = kAtoms * kBlockM * 32;  // 128 rows x DPAD x 2 B
    static_assert(DPAD % 16 == 0 && DPAD >= 16 && DPAD <= 128, "head dim block");
};

// Unsigned division by a divisor fixed at launch: q = (umulhi(n, m) + n) >> s
// with the magic number m and shift s the host derives (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994);
// valid for n < 2^31.
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const uint32_t (&fd)[2]) {
    return (__umulhi(n, fd[0]) + n) >> fd[1];
}

// Head and window kind (0 interior, 1 last window column, 2 last window row,
// 3 corner; 0 for every window without a shift) of a Swin slice: slices run
// head-fastest over windows numbered row-major within each image.
__device__ __forceinline__ void swin_slice_info(uint32_t slice, int H, int n_w, int n_ww, int n_wh, int shift,
                                                const uint32_t (&fd_h)[2], const uint32_t (&fd_w)[2],
                                                const uint32_t (&fd_ww)[2], int& h, int& kind) {
    const uint32_t bimg = fast_div(slice, fd_h);
    h = (int)(slice - bimg * (uint32_t)H);
    const uint32_t w = bimg - fast_div(bimg, fd_w) * (uint32_t)n_w;
    const uint32_t wr = fast_div(w, fd_ww);
    const uint32_t wc = w - wr * (uint32_t)n_ww;
    kind = shift ? (((int)wc == n_ww - 1 ? 1 : 0) | ((int)wr == n_wh - 1 ? 2 : 0)) : 0;
}

// Image-layout row of token t of Swin slice `slice`: the slice's window
// (wr, wc) and head h, token (r, c) = (t / win, t % win) of that window, taken
// from image position ((wr*win + r + shift) mod grid_h, (wc*win + c + shift)
// mod grid_w) -- the cyclic shift and window partition of "视觉大模型训练和推理
// 加速" section 一, as index mapping (section 二).  Rows are [image][y][x][head].
__device__ __forceinline__ size_t swin_image_row(uint32_t slice, uint32_t t, int H, int n_w, int n_ww, int win,
                                                 int grid_h, int grid_w, int shift, const uint32_t (&fd_h)[2],
                                                 const uint32_t (&fd_w)[2], const uint32_t (&fd_ww)[2],
                                                 const uint32_t (&fd_m)[2]) {
    const uint32_t bimg = fast_div(slice, fd_h);
    const int h = (int)(slice - bimg * (uint32_t)H);
    const uint32_t img = fast_div(bimg, fd_w);
    const uint32_t w = bimg - img * (uint32_t)n_w;
    const uint32_t wr = fast_div(w, fd_ww);
    const int wc = (int)(w - wr * (uint32_t)n_ww);
    const uint32_t r = fast_div(t, fd_m);
    const int c = (int)(t - r * (uint32_t)win);
    int y = (int)wr * win + (int)r + shift;
    if (y >= grid_h) y -= grid_h;
    int x = wc * win + c + shift;
    if (x >= grid_w) x -= grid_w;
    return ((size_t)(img * (uint32_t)grid_h + (uint32_t)y) * (size_t)grid_w + (size_t)x) * (size_t)H + (size_t)h;
}

__device__ __forceinline__ int swin_strip(int pos, int G, int M, int s) {
    return pos < G - M ? 0 : (pos < G - s ? 1 : 2);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Byte offset of element (row, k) in a K-major 32B-swizzled block of `rows`
// rows: 16-column blocks of rows x 32 bytes; inside a 32-byte row the two
// 16-byte halves swap on rows 4-7 of every 8 (the TMA/MMA 32B swizzle).
__device__ __forceinline__ uint32_t kmajor_offset(int rows, int row, int k) {
    return (uint32_t)((k >> 4) * rows * 32 + row * 32 + ((((k >> 3) & 1) ^ ((row >> 2) & 1)) << 4) +
                      (k & 7) * 2);
}

__device__ __forceinline__ uint16_t to_half_bits(float v, bool bf16) {
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

// Eight consecutive K-elements of a K-major row, rounded to the operand type,
// as one 16-byte shared-memory store.
__device__ __forceinline__ void store_half8(unsigned char* dst, const float* v, bool bf16) {
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
        w[u] = (uint32_t)to_half_bits(v[2 * u], bf16) | ((uint32_t)to_half_bits(v[2 * u + 1], bf16) << 16);
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Eight columns t0..t0+7 of row j (a key token) of a Swin table block:
// column t holds table[idx(t, j), h] * f, idx the relative-position index
// ("视觉大模型训练和推理加速" section 一, relative position bias):
// (dr + M - 1)(2M - 1) + (dc + M - 1) with dr, dc the row / column offsets of
// query token t from key token j, i.e. pos(t) - pos(j) + (M - 1)(2M) with
// pos(t) = r_t (2M - 1) + c_t. tok[] holds pos in its low 16 bits. The eight
// gathers are issued together; out-of-window entries are zeroed afterwards.
__device__ __forceinline__ void swin_table_group(unsigned char* dst, const float* tab, const int* tok, int t0,
                                                 int pos_j, bool key_ok, int h, int H, int M, int N, float f,
                                                 bool bf16) {
    const int c0 = 2 * M * (M - 1) - pos_j;
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = (key_ok && t0 + u < N) ? (tok[t0 + u] & 0xFFFF) + c0 : 0;
        v[u] = tab[idx * H + h];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = (key_ok && t0 + u < N) ? v[u] * f : 0.f;
    store_half8(dst, v, bf16);
}

// Barrel shift of a 128-entry register row: afterwards v[u] = v_in[u + sh]
// for every u with u + sh < 128 (0 <= sh < 128).  Unrolled selects keep the
// row in registers.
template <int W = 128, int BITS = 7>
__device__ __forceinline__ void shift_down(float (&v)[W], int sh) {
    // W values, shifts below 2^BITS (a row of G needs 2s - 1 values and a
    // shift below s, so narrow grids use a narrow, shallow network)
#pragma unroll
    for (int b = 0; b < BITS; ++b) {
        const int step = 1 << b;
        const bool on = (sh >> b) & 1;
#pragma unroll
        for (int u = 0; u + step < W; ++u) v[u] = on ? v[u + step] : v[u];
    }
}

// xs[c] = xs[c] * scale_log2 + bias row c (+ -100 log2(e) where the region
// bit of column c is set, MASK), the row read as float4 chunks XOR-swizzled by
// swz. With DBG the bias is in natural units and also written to dbg_row.
template <int SL, int NC, bool MASK, bool DBG>
__device__ __forceinline__ void swin_add_bias_row(float (&xs)[SL], const unsigned char* rowp, int swz,
                                                  const uint32_t* mrow, float scale_log2, float* dbg_row, int nk) {
    static_assert(NC <= SL, "columns");
    const float mneg = DBG ? -100.0f : -100.0f * kLog2e;
    const float2 s2 = make_float2(scale_log2, scale_log2);
    constexpr int kQ = (NC + 3) / 4;  // float4 chunks that hold the first NC columns
#pragma unroll
    for (int wd = 0; wd < (kQ + 7) / 8; ++wd) {
        const uint32_t mb = MASK ? mrow[wd] : 0u;
#pragma unroll
        for (int q = wd * 8; q < min(wd * 8 + 8, kQ); ++q) {
            const float4 b4 = *reinterpret_cast<const float4*>(rowp + ((q ^ swz) << 4));
            float b[4] = {b4.x, b4.y, b4.z, b4.w};
            if constexpr (MASK) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if ((mb >> (4 * (q - wd * 8) + e)) & 1u) b[e] += mneg;
            }
            if constexpr (DBG) {
                if (dbg_row) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * q + e < nk) dbg_row[4 * q + e] = b[e];
                }
            }
            const float2 y0 = __ffma2_rn(make_float2(xs[4 * q], xs[4 * q + 1]), s2, make_float2(b[0], b[1]));
            const float2 y1 = __ffma2_rn(make_float2(xs[4 * q + 2], xs[4 * q + 3]), s2, make_float2(b[2], b[3]));
            xs[4 * q] = y0.x;
            xs[4 * q + 1] = y0.y;
            xs[4 * q + 2] = y1.x;
            xs[4 * q + 3] = y1.y;
        }
    }
}

// Store N (16, 32 or 64) consecutive TMEM columns of this lane.
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
    static_assert(N % 8 == 0 && N <= 64, "columns");
    if constexpr (N == 64) {
        tmem_st64(taddr, v);
    } else {
        if constexpr (N >= 32) tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(&v[0]));
        if constexpr (N % 32 >= 16)
            tmem_st16(taddr + N / 32 * 32, *reinterpret_cast<const uint32_t(*)[16]>(&v[N / 32 * 32]));
        if constexpr (N % 16 == 8)
            tmem_st8(taddr + N / 16 * 16, *reinterpret_cast<const uint32_t(*)[8]>(&v[N / 16 * 16]));
    }
}

// Load N (multiple of 16, <= 128) consecutive TMEM columns of this lane.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[N]) {
    static_assert(N % 16 == 0 && N <= 128, "columns");
    if constexpr (N == 128) {
        tmem_ld128(taddr, v);
    } else {
        if constexpr (N >= 64) {
            uint32_t t[64];
            tmem_ld64(taddr, t);
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = t[i];
        }
        if constexpr (N % 64 >= 32) {
            uint32_t t[32];
            tmem_ld32(taddr + (N / 64) * 64, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[(N / 64) * 64 + i] = t[i];
        }
        if constexpr (N % 32 == 16) {
            uint32_t t[16];
            tmem_ld16(taddr + (N / 32) * 32, t);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[(N / 32) * 32 + i] = t[i];
        }
    }
}

// Max of N floats with independent partial maxima (short dependency chains).
template <int N>
__device__ __forceinline__ float row_max(const float* x) {
    static_assert(N >= 16, "row_max");
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = fmaxf(x[2 * i], x[2 * i + 1]);
#pragma unroll
    for (int c = 16; c + 16 <= N; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = max3f(m[i], x[c + 2 * i], x[c + 2 * i + 1]);
#pragma unroll
    for (int t = N / 16 * 16; t < N; ++t) m[t % 8] = fmaxf(m[t % 8], x[t]);
    return fmaxf(fmaxf(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5])), fmaxf(m[6], m[7]));
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Min of N floats, as row_max.
template <int N>
__device__ __forceinline__ float row_min(const float* x) {
    static_assert(N >= 16, "row_min");
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = fminf(x[2 * i], x[2 * i + 1]);
#pragma unroll
    for (int c = 16; c + 16 <= N; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = min3f(m[i], x[c + 2 * i], x[c + 2 * i + 1]);
#pragma unroll
    for (int t = N / 16 * 16; t < N; ++t) m[t % 8] = fminf(m[t % 8], x[t]);
    return fminf(fminf(min3f(m[0], m[1], m[2]), min3f(m[3], m[4], m[5])), fminf(m[6], m[7]));
}

// max over c of x[c] * sc: the largest x for sc >= 0, the smallest for a
// negative multiplier (a negative scale flips the order of the scores).
// Key columns masked with -inf must not be present when sc < 0; the callers
// mask with -inf only after scaling, or with sc >= 0.
template <int N>
__device__ __forceinline__ float row_max_scaled(const float* x, float sc) {
    return sc >= 0.f ? row_max<N>(x) * sc : row_min<N>(x) * sc;
}

// p = 2^(x*sc + off) for N columns (x = -inf gives 0), packed to 16-bit pairs;
// returns the fp32 sum of the p values.
template <int N>
__device__ __forceinline__ float exp_pack(const float* x, float sc, float off, bool bf16, uint32_t* pk) {
    const float2 sc2 = make_float2(sc, sc), off2 = make_float2(off, off);
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if (bf16) {
#pragma unroll
        for (int c = 0; c < N; c += 2) {
            const float2 a = __ffma2_rn(make_float2(x[c], x[c + 1]), sc2, off2);
            const float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
            acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], make_float2(p0, p1));
            pk[c / 2] = pack_bf16(p0, p1);
        }
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 2) {
            const float2 a = __ffma2_rn(make_float2(x[c], x[c + 1]), sc2, off2);
            const float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
            acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], make_float2(p0, p1));
            pk[c / 2] = pack_f16(p0, p1);
        }
    }
    const float2 s = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
    return s.x + s.y;
}

// One arrival per warp once every lane is done (the barriers that the
// softmax warps signal count four arrivals, one per warp of the slot).
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Shared-memory descriptor of a 32B-swizzled operand block at `addr`
// (K-major: 8-row groups 256 B apart).  Moving along a block only changes the
// start-address field (bits 0-13, in 16-byte units), so the issue loops add
// offsets to one precomputed descriptor instead of rebuilding it per MMA:
// the single issuing thread is latency-bound on that scalar work.
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return make_sdesc(addr, 16, 256, kSwizzle32B); }
// MN-major (V): 16-column blocks kBlockN*32 bytes apart, 8-key groups 256 B apart.
__device__ __forceinline__ uint64_t vdesc(uint32_t addr) { return make_sdesc(addr, kBlockN * 32, 256, kSwizzle32B); }
// the same for a V tile of `rows` keys
__device__ __forceinline__ uint64_t vdesc_rows(uint32_t addr, uint32_t rows) {
    return make_sdesc(addr, rows * 32, 256, kSwizzle32B);
}

// S = Q.K^T for one 128-row tile: one MMA per 16-column block of d.
template <int DPAD>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t qd, uint64_t kd, uint32_t idesc) {
#pragma unroll
    for (int ks = 0; ks < Tile<DPAD>::kAtoms; ++ks)
        mma_ss(d_tmem, qd + (uint64_t)(ks * (kBlockM * 32 / 16)), kd + (uint64_t)(ks * (kBlockN * 32 / 16)),
               idesc, ks > 0 ? 1u : 0u);
}

// The same against a key tile of ROWS rows (16-column blocks ROWS*32 bytes
// apart), e.g. the 64-key tiles of one SAM grid row.
template <int DPAD, int ROWS>
__device__ __forceinline__ void issue_qk_rows(uint32_t d_tmem, uint64_t qd, uint64_t kd, uint32_t idesc) {
#pragma unroll
    for (int ks = 0; ks < Tile<DPAD>::kAtoms; ++ks)
        mma_ss(d_tmem, qd + (uint64_t)(ks * (kBlockM * 32 / 16)), kd + (uint64_t)(ks * (ROWS * 32 / 16)), idesc,
               ks > 0 ? 1u : 0u);
}

// D[:, 0:SL] (+)= Qone . E^T with Qone [128][SL] and E [SL][SL] K-major.
template <int SL>
__device__ __forceinline__ void issue_bias(uint32_t d_tmem, uint64_t qone_d, uint64_t blk_d, uint32_t idesc,
                                          uint32_t acc0) {
#pragma unroll
    for (int ks = 0; ks < SL / 16; ++ks)
        mma_ss(d_tmem, qone_d + (uint64_t)(ks * (kBlockM * 32 / 16)), blk_d + (uint64_t)(ks * (SL * 32 / 16)),
               idesc, (ks > 0 || acc0) ? 1u : 0u);
}

// O (+)= P.V over 128 keys: P from TMEM (two 16-bit values per column),
// V MN-major; 16 keys (512 bytes of V) per MMA.
template <int NK = kBlockN>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t vd, uint32_t idesc,
                                         uint32_t accumulate) {
#pragma unroll
    for (int ks = 0; ks < NK / 16; ++ks)
        mma_ts(o_tmem, p_tmem + ks * 8, vd + (uint64_t)(ks * (512 / 16)), idesc, (accumulate || ks > 0) ? 1u : 0u);
}

// Table row of SAM's decomposed relative position for query coordinate i and
// key coordinate j along one axis: i * qs - j * ks + off in float32 (the
// published coordinate scalers), truncated ("Accelerating Generative AI
// (part 1), Segment Anything", section Bfloat16 半精度: q_coords / k_coords
// index rel_pos_resized).  Clamped to the table.
__device__ __forceinline__ int sam_rel_row(int i, int j, float qs, float ks, float off, int lout) {
    const float rel = __fadd_rn(__fsub_rn(__fmul_rn((float)i, qs), __fmul_rn((float)j, ks)), off);
    return min(max((int)rel, 0), lout - 1);
}

// Row m of the table resampled from lin to lout rows (linear, half-pixel
// centres, clamped) read off g, the row's dot products with the table as
// given: resampling is linear, so it commutes with Q.R.
__device__ __forceinline__ float sam_resampled(const float* g, int m, int lin, int lout) {
    if (lin == lout) return g[m];
    const float src = fmaxf(__fmul_rn((float)lin / (float)lout, (float)m + 0.5f) - 0.5f, 0.f);
    const int i0 = min((int)src, lin - 1);
    const int i1 = min(i0 + 1, lin - 1);
    const float w1 = src - (float)i0;
    return (1.f - w1) * g[i0] + w1 * g[i1];
}

// General SAM bias rows of one query row (qh, qw): rel_h for every key row
// and rel_w for every key column, from G_h (in tO) and G_w (in tS).  rel_h
// goes to shared memory reversed like the generic grids' rows (entry
// k_h - 1 - kh); rel_w likewise into sam_rw.  The G rows go through a local
// array because the rows they are read at vary per thread.
// Only the G columns of the table (its length rounded up to 16) are loaded:
// the slot's S and O areas may be narrower than 128 columns.
static __device__ __noinline__ void sam_g_row(uint32_t taddr, int cols, float f, float* g) {
    for (int c0 = 0; c0 < cols; c0 += 16) {  // cols: the same on every lane (tcgen05.ld is warp-wide)
        uint32_t v[16];
        tmem_ld16(taddr + (uint32_t)c0, v);
#pragma unroll
        for (int t = 0; t < 16; ++t) g[c0 + t] = __uint_as_float(v[t]) * f;
    }
}
static __device__ __noinline__ void sam_general_rows(uint32_t tS, uint32_t tO, const AttnParams& p, int qh, int qw,
                                                     float f, float* sam_rh, float* sam_rw, int r) {
    float g[kBlockN];
    sam_g_row(tS, p.n_rw, f, g);
    for (int kw = 0; kw < p.k_w; ++kw) {
        const int m = sam_rel_row(qw, kw, p.sam_qs_w, p.sam_ks_w, p.sam_off_w, p.sam_lout_w);
        const float val = sam_resampled(g, m, p.sam_lin_w, p.sam_lout_w);
        sam_rw[(p.k_w - 1 - kw) * kBlockM + r] = val;
    }
    sam_g_row(tO, p.n_rh, f, g);
    for (int kh = 0; kh < p.k_h; ++kh) {
        const int m = sam_rel_row(qh, kh, p.sam_qs_h, p.sam_ks_h, p.sam_off_h, p.sam_lout_h);
        sam_rh[(p.k_h - 1 - kh) * kBlockM + r] = sam_resampled(g, m, p.sam_lin_h, p.sam_lout_h);
    }
}

template <int DPAD, int BIAS, int MODE, int SW, int SL, bool DBG, bool VL, bool IMG, bool SWR, bool NS>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ TmaMaps tm, const AttnParams p, const __grid_constant__ VarlenArg<VL> vt) {
    using T = Tile<DPAD>;
    // IMG: the Swin image token layout (p.swin_image) is a separate
    // instantiation, so that the windows-layout kernel carries none of its
    // gather and scatter code (the tests below are written out in full).
    // SWR: the Swin bias added from per-CTA rows (the host's swin_rows), not
    // by MMAs, likewise a separate instantiation.  NS: a scale <= 0 without
    // bias in shared tiling (its softmax scales before the max), likewise
    static_assert(MODE == kModeShared || (SL == 32 || SL == 64 || SL == 128), "slot size");
    // Key columns of a score tile (S MMA N, P.V K): 128, or narrower in shared
    // tiling when that lets separate P buffers fit tensor memory -- without
    // bias and every key in one tile (SW > 0, e.g. 80 for 77 text tokens), or
    // SAM on 14x14 grids (112 = eight grid rows).
    //
    // SAM on the 64 x 64 grid (kDbS) takes one grid row of 64 keys per score
    // tile and keeps two score buffers per slot, so the tensor core computes
    // the next two tiles' scores while the softmax works on this one:
    //   slot x (256 columns from 256x): S0 [0,64) S1 [64,128) O [128,128+DPAD);
    //   P of a tile lies over the first 32 columns of its own score buffer, so
    //   P is double-buffered too: the tile that next uses that buffer has its
    //   scores computed after this tile's P.V (in-order issue), and the
    //   softmax never waits for a P.V before writing P.  At a job's start
    //   G_w = Q.R_w^T lands over S0/S1 and G_h = Q.R_h^T over [128,256).
    // The 48 x 48 grid (a 768-pixel input) runs the same way with 48-key
    // tiles: S0 [0,48), S1 [48,96), O [128,128+DPAD); G_w (95 rows) over the
    // score buffers, G_h over [128,224).
    constexpr bool kDbS = MODE == kModeShared && BIAS == kBiasSam && (SW == 64 || SW == 48) && DPAD <= 96;
    constexpr int kTw = SW == 48 ? 48 : 64;  // kDbS: keys per score tile (one grid row)
    constexpr int kCols = kDbS ? kTw
                          : (MODE == kModeShared && BIAS == kBiasNone && SW > 0)  ? SW
                          : (MODE == kModeShared && BIAS == kBiasSam && SW == 14) ? 112
                                                                                  : 128;
    static_assert(kCols % 16 == 0 && kCols <= 128, "key columns");
    // Tensor memory: separate P buffers when they fit,
    //   S_A [0,kCols) S_B [kCols,2kCols) P_A/P_B 64 columns each from 2kCols,
    //   O_A/O_B kOw columns each from 2kCols + 128,
    // so the next score tile of a slot is issued as soon as its softmax has
    // read the current one (Q.K^T overlaps the softmax).  Otherwise P lies
    // over the first half of S, S_x = 128x, O_x = 256 + 128x.
    constexpr int kOffP = 2 * kCols;
    // Shared tiling with every key in one narrow tile (no bias, SW > 0, e.g.
    // 77 text tokens): a job is one score tile, so the next job's S is issued
    // as soon as the softmax has read this one, and a job's output is written
    // after the next job's softmax, while that job's P.V runs (two O buffers
    // per slot).  The output is staged in its own shared-memory area, so a Q
    // buffer is free again once its S is computed.
    constexpr bool kShDbl = MODE == kModeShared && BIAS == kBiasNone && SW > 0 && !DBG &&
                            kOffP + 128 + 4 * DPAD <= 512;
    constexpr int kOw = kShDbl ? 2 * DPAD : (DPAD <= 64 ? 64 : DPAD);
    constexpr int kOffO = kOffP + 128;
    constexpr bool kSepP = !kDbS && kOffO + 2 * kOw <= 512 && (BIAS != kBiasSam || SW == 14);
    // SAM on the 14 x 14 grid: G_w and G_h (32 columns each) land in the
    // slot's P buffer, columns [0,32) and [32,64), so a job's G and first S
    // need neither the previous job's epilogue (O) nor the gather (S): both
    // are issued as soon as the previous job's last S was read and its last
    // P.V issued, and overlap that job's epilogue.  The first P.V of the job
    // (which overwrites O) waits for that epilogue.
    constexpr bool kGinP = MODE == kModeShared && BIAS == kBiasSam && SW == 14 && kSepP;
    // Output rows staged per warp leave in one bulk copy (short jobs: the
    // one-tile pipeline and the SAM 14 x 14 windows), else as the warp's
    // own coalesced stores (long jobs, where the copy measured slower)
    constexpr bool kBulkOut = kShDbl || kGinP;
    // Packed tiling with head dims up to 32 and slots up to 64 rows: two O
    // buffers per slot (O_x holds 64 columns), so a tile's output is written
    // while the next tile's P.V runs.
    constexpr bool kDblO = MODE == kModeSeparate && DPAD <= 32 && SL <= 64 && !VL;
    // Packed variable-length batch: each slice of a tile is one (sequence,
    // head) of at most SL query and SL key tokens, its rows gathered with
    // zero fill past the sequence.  P.V runs one slice at a time (K = SL, its
    // own keys and values only) into the slot's O, which the slice's rows
    // read before the next slice's products overwrite it: a row never meets
    // another sequence's values, so the sequences stay apart whatever those
    // hold (block-diagonal P alone would still form 0 * inf there).
    constexpr bool kVP = MODE == kModeSeparate && VL;
    static_assert(!kVP || (BIAS == kBiasNone && SL <= 64), "packed variable-length batches: no bias, slots <= 64");
    // Packed Swin with the key count fixed at compile time (SW > 0, e.g. 49 for
    // 7x7 windows): the softmax touches only those columns (kNe: rounded up to
    // a pair), not the whole slot.
    constexpr int kNc = (MODE == kModeSeparate && BIAS == kBiasSwin && SW > 0) ? SW : (SL > 0 ? SL : 1);
    constexpr int kNe = (kNc + 1) & ~1;
    static_assert(MODE == kModeShared || kSepP, "the packed tiling uses separate P buffers");
    // Shared tiling without the varlen fix-up: the K and V copies of a ring
    // stage complete one barrier, so the MMA thread waits once per stage (its
    // waits are costly while earlier MMAs are queued); a tile's P.V always
    // follows its S, whose issue waited for the stage.
    constexpr bool kMergeKV = MODE == kModeShared && !VL;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1 KB-aligned base, formed by offsetting the array itself so that the
    // compiler keeps every derived access in the shared state space
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* sQ = smem + p.off_q;        // shared mode: [slot][buffer] Q tiles
    unsigned char* sRing = smem + p.off_ring;  // ring stages
    unsigned char* sExtraB = smem + p.off_extra;
    float* sExtra = reinterpret_cast<float*>(sExtraB);

    __shared__ uint64_t bar_q_full[2][2], bar_q_empty[2][2];
    __shared__ uint64_t bar_full_k[kMaxStages], bar_full_v[kMaxStages], bar_empty[kMaxStages];
    // variable-length batches: the V copy lands on bar_landed_v; the fix-up
    // warp then clears the tile's rows past the sequence and arrives on
    // bar_full_v
    __shared__ uint64_t bar_landed_v[VL ? kMaxStages : 1];
    __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2], bar_g[2], bar_gdone[2], bar_oempty[2];
    __shared__ uint64_t bar_sfree[2], bar_pvd[2];
    __shared__ uint64_t bar_sb[kDbS ? 2 : 1][2];  // kDbS: [slot][score buffer] scores ready
    // kVP: [slot][slice] that slice's P.V done; [slot] a slice's rows have read O
    __shared__ uint64_t bar_og[kVP ? 2 : 1][kVP ? kBlockM / SL : 1], bar_ohand[kVP ? 2 : 1];
    __shared__ uint64_t bar_final;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    __shared__ int s_tok[128];  // Swin: per-token position and region labels

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int* abort_flag = &abort_sh;
    const int nst = p.nst;
    const bool bf = p.is_bf16 != 0;
    // bytes of one K (or V) tile of a shared-tiling ring stage: box_kv rows
    const uint32_t kv_tile_bytes = (uint32_t)T::kAtoms * (uint32_t)p.box_kv * 32u;

    // A kernel launched after this one on the stream may start its set-up
    // while this grid drains (programmatic dependent launch); it reads
    // nothing before its own griddepcontrol.wait below.
    griddep_launch_dependents();
    if (tid == 0) {
        abort_sh = 0;
        for (int x = 0; x < 2; ++x) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&bar_q_full[x][b], 1);
                // double-buffered Q: the softmax warps release it after using it
                // as output staging; single Q: the last P.V's commit releases it;
                // the one-tile pipeline: the commit of its S releases it
                mbar_init(&bar_q_empty[x][b], (p.nq == 2 && !kShDbl) ? 4 : 1);
            }
            mbar_init(&bar_s[x], 1);
            mbar_init(&bar_p[x], 4);
            mbar_init(&bar_o[x], 1);
            mbar_init(&bar_g[x], 1);
            mbar_init(&bar_gdone[x], 4);
            mbar_init(&bar_oempty[x], 4);
            mbar_init(&bar_sfree[x], 4);
            mbar_init(&bar_pvd[x], 1);
            if constexpr (kDbS) {
                mbar_init(&bar_sb[x][0], 1);
                mbar_init(&bar_sb[x][1], 1);
            }
            if constexpr (kVP) {
                for (int g = 0; g < kBlockM / SL; ++g) mbar_init(&bar_og[x][g], 1);
                mbar_init(&bar_ohand[x], SL / 32);  // the warps of one slice
            }
        }
        for (int i = 0; i < kMaxStages; ++i) {
            // the image-layout Swin stages are filled by two warps
            mbar_init(&bar_full_k[i], (kVP || (MODE == kModeSeparate && BIAS == kBiasSwin && IMG && p.swin_image)) ? 64 : 1);
            mbar_init(&bar_full_v[i], 1);
            mbar_init(&bar_empty[i], MODE == kModeShared ? 2 : 1);
            if constexpr (VL) mbar_init(&bar_landed_v[i], 1);
        }
        mbar_init(&bar_final, 2);
        fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tm.q);
        prefetch_tensormap(&tm.k);
        prefetch_tensormap(&tm.v);
        if constexpr (BIAS == kBiasSam) {
            prefetch_tensormap(&tm.rh);
            prefetch_tensormap(&tm.rw);
        }
    }
    // Global memory is touched only after the grids this launch depends on
    // have completed and their writes are visible.
    griddep_wait();
    if (BIAS == kBiasSwin && SL <= 64 && SWR) {
        // Per head h: row i (query token), column j (key token) holds
        // table[idx(i, j), h] in log2 units (natural units when debugging);
        // idx is the relative-position index ("视觉大模型训练和推理加速"
        // section 一, relative position bias), pos(i) - pos(j) + 2M(M - 1)
        // with pos(t) = r_t (2M - 1) + c_t. Then, per window kind k = 1..3,
        // bit j of row i is set when i and j fall in different regions of the
        // shifted window (cut by the last column (k = 1), the last row (k = 2)
        // or both (k = 3)): those pairs get -100 more.
        const int M = p.win, N = p.Nk, T = 2 * M - 1;
        const float fl = DBG ? 1.0f : kLog2e;
        const int yb = (p.n_wh - 1) * M, xb = (p.n_ww - 1) * M;  // last window row / column origin
        for (int t = tid; t < SL; t += kThreads) {
            const int rt = t / M, ct = t - (t / M) * M;
            const int lab = swin_strip(xb + ct, p.grid_w, M, p.shift) | (swin_strip(yb + rt, p.grid_h, M, p.shift) << 2);
            s_tok[t] = (rt * T + ct) | (lab << 16);
        }
        // the table passes through the (not yet loaded) ring
        float* stab = reinterpret_cast<float*>(smem + p.off_ring);
        for (int i = tid; i < T * T * p.H; i += kThreads) stab[i] = p.table[i];
        __syncthreads();
        const int c0 = 2 * M * (M - 1);
        for (int w = tid; w < p.H * SL * (SL / 4); w += kThreads) {
            const int q = w % (SL / 4), i = (w / (SL / 4)) % SL, h = w / (SL * (SL / 4));
            const int pi = s_tok[i] & 0xFFFF;
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 4 * q + e;
                const bool ok = i < N && j < N;
                const int idx = ok ? pi - (s_tok[j] & 0xFFFF) + c0 : 0;
                v[e] = stab[idx * p.H + h];
                v[e] = ok ? v[e] * fl : 0.f;
            }
            *reinterpret_cast<float4*>(sExtraB + (h * SL + i) * SL * 4 + ((q ^ (i & 7)) << 4)) =
                make_float4(v[0], v[1], v[2], v[3]);
        }
        uint32_t* mbits = reinterpret_cast<uint32_t*>(sExtraB + p.H * SL * SL * 4);
        for (int w = tid; w < 3 * SL * (SL / 32); w += kThreads) {
            const int wd = w % (SL / 32), i = (w / (SL / 32)) % SL, kind = w / (SL * (SL / 32)) + 1;
            const int sel = ((kind & 1) ? 0x3 : 0) | ((kind & 2) ? 0xC : 0);
            const int li = s_tok[i] >> 16;
            uint32_t bits = 0;
            if (i < N && p.shift) {
                for (int e = 0; e < 32; ++e) {
                    const int j = wd * 32 + e;
                    if (j < N && (((s_tok[j] >> 16) ^ li) & sel)) bits |= 1u << e;
                }
            }
            mbits[w] = bits;
        }
    } else if constexpr (BIAS == kBiasSwin) {
        // Qone [128][SL]: row r has a single 1 at column r mod SL.
        // Blocks [SL][SL] (row = key token j, column = query token t):
        //   h < H        : table[idx(t, j), h] / scale      (natural units when debugging)
        //   H + kind - 1 : -100 / scale where t and j fall in different regions
        //                  of a window on the last column (kind 1), last row
        //                  (kind 2) or both (kind 3)
        // Slot rows past the slice length need no clearing: the TMA box covers
        // them and fills them with zeros.
        const int M = p.win, N = p.Nk, T = 2 * M - 1;
        const float f = DBG ? 1.0f : 1.0f / p.scale;
        unsigned char* qone_b = sExtraB;
        unsigned char* blocks_b = sExtraB + kBlockM * SL * 2;
        // the table goes through shared memory (the Qone area, built last) when
        // it fits, so each thread's gathers are shared-memory loads
        const int ntab = T * T * p.H;
        const bool tab_smem = ntab * 4 <= kBlockM * SL * 2;
        float* stab = reinterpret_cast<float*>(qone_b);
        if (tab_smem)
            for (int i = tid; i < ntab; i += kThreads) stab[i] = p.table[i];
        __syncthreads();
        const float* tab = tab_smem ? stab : p.table;
        const int nblk = p.H + 3;
        // per query/key token: pos = r (2M - 1) + c, region labels of the
        // token in a window on the last column (bits 16-17) and last row
        // (bits 18-19)
        const int yb = (p.n_wh - 1) * M, xb = (p.n_ww - 1) * M;  // last window row / column origin
        for (int t = tid; t < SL; t += kThreads) {
            const int rt = t / M, ct = t - (t / M) * M;
            const int lab = swin_strip(xb + ct, p.grid_w, M, p.shift) | (swin_strip(yb + rt, p.grid_h, M, p.shift) << 2);
            s_tok[t] = (rt * T + ct) | (lab << 16);
        }
        __syncthreads();
        // one work item = 8 columns of one row (key token j) of one block
        for (int w = tid; w < nblk * SL * (SL / 8); w += kThreads) {
            const int j = w % SL, g = (w / SL) % (SL / 8), b = w / (SL * (SL / 8));
            const int t0 = g * 8;
            const bool key_ok = j < N;
            const int tj = s_tok[j];
            unsigned char* dst = blocks_b + b * SL * SL * 2 + kmajor_offset(SL, j, t0);
            if (b < p.H) {
                if (tab_smem) swin_table_group(dst, stab, s_tok, t0, tj & 0xFFFF, key_ok, b, p.H, M, N, f, bf);
                else swin_table_group(dst, p.table, s_tok, t0, tj & 0xFFFF, key_ok, b, p.H, M, N, f, bf);
            } else {
                // mask blocks 1..3: -100 where t and j carry different region
                // labels along the axes the window kind cuts
                const int kind = b - p.H + 1;
                const int sel = ((kind & 1) ? 0x3 : 0) | ((kind & 2) ? 0xC : 0);
                const float mv = -100.0f * f;
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const bool diff = ((((s_tok[t0 + u] ^ tj) >> 16) & sel) != 0);
                    v[u] = (key_ok && t0 + u < N && p.shift && diff) ? mv : 0.f;
                }
                store_half8(dst, v, bf);
            }
        }
        __syncthreads();  // the table's area becomes Qone
        const uint32_t one = to_half_bits(1.0f, bf);
        for (int c = tid; c < kBlockM * SL / 8; c += kThreads) {
            const int r = c / (SL / 8), t0 = (c - r * (SL / 8)) * 8;
            const int e = (r % SL) - t0;  // position of the 1 in this chunk, if any
            uint32_t pk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                pk[u] = (e == 2 * u ? one : 0u) | (e == 2 * u + 1 ? one << 16 : 0u);
            *reinterpret_cast<uint4*>(qone_b + kmajor_offset(kBlockM, r, t0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
    }
    if constexpr (MODE == kModeSeparate) fence_proxy_async_smem();
    if constexpr (BIAS == kBiasSam) {
        if (p.sam_resample) {
            // rel_pos_resized: each table linearly resampled to 2 * side - 1
            // rows (half-pixel centres, clamped), rounded to the operand type
            // as the model's resized table is, laid out as the MMA's K-major
            // operand; rows past the table and columns past d are zero
            constexpr int kChunks = DPAD / 8;
            for (int i = tid; i < 2 * kBlockN * kChunks; i += kThreads) {
                const int tb = i / (kBlockN * kChunks);  // 0: R_w, 1: R_h
                const int m = (i / kChunks) % kBlockN;
                const int c8 = i % kChunks;
                const int lin = tb ? p.sam_lin_h : p.sam_lin_w, lout = tb ? p.sam_lout_h : p.sam_lout_w;
                const uint16_t* src = static_cast<const uint16_t*>(tb ? p.rel_h : p.rel_w);
                uint32_t pk[4] = {0u, 0u, 0u, 0u};
                if (m < lout && c8 * 8 < p.d) {
                    const float pos = fmaxf(__fmul_rn((float)lin / (float)lout, (float)m + 0.5f) - 0.5f, 0.f);
                    const int i0 = min((int)pos, lin - 1), i1 = min(i0 + 1, lin - 1);
                    const float w1 = pos - (float)i0;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        float v[2];
#pragma unroll
                        for (int z = 0; z < 2; ++z) {
                            const int col = c8 * 8 + e + z;
                            const uint16_t a = src[(size_t)i0 * p.d + col], b = src[(size_t)i1 * p.d + col];
                            const float fa = bf ? __bfloat162float(__ushort_as_bfloat16(a)) : __half2float(__ushort_as_half(a));
                            const float fb = bf ? __bfloat162float(__ushort_as_bfloat16(b)) : __half2float(__ushort_as_half(b));
                            v[z] = (1.f - w1) * fa + w1 * fb;
                        }
                        pk[e / 2] = (uint32_t)to_half_bits(v[0], bf) | ((uint32_t)to_half_bits(v[1], bf) << 16);
                    }
                }
                *reinterpret_cast<uint4*>(smem + p.off_rtab + tb * T::kBytes + kmajor_offset(kBlockN, m, c8 * 8)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            fence_proxy_async_smem();  // read by the tensor core
        }
    }
    if constexpr (BIAS == kBiasSam && SW == 0) {
        // key table for generic grids: (k_h-1-kh) | (k_w-1-kw) << 16
        int* kt = reinterpret_cast<int*>(sExtra + 2 * (p.k_h + p.k_w) * kBlockM);
        for (int k = tid; k < p.Nk; k += kThreads) {
            const int kh = k / p.k_w, kw = k % p.k_w;
            kt[k] = (p.k_h - 1 - kh) | ((p.k_w - 1 - kw) << 16);
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const int job0 = blockIdx.x, job_step = gridDim.x;

    if (warp >= 8) {
      regs_dec<kControlRegs>();
      if (warp == kProducerWarp ||
          (warp == kGatherWarp && (kVP || (MODE == kModeSeparate && BIAS == kBiasSwin && IMG && p.swin_image)))) {
        // =========================================================== producer
        if constexpr (kVP) {
            // Packed variable-length batch: this warp and the gather warp
            // copy alternate slices of each tile with 16-byte cp.async copies,
            // kLanesRow lanes per row, into the swizzled tiles the TMA path
            // lands.  A slice is one (sequence, head): query rows from its
            // [H][Lq][d] block, key and value rows from its [H][Lk][d] block;
            // rows past the sequence, padding columns and slices past the last
            // are written as zeros.  Arrivals as in the image-layout gather.
            constexpr int kChunks = DPAD / 8;
            constexpr int kLanesRow = kChunks <= 2 ? 2 : (kChunks <= 4 ? 4 : 8);
            constexpr int kRowsIt = 32 / kLanesRow;
            constexpr int kG = kBlockM / SL;
            static_assert(SL % kRowsIt == 0 && kG >= 2, "a warp instruction stays inside one slice");
            const int half = warp == kProducerWarp ? 0 : 1;
            const int c = lane % kLanesRow;
            const int rsub = lane / kLanesRow;
            const bool lane_on = c < kChunks;
            const bool c_data = c * 8 < p.d;
            const uint32_t dchunk = (uint32_t)((c >> 1) * (kBlockM * 32));
            const size_t rowb = (size_t)p.d * 2;
            int ring = 0;
            bool ok = true;
            for (int job = job0; ok && job < p.n_jobs; job += job_step) {
                for (int x = 0; x < 2; ++x) {
                    const int st = ring % nst;
                    if (ring >= nst) {
                        __syncwarp();
                        if (!__all_sync(0xffffffffu, mbar_wait(&bar_empty[st], ((ring / nst) + 1) & 1, abort_flag,
                                                               kStatusWaitEmpty))) {
                            ok = false;
                            break;
                        }
                    }
                    ++ring;
                    const int tile = 2 * job + x;
                    unsigned char* base = sRing + st * p.ring_stage_bytes;
                    if (lane_on) {
#pragma unroll 1
                        for (int g = half; g < kG; g += 2) {
                            const int slice = tile * kG + g;
                            int lq = 0, lk = 0;
                            size_t qrow = 0, krow = 0;
                            if (slice < p.BH) {
                                const int e = slice / p.H, h = slice - e * p.H;
                                lq = vt.q_len[e];
                                lk = vt.k_len[e];
                                qrow = (size_t)p.H * (size_t)vt.q_off[e] + (size_t)h * (size_t)lq;
                                krow = (size_t)p.H * (size_t)vt.k_off[e] + (size_t)h * (size_t)lk;
                            }
#pragma unroll 4
                            for (int it = 0; it < SL / kRowsIt; ++it) {
                                const int t = it * kRowsIt + rsub;
                                const int R = g * SL + t;
                                const bool onq = c_data && t < lq, onk = c_data && t < lk;
                                const size_t offq = onq ? (qrow + t) * rowb + (size_t)c * 16 : 0;
                                const size_t offk = onk ? (krow + t) * rowb + (size_t)c * 16 : 0;
                                const uint32_t dst = smem_u32(base + R * 32) + dchunk +
                                                     ((((uint32_t)c & 1u) ^ (((uint32_t)R >> 2) & 1u)) << 4);
                                cp_async16(dst, static_cast<const unsigned char*>(p.q) + offq, onq ? 16u : 0u);
                                cp_async16(dst + T::kBytes, static_cast<const unsigned char*>(p.k) + offk, onk ? 16u : 0u);
                                cp_async16(dst + 2 * T::kBytes, static_cast<const unsigned char*>(p.v) + offk,
                                           onk ? 16u : 0u);
                            }
                        }
                    }
                    cp_async_arrive_noinc(&bar_full_k[st]);
                }
            }
            cp_async_wait<0>();
        } else if (MODE == kModeSeparate && BIAS == kBiasSwin && IMG && p.swin_image) {
            // Image layout: this warp and the gather warp copy each window's
            // token rows with 16-byte cp.async copies, the cyclic shift and
            // the window partition folded into the source addresses,
            // kLanesRow lanes per row, into the swizzled tiles the TMA path
            // lands (padding rows and columns written as zeros).  The warps
            // take alternate slices of a tile, or alternate row groups when a
            // tile holds one slice.  (Rows of one head are 2d bytes out of
            // every 2Hd, too short for box copies to pay.)  A stage's barrier
            // counts one arrival per lane of the two warps, each made by the
            // copy hardware once that lane's copies have landed; the MMA
            // warps fence the proxies after their wait.
            constexpr int kChunks = DPAD / 8;  // 16-byte chunks of a padded row
            constexpr int kLanesRow = kChunks <= 2 ? 2 : (kChunks <= 4 ? 4 : 8);
            constexpr int kRowsIt = 32 / kLanesRow;      // rows per warp instruction
            constexpr int kSL = SL > 0 ? SL : kBlockM;  // (SL is 0 only in shared mode)
            constexpr int kG = kBlockM / kSL;            // slices per tile
            static_assert(kSL % kRowsIt == 0, "a warp instruction stays inside one slice");
            const int half = warp == kProducerWarp ? 0 : 1;  // which slices (or row groups) this warp copies
            const int c = lane % kLanesRow;  // this lane's chunk of every row it copies
            const int rsub = lane / kLanesRow;
            const bool lane_on = c < kChunks;  // lanes past the padded row copy nothing
            const bool c_data = c * 8 < p.d;   // else the chunk is zero padding
            const uint32_t dchunk = (uint32_t)((c >> 1) * (kBlockM * 32));
            const size_t rowb = (size_t)p.d * 2;
            int ring = 0;
            bool ok = true;
            for (int job = job0; ok && job < p.n_jobs; job += job_step) {
                for (int x = 0; x < 2; ++x) {
                    const int st = ring % nst;
                    if (ring >= nst) {
                        __syncwarp();
                        if (!__all_sync(0xffffffffu, mbar_wait(&bar_empty[st], ((ring / nst) + 1) & 1, abort_flag,
                                                               kStatusWaitEmpty))) {
                            ok = false;
                            break;
                        }
                    }
                    const int use = ring++;
                    const int tile = 2 * job + x;
                    unsigned char* base = sRing + st * p.ring_stage_bytes;
                    if (lane_on) {
#pragma unroll 1
                        for (int g = (kG > 1 ? half : 0); g < kG; g += (kG > 1 ? 2 : 1)) {
                            // the slice's image, window origin after the shift
                            // and head; rows past the window or of a missing
                            // slice read as zero
                            const uint32_t slice = (uint32_t)(tile * kG + g);
                            const bool sv = (int)slice < p.BH;
                            const uint32_t bimg = fast_div(slice, p.fd_h);
                            const uint32_t hh = slice - bimg * (uint32_t)p.H;
                            const uint32_t img = fast_div(bimg, p.fd_w);
                            const uint32_t w = bimg - img * (uint32_t)p.n_w;
                            const uint32_t wr = fast_div(w, p.fd_ww);
                            const uint32_t ib = img * (uint32_t)p.grid_h;
                            const uint32_t yb = wr * (uint32_t)p.win + (uint32_t)p.shift;
                            const uint32_t xb = (w - wr * (uint32_t)p.n_ww) * (uint32_t)p.win + (uint32_t)p.shift;
#pragma unroll 4
                            for (int it = (kG > 1 ? 0 : half); it < kSL / kRowsIt; it += (kG > 1 ? 1 : 2)) {
                                const uint32_t t = (uint32_t)(it * kRowsIt + rsub);
                                const int R = g * kSL + (int)t;
                                const uint32_t r = fast_div(t, p.fd_m);
                                uint32_t yy = yb + r;
                                if (yy >= (uint32_t)p.grid_h) yy -= (uint32_t)p.grid_h;
                                uint32_t xx = xb + (t - r * (uint32_t)p.win);
                                if (xx >= (uint32_t)p.grid_w) xx -= (uint32_t)p.grid_w;
                                const bool on = c_data && sv && (int)t < p.Nk;
                                const size_t row = ((size_t)(ib + yy) * (size_t)p.grid_w + xx) * (size_t)p.H + hh;
                                const size_t off = on ? row * rowb + (size_t)c * 16 : 0;
                                const uint32_t dst = smem_u32(base + R * 32) + dchunk +
                                                     ((((uint32_t)c & 1u) ^ (((uint32_t)R >> 2) & 1u)) << 4);
                                const uint32_t nb = on ? 16u : 0u;
                                cp_async16(dst, static_cast<const unsigned char*>(p.q) + off, nb);
                                cp_async16(dst + T::kBytes, static_cast<const unsigned char*>(p.k) + off, nb);
                                cp_async16(dst + 2 * T::kBytes, static_cast<const unsigned char*>(p.v) + off, nb);
                            }
                        }
                    }
                    // every lane's arrival lands with its copies: the warp
                    // never waits for them and runs ahead to the next stage
                    cp_async_arrive_noinc(&bar_full_k[st]);
                }
            }
            cp_async_wait<0>();
        } else if (lane == 0) {
            const uint32_t q_tx = (uint32_t)T::kAtoms * (uint32_t)p.box_q * 32u;
            const uint32_t kv_tx = (uint32_t)T::kAtoms * (uint32_t)p.box_kv * 32u;
            int ring = 0;  // stage uses issued
            bool ok = true;
            int ju = 0;
            for (int job = job0; ok && job < p.n_jobs; job += job_step, ++ju) {
                if constexpr (MODE == kModeShared) {
                    const JobRows jr = shared_job<VL>(p, vt, job);
                    const int qb = ju % p.nq;
                    for (int x = 0; x < 2; ++x) {
                        if (ju >= p.nq &&
                            !mbar_wait(&bar_q_empty[x][qb], ((ju / p.nq) + 1) & 1, abort_flag, kStatusWaitEmpty)) {
                            ok = false;
                            break;
                        }
                        unsigned char* dq = sQ + (x * p.nq + qb) * T::kBytes;
                        mbar_arrive_expect_tx(&bar_q_full[x][qb], q_tx);
                        tma_load_4d(dq, &tm.q, &bar_q_full[x][qb], 0, jr.q_row + x * kBlockM, jr.q_slice, 0);
                        if (p.part)
                            tma_load_3d(dq + p.full_atoms * kBlockM * 32, &tm.qp, &bar_q_full[x][qb], 0, jr.q_row + x * kBlockM,
                                        jr.q_slice);
                    }
                    // SAM: a first stage with the tables, unless the CTA resampled them;
                    // with 64-row tiles two stages: R_w rows [0,64) and [64,128) in
                    // the K and V tiles of the first, R_h likewise in the second
                    const int t_use = (BIAS == kBiasSam && !p.sam_resample) ? (kDbS ? 2 : 1) : 0;
                    const int n_uses = jr.n_kv + t_use;
                    for (int u = 0; ok && u < n_uses; ++u) {
                        const int st = ring % nst;
                        if (ring >= nst &&
                            !mbar_wait(&bar_empty[st], ((ring / nst) + 1) & 1, abort_flag, kStatusWaitEmpty)) {
                            ok = false;
                            break;
                        }
                        ++ring;
                        unsigned char* dk = sRing + st * p.ring_stage_bytes;
                        unsigned char* dv = dk + kv_tile_bytes;
                        // the V half lands on the stage's K barrier (kMergeKV) or its own
                        uint64_t* const bk = &bar_full_k[st];
                        uint64_t* const bv = kMergeKV ? bk : (VL ? &bar_landed_v[st] : &bar_full_v[st]);
                        if (kDbS && u < t_use) {
                            const CUtensorMap* tfull = u == 0 ? &tm.rw : &tm.rh;
                            const CUtensorMap* tpart = u == 0 ? &tm.rwp : &tm.rhp;
                            mbar_arrive_expect_tx(bk, kMergeKV ? 2 * kv_tx : kv_tx);
                            tma_load_3d(dk, tfull, bk, 0, 0, 0);
                            if (p.part) tma_load_2d(dk + p.full_atoms * p.box_kv * 32, tpart, bk, 0, 0);
                            if (!kMergeKV) mbar_arrive_expect_tx(bv, kv_tx);
                            tma_load_3d(dv, tfull, bv, 0, kTw, 0);
                            if (p.part) tma_load_2d(dv + p.full_atoms * p.box_kv * 32, tpart, bv, 0, kTw);
                        } else if (BIAS == kBiasSam && u < t_use) {
                            // rel-pos tables: R_w in the K slot, R_h in the V slot
                            const uint32_t r_tx = (uint32_t)T::kAtoms * kBlockN * 32u;
                            mbar_arrive_expect_tx(bk, kMergeKV ? 2 * r_tx : r_tx);
                            tma_load_3d(dk, &tm.rw, bk, 0, 0, 0);
                            if (p.part) tma_load_2d(dk + p.full_atoms * kBlockN * 32, &tm.rwp, bk, 0, 0);
                            if (!kMergeKV) mbar_arrive_expect_tx(bv, r_tx);
                            tma_load_3d(dv, &tm.rh, bv, 0, 0, 0);
                            if (p.part) tma_load_2d(dv + p.full_atoms * kBlockN * 32, &tm.rhp, bv, 0, 0);
                        } else {
                            const int j = u - t_use;
                            const int kr = jr.k_row + j * p.kv_w;
                            mbar_arrive_expect_tx(bk, kMergeKV ? 2 * kv_tx : kv_tx);
                            tma_load_4d(dk, &tm.k, bk, 0, kr, jr.k_slice, 0);
                            if (p.part) tma_load_3d(dk + p.full_atoms * p.box_kv * 32, &tm.kp, bk, 0, kr, jr.k_slice);
                            if (!kMergeKV) mbar_arrive_expect_tx(bv, kv_tx);
                            tma_load_4d(dv, &tm.v, bv, 0, kr, jr.k_slice, 0);
                            if (p.part) tma_load_3d(dv + p.full_atoms * p.box_kv * 32, &tm.vp, bv, 0, kr, jr.k_slice);
                        }
                    }
                } else {
                    for (int x = 0; x < 2; ++x) {
                        const int st = ring % nst;
                        if (ring >= nst &&
                            !mbar_wait(&bar_empty[st], ((ring / nst) + 1) & 1, abort_flag, kStatusWaitEmpty)) {
                            ok = false;
                            break;
                        }
                        ++ring;
                        const int tile = 2 * job + x;
                        unsigned char* dq = sRing + st * p.ring_stage_bytes;
                        unsigned char* dk = dq + T::kBytes;
                        unsigned char* dv = dk + T::kBytes;
                        // one copy per operand: g slices of SL rows (rows past
                        // the slice length read as zero), all column blocks
                        mbar_arrive_expect_tx(&bar_full_k[st], 3u * T::kBytes);
                        const int s0 = tile * p.g;
                        tma_load_4d(dq, &tm.q, &bar_full_k[st], 0, 0, s0, 0);
                        tma_load_4d(dk, &tm.k, &bar_full_k[st], 0, 0, s0, 0);
                        tma_load_4d(dv, &tm.v, &bar_full_k[st], 0, 0, s0, 0);
                        if (p.part) {
                            const int po = p.full_atoms * kBlockM * 32;
                            tma_load_3d(dq + po, &tm.qp, &bar_full_k[st], 0, 0, s0);
                            tma_load_3d(dk + po, &tm.kp, &bar_full_k[st], 0, 0, s0);
                            tma_load_3d(dv + po, &tm.vp, &bar_full_k[st], 0, 0, s0);
                        }
                    }
                }
            }
            if (*abort_flag) {
                // let copies still in flight land before the CTA retires
                for (int u = (ring > nst ? ring - nst : 0); u < ring; ++u) {
                    const int st = u % nst;
                    mbar_wait(&bar_full_k[st], (u / nst) & 1, nullptr, 0);
                    if (MODE == kModeShared && !kMergeKV)
                        mbar_wait(VL ? &bar_landed_v[st] : &bar_full_v[st], (u / nst) & 1, nullptr, 0);
                }
            }
        }
      } else if (VL && MODE == kModeShared && warp == kGatherWarp) {
        // ============================================ variable-length fix-up
        // A key tile that runs past its sequence holds the next sequence's
        // rows.  Their scores are masked to -inf, so they get P = 0, but a
        // non-finite value there would still reach the output through
        // 0 * inf = NaN in P.V: clear those V rows (whole 32-byte rows of
        // every 16-column block, so the swizzle does not matter) before the
        // tile is released to the MMA issuers.  Sequences then never
        // interact, whatever the neighbouring data hold.
        int ring = 0;
        bool ok = true;
        for (int job = job0; ok && job < p.n_jobs; job += job_step) {
            const JobRows jr = shared_job<VL>(p, vt, job);
            for (int u = 0; u < jr.n_kv; ++u, ++ring) {
                const int st = ring % nst;
                __syncwarp();
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_landed_v[st], (ring / nst) & 1, abort_flag, kStatusWaitV))) {
                    ok = false;
                    break;
                }
                const int hi = jr.nk - u * p.kv_w;  // rows of the sequence in this tile
                if (hi < kBlockN) {
                    unsigned char* dv = sRing + st * p.ring_stage_bytes + kv_tile_bytes;
                    const int n16 = 2 * (kBlockN - hi);  // 16-byte chunks per column block
                    for (int c = lane; c < T::kAtoms * n16; c += 32) {
                        const int blk = c / n16, rc = c - blk * n16;
                        *reinterpret_cast<uint4*>(dv + blk * (kBlockN * 32) + (hi + (rc >> 1)) * 32 + (rc & 1) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();  // read by the tensor core next
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_full_v[st]);
            }
        }
      } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // ================================================================ MMA
        // One issuing warp per slot (warp 9: slot A, warp 10: slot B), all
        // lanes converged, lane 0 issuing: tcgen05.commit tracks the MMAs of
        // the issuing lane, so each slot's products run on their own
        // schedule; a shared K/V stage is released after both warps have
        // committed their last use of it.
        {
            const int x = warp - kMmaWarp;
            const uint32_t idesc_s = make_idesc_f16(bf, kBlockM, MODE == kModeShared ? kCols : kBlockN, false);
            const uint32_t idesc_o = make_idesc_f16(bf, kBlockM, DPAD, true);
            const uint32_t idesc_b = make_idesc_f16(bf, kBlockM, MODE == kModeSeparate ? SL : 16, false);
            const uint32_t tSx = tmem + (uint32_t)(kDbS ? 256 * x : (kSepP ? kCols : 128) * x);
            const uint32_t tPx = kSepP ? tmem + (uint32_t)(kOffP + 64 * x) : tSx;  // kDbS: + 64 * buffer
            const uint32_t tOx = kDbS ? tSx + 128 : tmem + (uint32_t)(kSepP ? kOffO + kOw * x : 256 + 128 * x);
            uint64_t* const bs = &bar_s[x];
            uint64_t* const bp = &bar_p[x];
            uint64_t* const bo = &bar_o[x];
            uint64_t* const bsf = &bar_sfree[x];
            uint64_t* const bpv = &bar_pvd[x];
            int ring = 0;  // stage uses consumed
            uint32_t ph_p = 0;
            int s_cnt = 0;  // score tiles issued
            int hand_cnt = 0;  // kVP: slice hand-overs of O awaited
            int ju = 0;
            bool ok = true;
            const uint64_t qone_d = kdesc(smem_u32(sExtraB));
            const uint32_t blocks = smem_u32(sExtraB) + kBlockM * SL * 2;
            // every lane waits (no warp vote: the lanes run in step)
            auto waitb = [&](uint64_t* bar, uint32_t parity, int code) -> bool {
                if (!mbar_wait(bar, parity, abort_flag, code)) return false;
                tc_fence_after();
                return true;
            };
            // Before the next score tile overwrites S_x its softmax must have
            // read the previous one (separate P buffers only).
            auto s_free = [&]() -> bool {
                if (!kSepP || s_cnt == 0) return true;
                return waitb(bsf, (s_cnt - 1) & 1, kStatusWaitS);
            };
            // S of packed tile `tile` (separate mode), with the Swin bias
            auto sep_scores = [&](int tile, uint32_t qa) {
                if (!DBG || BIAS != kBiasSwin || (SL <= 64 && SWR))
                    issue_qk<DPAD>(tSx, kdesc(qa), kdesc(qa + T::kBytes), idesc_s);
                if (BIAS == kBiasSwin && !(SL <= 64 && SWR)) {
                    for (int sl = 0; sl < p.g; ++sl) {
                        const uint32_t slice = (uint32_t)(tile * p.g + sl);
                        if ((int)slice >= p.BH) break;
                        int h, kind;
                        swin_slice_info(slice, p.H, p.n_w, p.n_ww, p.n_wh, p.shift, p.fd_h, p.fd_w, p.fd_ww, h, kind);
                        const uint32_t d = tSx + sl * SL;
                        issue_bias<SL>(d, qone_d, kdesc(blocks + h * SL * SL * 2), idesc_b, DBG ? 0u : 1u);
                        if (kind) issue_bias<SL>(d, qone_d, kdesc(blocks + (p.H + kind - 1) * SL * SL * 2), idesc_b, 1u);
                    }
                }
            };
            for (int job = job0; ok && job < p.n_jobs; job += job_step, ++ju) {
                if constexpr (kDbS) {
                    // SAM, 64 x 64 (48 x 48) grid: one grid row of keys per score tile,
                    // two score buffers
                    const int qb = ju % p.nq;
                    const uint64_t qa = kdesc(smem_u32(sQ + (x * p.nq + qb) * T::kBytes));
                    if (!waitb(&bar_q_full[x][qb], (ju / p.nq) & 1, kStatusWaitQ)) { ok = false; break; }
                    // G_w = Q.R_w^T over the score buffers, G_h = Q.R_h^T over O and
                    // P, from the tables the CTA staged once.  O must have been read by
                    // the previous job's epilogue; P was read by this thread's last
                    // P.V, which the tensor core finishes first (in-order issue).
                    if (ju > 0 && !waitb(&bar_oempty[x], (ju - 1) & 1, kStatusWaitO)) { ok = false; break; }
                    if (p.sam_resample) {
                        const uint32_t rt = smem_u32(smem + p.off_rtab);
                        issue_qk<DPAD>(tSx, qa, kdesc(rt), make_idesc_f16(bf, kBlockM, p.n_rw, false));
                        issue_qk<DPAD>(tOx, qa, kdesc(rt + T::kBytes), make_idesc_f16(bf, kBlockM, p.n_rh, false));
                        mma_commit(&bar_g[x]);
                    } else {
                        // two ring stages: R_w rows [0,kTw) | [kTw,2kTw), then R_h's
                        for (int t = 0; t < 2; ++t) {
                            const int use = ring + t, st = use % nst;
                            if (!waitb(&bar_full_k[st], (use / nst) & 1, kStatusWaitK) ||
                                (!kMergeKV && !waitb(&bar_full_v[st], (use / nst) & 1, kStatusWaitV))) {
                                ok = false;
                                break;
                            }
                            const uint32_t kt = smem_u32(sRing + st * p.ring_stage_bytes);
                            const uint32_t dst = t == 0 ? tSx : tOx;
                            issue_qk_rows<DPAD, kTw>(dst, qa, kdesc(kt), idesc_s);
                            issue_qk_rows<DPAD, kTw>(dst + kTw, qa, kdesc(kt + kv_tile_bytes), idesc_s);
                        }
                        if (!ok) break;
                        mma_commit(&bar_g[x]);
                        mma_commit(&bar_empty[ring % nst]);
                        mma_commit(&bar_empty[(ring + 1) % nst]);
                        ring += 2;
                    }
                    // the scores overwrite G_w: every row must have gathered its terms
                    if (!waitb(&bar_gdone[x], ju & 1, kStatusWaitG)) { ok = false; break; }
                    const int n = shared_job<VL>(p, vt, job).n_kv;
                    const int sbase = s_cnt;
                    // S of key tile j into score buffer (sbase + j) & 1
                    auto issue_s = [&](int j) -> bool {
                        const int use = ring + j, st = use % nst, b = (sbase + j) & 1;
                        if (!waitb(&bar_full_k[st], (use / nst) & 1, kStatusWaitK)) return false;
                        issue_qk_rows<DPAD, kTw>(tSx + (uint32_t)kTw * (uint32_t)b, qa,
                                                kdesc(smem_u32(sRing + st * p.ring_stage_bytes)), idesc_s);
                        mma_commit(&bar_sb[x][b]);
                        return true;
                    };
                    for (int j = 0; ok && j < n && j < 2; ++j) ok = issue_s(j);
                    for (int j = 0; ok && j < n; ++j) {
                        const int use = ring + j, st = use % nst;
                        if (!waitb(bp, ph_p, kStatusWaitP) || (!kMergeKV && !waitb(&bar_full_v[st], (use / nst) & 1, kStatusWaitV))) {
                            ok = false;
                            break;
                        }
                        ph_p ^= 1;
                        issue_pv<kTw>(tOx, tPx + (uint32_t)kTw * (uint32_t)((sbase + j) & 1),
                                     vdesc_rows(smem_u32(sRing + st * p.ring_stage_bytes) + kv_tile_bytes, (uint32_t)kTw), idesc_o,
                                     j > 0 ? 1u : 0u);
                        if (j == n - 1) {
                            mma_commit(bo);
                            if (p.nq == 1) mma_commit(&bar_q_empty[x][qb]);
                        } else {
                            mma_commit(bpv);
                        }
                        mma_commit(&bar_empty[st]);
                        // tile j + 2 reuses tile j's score buffer: the softmax read it
                        // before it wrote P(j) there, and the P.V just issued reads
                        // P(j) before these scores land (in-order issue)
                        if (j + 2 < n) ok = issue_s(j + 2);
                    }
                    if (!ok) break;
                    s_cnt += n;
                    ring += n;
                } else if constexpr (kShDbl) {
                    // one score tile per job: S of the next job as soon as the
                    // softmax has read this one, then this job's P.V into O
                    // buffer ju & 1; Q is released by the commit of its S
                    const int st = ring % nst;
                    if (ju == 0) {
                        if (!waitb(&bar_q_full[x][0], 0, kStatusWaitQ) || !waitb(&bar_full_k[st], (ring / nst) & 1, kStatusWaitK)) {
                            ok = false;
                            break;
                        }
                        issue_qk<DPAD>(tSx, kdesc(smem_u32(sQ + (x * p.nq) * T::kBytes)),
                                       kdesc(smem_u32(sRing + st * p.ring_stage_bytes)), idesc_s);
                        mma_commit(bs);
                        mma_commit(&bar_q_empty[x][0]);
                        ++s_cnt;
                    }
                    if (job + job_step < p.n_jobs) {
                        const int ju2 = ju + 1, qb2 = ju2 % p.nq, st2 = (ring + 1) % nst;
                        if (!waitb(&bar_q_full[x][qb2], (ju2 / p.nq) & 1, kStatusWaitQ) ||
                            !waitb(&bar_full_k[st2], ((ring + 1) / nst) & 1, kStatusWaitK) || !s_free()) {
                            ok = false;
                            break;
                        }
                        issue_qk<DPAD>(tSx, kdesc(smem_u32(sQ + (x * p.nq + qb2) * T::kBytes)),
                                       kdesc(smem_u32(sRing + st2 * p.ring_stage_bytes)), idesc_s);
                        mma_commit(bs);
                        mma_commit(&bar_q_empty[x][qb2]);
                        ++s_cnt;
                    }
                    if (!waitb(bp, ph_p, kStatusWaitP) || (!kMergeKV && !waitb(&bar_full_v[st], (ring / nst) & 1, kStatusWaitV))) {
                        ok = false;
                        break;
                    }
                    ph_p ^= 1;
                    issue_pv<kCols>(tOx + (uint32_t)((ju & 1) * DPAD), tPx,
                                    vdesc(smem_u32(sRing + st * p.ring_stage_bytes + T::kBytes)), idesc_o, 0u);
                    mma_commit(bo);
                    mma_commit(&bar_empty[st]);
                    ring += 1;
                } else if constexpr (MODE == kModeShared) {
                    const int qb = ju % p.nq;
                    const uint64_t qa = kdesc(smem_u32(sQ + (x * p.nq + qb) * T::kBytes));
                    if (!waitb(&bar_q_full[x][qb], (ju / p.nq) & 1, kStatusWaitQ)) { ok = false; break; }
                    if constexpr (BIAS == kBiasSam) {
                        // the tables: a ring stage, or the CTA's resampled copies
                        const int st = ring % nst;
                        const uint32_t par = (ring / nst) & 1;
                        if (!p.sam_resample &&
                            (!waitb(&bar_full_k[st], par, kStatusWaitK) || (!kMergeKV && !waitb(&bar_full_v[st], par, kStatusWaitV)))) {
                            ok = false;
                            break;
                        }
                        // G_h rewrites O_x: the previous job's epilogue must be done with
                        // it.  (G in P_x: P_x was last read by this thread's P.V, which
                        // the tensor core finishes first, and written before that P.V;
                        // O_x is next written by this job's first P.V, which waits for
                        // P, which the softmax writes after its epilogue read O_x.)
                        if (!kGinP && ju > 0 && !waitb(&bar_oempty[x], (ju - 1) & 1, kStatusWaitO)) { ok = false; break; }
                        const uint32_t rw_a = p.sam_resample ? smem_u32(smem + p.off_rtab)
                                                             : smem_u32(sRing + st * p.ring_stage_bytes);
                        issue_qk<DPAD>(kGinP ? tPx : tSx, qa, kdesc(rw_a), make_idesc_f16(bf, kBlockM, p.n_rw, false));
                        issue_qk<DPAD>(kGinP ? tPx + 32 : tOx, qa, kdesc(rw_a + T::kBytes),
                                       make_idesc_f16(bf, kBlockM, p.n_rh, false));
                        mma_commit(&bar_g[x]);
                        if (!p.sam_resample) {
                            mma_commit(&bar_empty[st]);
                            ++ring;
                        }
                    }
                    const int n = shared_job<VL>(p, vt, job).n_kv;
                    {
                        const int st = ring % nst;
                        if (!waitb(&bar_full_k[st], (ring / nst) & 1, kStatusWaitK)) { ok = false; break; }
                        // with the SAM bias S_x rewrites the G_w values the slot is still gathering
                        if (BIAS == kBiasSam && !kGinP && !waitb(&bar_gdone[x], ju & 1, kStatusWaitG)) { ok = false; break; }
                        if (!s_free()) { ok = false; break; }
                        issue_qk<DPAD>(tSx, qa, kdesc(smem_u32(sRing + st * p.ring_stage_bytes)), idesc_s);
                        mma_commit(bs);
                        ++s_cnt;
                    }
                    for (int j = 0; j < n; ++j) {
                        const int use = ring + j;
                        const int st = use % nst;
                        const int st1 = (use + 1) % nst;
                        const uint64_t ka1 = kdesc(smem_u32(sRing + st1 * p.ring_stage_bytes));
                        const bool last = j == n - 1;
                        if (kSepP && !last) {
                            // next score tile first: it overlaps this tile's softmax
                            if (!waitb(&bar_full_k[st1], ((use + 1) / nst) & 1, kStatusWaitK) || !s_free()) { ok = false; break; }
                            issue_qk<DPAD>(tSx, qa, ka1, idesc_s);
                            mma_commit(bs);
                            ++s_cnt;
                        }
                        if (!waitb(bp, ph_p, kStatusWaitP) || (!kMergeKV && !waitb(&bar_full_v[st], (use / nst) & 1, kStatusWaitV))) {
                            ok = false;
                            break;
                        }
                        ph_p ^= 1;
                        issue_pv<kCols>(tOx, tPx, vdesc(smem_u32(sRing + st * p.ring_stage_bytes + T::kBytes)), idesc_o,
                                 j > 0 ? 1u : 0u);
                        if (last) {
                            mma_commit(bo);
                            if (p.nq == 1) mma_commit(&bar_q_empty[x][qb]);
                        } else if (kSepP) {
                            mma_commit(bpv);
                        }
                        mma_commit(&bar_empty[st]);
                        if (!kSepP && !last) {
                            if (!waitb(&bar_full_k[st1], ((use + 1) / nst) & 1, kStatusWaitK)) { ok = false; break; }
                            issue_qk<DPAD>(tSx, qa, ka1, idesc_s);
                            mma_commit(bs);
                            ++s_cnt;
                        }
                    }
                    ring += n;
                } else {
                    // separate mode: this slot's tile of the job is ring use `ring + x`
                    const int u = ring + x;
                    const uint32_t qa = smem_u32(sRing + (u % nst) * p.ring_stage_bytes);
                    // The next tile's scores are issued ahead (they overlap this
                    // tile's softmax) while this tile holds its stage: with both
                    // slots doing so that needs three stages, else a slot would
                    // wait for the stage it holds.
                    const bool ahead = nst >= 3;
                    // image-layout tiles are written by cp.async copies (generic
                    // proxy) that signal the barrier themselves: the reader's
                    // proxy fence orders them before its MMAs
                    const bool gathered = kVP || (BIAS == kBiasSwin && IMG && p.swin_image);
                    if (ju == 0 || !ahead) {
                        if (!waitb(&bar_full_k[u % nst], (u / nst) & 1, kStatusWaitK) || !s_free()) { ok = false; break; }
                        if (gathered) fence_proxy_async_smem();
                        sep_scores(2 * job + x, qa);
                        mma_commit(bs);
                        ++s_cnt;
                    }
                    const int next = job + job_step;
                    if (ahead && next < p.n_jobs) {
                        // next tile's scores first: they overlap this tile's softmax
                        const int u2 = u + 2;
                        if (!waitb(&bar_full_k[u2 % nst], (u2 / nst) & 1, kStatusWaitK) || !s_free()) { ok = false; break; }
                        if (gathered) fence_proxy_async_smem();
                        sep_scores(2 * next + x, smem_u32(sRing + (u2 % nst) * p.ring_stage_bytes));
                        mma_commit(bs);
                        ++s_cnt;
                    }
                    if (!waitb(bp, ph_p, kStatusWaitP)) { ok = false; break; }
                    ph_p ^= 1;
                    if constexpr (kVP) {
                        // one slice at a time: its P columns against its own
                        // value rows, after the previous slice's rows have read O
                        const uint64_t vd = vdesc(qa + 2 * T::kBytes);
                        for (int g = 0; g < kBlockM / SL; ++g) {
                            if (g > 0) {
                                if (!waitb(&bar_ohand[x], hand_cnt & 1, kStatusWaitO)) { ok = false; break; }
                                ++hand_cnt;
                            }
                            issue_pv<SL>(tOx, tPx + (uint32_t)(g * (SL / 2)), vd + (uint64_t)(g * (SL / 16) * 32), idesc_o,
                                         0u);
                            mma_commit(&bar_og[x][g]);
                        }
                        if (!ok) break;
                        mma_commit(&bar_empty[u % nst]);
                    } else {
                        issue_pv(tOx + (kDblO ? (uint32_t)((ju & 1) * DPAD) : 0u), tPx, vdesc(qa + 2 * T::kBytes),
                                 idesc_o, 0u);
                        mma_commit(&bar_empty[u % nst]);
                        mma_commit(bo);
                    }
                    ring += 2;
                }
            }
            // every MMA issued has retired before tensor memory is released
            mma_commit(&bar_final);
            mbar_wait(&bar_final, 0, nullptr, 0);
        }
      }
    } else {
        regs_inc<kSoftmaxRegs>();
        // ============================================================ softmax
        const int x = warp >> 2;                // slot A or B
        const int r = tid & 127;                // row in tile == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + (uint32_t)(kDbS ? 256 * x : (kSepP ? kCols : 128) * x);
        const uint32_t tP = kSepP ? tmem + lane_base + (uint32_t)(kOffP + 64 * x) : tS;  // kDbS: + 64 * buffer
        const uint32_t tO = kDbS ? tS + 128 : tmem + lane_base + (uint32_t)(kSepP ? kOffO + kOw * x : 256 + 128 * x);
        int pvd_cnt = 0;  // P.V completions of this slot awaited (separate P buffers)
        // Q buffer whose staged output rows a bulk copy is still reading (-1:
        // none); it goes back to the producer during the next job
        int q_pending = -1;
        auto release_q = [&]() {
            if (q_pending < 0) return;
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            warp_arrive(&bar_q_empty[x][q_pending]);
            q_pending = -1;
        };
        int cnt_s = 0, ju = 0;
        bool ok = true;
        const float2 scale2 = make_float2(p.scale_log2, p.scale_log2);
        float* sam_rh = nullptr;
        float* sam_rw = nullptr;
        const int* sam_kt = nullptr;
        if constexpr (BIAS == kBiasSam) {
            sam_rh = sExtra + x * (p.k_h * kBlockM);
            sam_rw = sExtra + 2 * p.k_h * kBlockM + x * (p.k_w * kBlockM);
            sam_kt = reinterpret_cast<const int*>(sExtra + 2 * (p.k_h + p.k_w) * kBlockM);
        }

        // kVP: this warp's slice is not the tile's last, so its reading of O
        // hands O over to the next slice's P.V
        bool vp_hand = false;
        // O / l rounded to the output type and stored (row-per-thread, 16 bytes at a time)
        // m: the row's reference maximum in log2 units (P = 2^(x - m)), for the
        // row's log-sum-exp (m + log2 l) ln 2 when the caller asked for it
        auto epilogue = [&](uint32_t tObuf, float l, float m, int slice, int tok, bool rok, int qbuf) {
            const float inv_l = l > 0.f ? 1.0f / l : 0.f;
            if (p.lse != nullptr && rok && !DBG)
                p.lse[(size_t)slice * p.Nq + tok] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            uint32_t o[DPAD / 2];
            {
                uint32_t v[DPAD];
                tmem_ld_cols<DPAD>(tObuf, v);
                if (bf) {
#pragma unroll
                    for (int t = 0; t < DPAD; t += 2)
                        o[t / 2] = pack_bf16(__uint_as_float(v[t]) * inv_l, __uint_as_float(v[t + 1]) * inv_l);
                } else {
#pragma unroll
                    for (int t = 0; t < DPAD; t += 2)
                        o[t / 2] = pack_f16(__uint_as_float(v[t]) * inv_l, __uint_as_float(v[t + 1]) * inv_l);
                }
            }
            if constexpr (BIAS == kBiasSam) {
                // O_x is free for the next job's G_h
                tc_fence_before();
                warp_arrive(&bar_oempty[x]);
            }
            if constexpr (kVP) {
                if (vp_hand) {
                    tc_fence_before();
                    warp_arrive(&bar_ohand[x]);
                }
            }
            if (MODE == kModeShared && (kShDbl || p.nq == 2)) {
                // The warp's 32 output rows, consecutive tokens of one slice,
                // are staged: in the slot's finished Q tile (every P.V of the
                // job is done), which then goes back to the producer, or, in
                // the one-tile pipeline, in its own staging area, written
                // again one job later.  With kBulkOut they leave in one bulk
                // copy (async proxy) of their contiguous bytes, issued by lane
                // 0, so the warp issues no stores; a Q tile then goes back
                // once the copy has read it -- during the next job, after its
                // first scores, so that the copy is not waited for here.
                // Otherwise the warp stores them, 512 contiguous bytes per
                // instruction.
                const int rb = p.d * 2;  // bytes per output row (a multiple of 16)
                unsigned char* stg = (kShDbl ? sExtraB + x * (kBlockM * rb) : sQ + (x * p.nq + qbuf) * T::kBytes) +
                                     (warp & 3) * (32 * rb);
                if (!DBG) {
                    if constexpr (kShDbl) {
                        // the copy of this warp's previous rows has read them
                        if (lane == 0) bulk_wait_read0();
                        __syncwarp();
                    }
#pragma unroll
                    for (int c = 0; c < DPAD / 8; ++c)
                        if (c * 8 < p.d)
                            *reinterpret_cast<uint4*>(stg + lane * rb + c * 16) =
                                make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                    if constexpr (kBulkOut) fence_proxy_async_smem();  // read through the async proxy
                    __syncwarp();
                    const int nvalid = __popc(__ballot_sync(0xffffffffu, rok));  // a prefix of the lanes
                    unsigned char* dst = reinterpret_cast<unsigned char*>(p.out) +
                                         ((size_t)__shfl_sync(0xffffffffu, slice, 0) * p.Nq +
                                          __shfl_sync(0xffffffffu, tok, 0)) * (size_t)rb;
                    if constexpr (kBulkOut) {
                        if (lane == 0 && nvalid > 0) {
                            bulk_s2g(dst, stg, (uint32_t)(nvalid * rb));
                            bulk_commit();
                        }
                    } else {
                        const int nch = nvalid * rb / 16;
                        for (int q = lane; q < nch; q += 32)
                            *reinterpret_cast<uint4*>(dst + (size_t)q * 16) = *reinterpret_cast<const uint4*>(stg + q * 16);
                    }
                }
                if constexpr (!kShDbl) {
                    if (!kBulkOut || DBG) {
                        // generic accesses before the producer's next TMA write here
                        fence_proxy_async_smem();
                        warp_arrive(&bar_q_empty[x][qbuf]);
                    } else {
                        q_pending = qbuf;
                    }
                } else {
                    __syncwarp();
                }
            } else if (rok && !DBG) {
                // windows layout: [slice][token]; image layout: the token's
                // place in the image (shift and partition undone)
                const size_t orow = (MODE == kModeSeparate && BIAS == kBiasSwin && IMG && p.swin_image)
                                        ? swin_image_row((uint32_t)slice, (uint32_t)tok, p.H, p.n_w, p.n_ww, p.win,
                                                         p.grid_h, p.grid_w, p.shift, p.fd_h, p.fd_w, p.fd_ww, p.fd_m)
                                        : (size_t)slice * p.Nq + tok;
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(p.out) + orow * (size_t)p.d * 2);
#pragma unroll
                for (int c = 0; c < DPAD / 8; ++c)
                    if (c * 8 < p.d) dst[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            }
        };
        // the previous job's row (pipelined epilogue)
        float pv_l = 0.f, pv_m = 0.f;
        int pv_slice = 0, pv_tok = 0;
        bool pv_ok = false;

        for (int job = job0; ok && job < p.n_jobs; job += job_step, ++ju) {
            // ------------------------------------------------- row of this job
            int my_slice, my_tok, my_sl = 0;
            int vp_nk = 0, vp_orow = 0;  // kVP: the slice's key count, the row's output row
            bool row_ok;
            JobRows jr{};
            if constexpr (MODE == kModeShared) {
                jr = shared_job<VL>(p, vt, job);
                my_slice = jr.q_slice;
                my_tok = jr.q0 + x * kBlockM + r;
                row_ok = my_tok < jr.nq;
            } else {
                const int tile = 2 * job + x;
                my_sl = r / SL;
                my_slice = tile * p.g + my_sl;
                my_tok = r - my_sl * SL;
                row_ok = (my_tok < p.Nq) && (my_sl < p.g) && (my_slice < p.BH);
                if constexpr (kVP) {
                    // the slice's sequence and head (a slice past the last has
                    // no rows and no keys)
                    int lq = 0;
                    if (my_slice < p.BH) {
                        const int e = my_slice / p.H, h = my_slice - e * p.H;
                        lq = vt.q_len[e];
                        vp_nk = vt.k_len[e];
                        vp_orow = p.H * vt.q_off[e] + h * lq + my_tok;
                    }
                    row_ok = my_tok < lq;
                }
            }
            float l_run = 0.f;
            float m_fin = 0.f;  // the row's reference maximum (log2 units) once its keys are done

            if constexpr (MODE == kModeSeparate) {
                // ---------------------------- one key tile: own slot's SL columns
                __syncwarp();
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_s[x], cnt_s & 1, abort_flag, kStatusWaitS))) { ok = false; break; }
                ++cnt_s;
                tc_fence_after();
                float xs[SL];
                {
                    uint32_t v[SL];
                    tmem_ld_cols<SL>(tS + my_sl * SL, v);
#pragma unroll
                    for (int t = 0; t < SL; ++t) xs[t] = __uint_as_float(v[t]);
                }
                // S_x may now be overwritten by the next tile's scores
                tc_fence_before();
                warp_arrive(&bar_sfree[x]);
                const int nk = kVP ? vp_nk : p.Nk;
                float sc = p.scale_log2;  // multiplier of xs in the exponent
                if (BIAS == kBiasSwin && SL <= 64 && SWR) {
                    // xs = s * scale * log2(e) + bias row (+ region mask), log2 units
                    int h, kind;
                    swin_slice_info((uint32_t)min(my_slice, p.BH - 1), p.H, p.n_w, p.n_ww, p.n_wh, p.shift, p.fd_h,
                                    p.fd_w, p.fd_ww, h, kind);
                    const unsigned char* rowp = sExtraB + (h * SL + my_tok) * SL * 4;
                    float* dbg_row = (DBG && row_ok) ? p.dbg + ((size_t)my_slice * p.Nq + my_tok) * p.Nk : nullptr;
                    if (kind) {
                        const uint32_t* mrow = reinterpret_cast<const uint32_t*>(sExtraB + p.H * SL * SL * 4) +
                                               ((kind - 1) * SL + my_tok) * (SL / 32);
                        swin_add_bias_row<SL, kNc, true, DBG>(xs, rowp, my_tok & 7, mrow, p.scale_log2, dbg_row, nk);
                    } else {
                        swin_add_bias_row<SL, kNc, false, DBG>(xs, rowp, my_tok & 7, nullptr, p.scale_log2, dbg_row, nk);
                    }
                    sc = 1.0f;
                } else if constexpr (DBG) {
                    // the scores hold only the bias when debugging (no Q.K^T)
                    if (row_ok) {
                        float* dst = p.dbg + ((size_t)my_slice * p.Nq + my_tok) * p.Nk;
#pragma unroll
                        for (int c = 0; c < SL; ++c)
                            if (c < nk) dst[c] = (BIAS == kBiasSwin) ? xs[c] : 0.f;
                    }
                }
                if (!(sc > 0.f)) {
                    // a scale <= 0: the multiplier goes on first, so that the
                    // -inf of the masked keys below stays -inf
                    const float2 s2 = make_float2(sc, sc);
#pragma unroll
                    for (int c = 0; c < kNe; c += 2) {
                        const float2 y = __fmul2_rn(make_float2(xs[c], xs[c + 1]), s2);
                        xs[c] = y.x;
                        xs[c + 1] = y.y;
                    }
                    sc = 1.0f;
                }
                if constexpr (kNc == SL) {
                    // keys past the slice length: -inf (16-column chunks, uniform branches)
#pragma unroll
                    for (int c0 = 0; c0 < SL; c0 += 16) {
                        if (c0 + 16 > nk) {
#pragma unroll
                            for (int t = 0; t < 16; ++t)
                                if (c0 + t >= nk) xs[c0 + t] = -INFINITY;
                        }
                    }
                } else if constexpr (kNe > kNc) {
                    xs[kNc] = -INFINITY;  // the odd column that completes the last pair
                }
                const float m = row_max<kNc>(xs) * sc;
                const float m_use = (m == -INFINITY) ? 0.f : m;
                m_fin = m_use;
                uint32_t own[SL / 2];
#pragma unroll
                for (int t = kNe / 2; t < SL / 2; ++t) own[t] = 0u;  // keys past the window
                l_run = exp_pack<kNe>(xs, sc, -m_use, bf, own);
                if constexpr (kDblO) {
                    // the previous tile's output, while this tile's P waits in
                    // registers: its P.V has run during this tile's softmax
                    if (ju > 0) {
                        __syncwarp();
                        if (!__all_sync(0xffffffffu, mbar_wait(&bar_o[x], (ju - 1) & 1, abort_flag, kStatusWaitO))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        epilogue(tO + ((ju - 1) & 1) * DPAD, pv_l, pv_m, pv_slice, pv_tok, pv_ok, 0);
                    }
                }
                if (ju == 0) {
                    // a row's columns outside its own slice stay zero from here on:
                    // only this row's thread writes them
                    uint32_t pk[64];
#pragma unroll
                    for (int t = 0; t < 64; ++t) pk[t] = 0u;
#pragma unroll
                    for (int s = 0; s < 128 / SL; ++s)
                        if (s == my_sl)
#pragma unroll
                            for (int t = 0; t < SL / 2; ++t) pk[s * (SL / 2) + t] = own[t];
                    tmem_st64(tP, pk);
                } else {
                    tmem_st_cols<SL / 2>(tP + (uint32_t)(my_sl * (SL / 2)), own);
                }
                tmem_st_wait();
                tc_fence_before();
                warp_arrive(&bar_p[x]);
                if constexpr (kDblO) {
                    pv_l = l_run;
                    pv_m = m_fin;
                    pv_slice = my_slice;
                    pv_tok = my_tok;
                    pv_ok = row_ok;
                    continue;
                }
            } else if constexpr (kDbS) {
                // -------------- SAM, 64 x 64 (48 x 48) grid: one grid row per score tile
                // Key tile j is key row kh = j.  rel_w of the row (kTw values,
                // log2 units) stays in registers for the job as aligned pairs,
                // one 64-bit operand of the packed FMA each; rel_h goes to shared
                // memory as fp16, [slot][kh][row], one load per tile.
                __half* const rh16 = reinterpret_cast<__half*>(sExtraB) + x * (64 * kBlockM);
                const int qh = min(my_tok / kTw, kTw - 1), qw = my_tok % kTw;
                __syncwarp();
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_g[x], ju & 1, abort_flag, kStatusWaitG))) { ok = false; break; }
                tc_fence_after();
                const float f = DBG ? 1.0f : kLog2e;
                float2 rw2[kTw / 2];
                {
                    float gv[128];
                    {
                        uint32_t v[128];
                        tmem_ld_cols<128>(tS, v);  // G_w row
#pragma unroll
                        for (int t = 0; t < 128; ++t) gv[t] = __uint_as_float(v[t]) * f;
                    }
                    // rel_w for key column kw is G_w[qw + kTw - 1 - kw]
                    shift_down<128, 6>(gv, qw);
#pragma unroll
                    for (int u = 0; u < kTw / 2; ++u) rw2[u] = make_float2(gv[kTw - 1 - 2 * u], gv[kTw - 2 - 2 * u]);
                    {
                        uint32_t v[128];
                        tmem_ld_cols<128>(tO, v);  // G_h row
#pragma unroll
                        for (int t = 0; t < 128; ++t) gv[t] = __uint_as_float(v[t]) * f;
                    }
                    // rel_h for key row kh is G_h[qh + kTw - 1 - kh]
                    shift_down<128, 6>(gv, qh);
#pragma unroll
                    for (int u = 0; u < kTw; ++u) rh16[u * kBlockM + r] = __float2half_rn(gv[kTw - 1 - u]);
                }
                tc_fence_before();
                warp_arrive(&bar_gdone[x]);

                float m_run = -INFINITY;
                for (int j = 0; j < jr.n_kv; ++j) {
                    const int b = cnt_s & 1;
                    __syncwarp();
                    if (!__all_sync(0xffffffffu, mbar_wait(&bar_sb[x][b], (cnt_s >> 1) & 1, abort_flag, kStatusWaitS))) {
                        ok = false;
                        break;
                    }
                    ++cnt_s;
                    tc_fence_after();
                    float xs[kTw];
                    {
                        uint32_t v[kTw];
                        tmem_ld_cols<kTw>(tS + (uint32_t)kTw * (uint32_t)b, v);
#pragma unroll
                        for (int t = 0; t < kTw; ++t) xs[t] = __uint_as_float(v[t]);
                    }
                    const float rh = __half2float(rh16[min(j, kTw - 1) * kBlockM + r]);
                    if constexpr (DBG) {
                        if (row_ok) {
                            float* dst = p.dbg + ((size_t)my_slice * p.Nq + my_tok) * p.Nk + j * kTw;
#pragma unroll
                            for (int c = 0; c < kTw; c += 2) {
                                dst[c] = rw2[c / 2].x + rh;
                                dst[c + 1] = rw2[c / 2].y + rh;
                            }
                        }
                    }
                    // x = s * scale * log2(e) + rel_w; the row's rel_h is constant
                    // over the tile and joins through the max and the exponent's
                    // offset (the bias goes on first, so any sign of the scale works)
#pragma unroll
                    for (int c = 0; c < kTw; c += 2) {
                        const float2 y = __ffma2_rn(make_float2(xs[c], xs[c + 1]), scale2, rw2[c / 2]);
                        xs[c] = y.x;
                        xs[c + 1] = y.y;
                    }
                    const float m_tile = row_max<kTw>(xs) + rh;
                    // the previous P.V must be done before O is rescaled; every tile
                    // after the first consumes that completion, at the latest just
                    // before its P is handed over
                    bool pv_waited = j == 0;
                    auto wait_pv = [&]() -> bool {
                        if (pv_waited) return true;
                        pv_waited = true;
                        __syncwarp();
                        if (!__all_sync(0xffffffffu, mbar_wait(&bar_pvd[x], pvd_cnt & 1, abort_flag, kStatusWaitO))) return false;
                        ++pvd_cnt;
                        tc_fence_after();
                        return true;
                    };
                    const float m_new = fmaxf(m_run, m_tile);
                    const bool need = m_new > m_run + kRescaleThreshold;
                    const bool any_rescale = __any_sync(0xffffffffu, need && j > 0);
                    if (any_rescale) {
                        if (!wait_pv()) { ok = false; break; }
                        const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
#pragma unroll
                        for (int c0 = 0; c0 < DPAD; c0 += 16) {
                            uint32_t w16[16];
                            tmem_ld16(tO + c0, w16);
#pragma unroll
                            for (int t = 0; t < 16; ++t) w16[t] = __float_as_uint(__uint_as_float(w16[t]) * alpha);
                            tmem_st16(tO + c0, w16);
                        }
                    }
                    if (need) {
                        l_run *= ex2_approx(m_run - m_new);
                        m_run = m_new;
                    }
                    const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
                    uint32_t pk[kTw / 2];
                    l_run += exp_pack<kTw>(xs, 1.0f, rh - m_use, bf, pk);
                    tmem_st_cols<kTw / 2>(tP + (uint32_t)kTw * (uint32_t)b, pk);
                    tmem_st_wait();
                    if (!wait_pv()) { ok = false; break; }
                    tc_fence_before();
                    warp_arrive(&bar_p[x]);
                }
                if (!ok) break;
                m_fin = (m_run == -INFINITY) ? 0.f : m_run;
            } else {
                // ------------------------------------------------- bias row setup
                // rel_w of the row for kw = 2u, 2u + 1, held as fp16 pairs (half the
                // registers of fp32; grid widths here are even, so a pair never
                // straddles two key rows)
                __half2 sam_rw_h2[SW > 0 ? SW / 2 : 1];
                if constexpr (BIAS == kBiasSam) {
                    const int qh = my_tok / p.s_w, qw = my_tok % p.s_w;
                    __syncwarp();
                    if (!__all_sync(0xffffffffu, mbar_wait(&bar_g[x], ju & 1, abort_flag, kStatusWaitG))) { ok = false; break; }
                    tc_fence_after();
                    const float f = DBG ? 1.0f : kLog2e;
                    if (SW == 0 && p.sam_general) {
                        // unequal grids (the generic kernel only: the host sends
                        // square grids alone to the kernels specialised for a side):
                        // each key row / column reads its table row through the
                        // coordinate scalers, linearly resampled from G when the
                        // tables have another length (resampling commutes with Q.R)
                        sam_general_rows(tS, tO, p, min(qh, p.s_h - 1), min(qw, p.s_w - 1), f, sam_rh, sam_rw, r);
                        tc_fence_before();
                        warp_arrive(&bar_gdone[x]);
                    } else {
                    // square grids of side SW <= 16 need 32-value G rows and 4-bit
                    // shifts, side 64 needs 6-bit shifts
                    constexpr int kGW = (SW > 0 && SW <= 16) ? 32 : 128;
                    constexpr int kGB = (SW > 0 && SW <= 16) ? 4 : (SW > 0 ? 6 : 7);
                    float gv[kGW];
                    // G_w row: rel_w for key column kw is G_w[qw + s_w - 1 - kw]
                    {
                        uint32_t v[kGW];
                        tmem_ld_cols<kGW>(kGinP ? tP : tS, v);
#pragma unroll
                        for (int t = 0; t < kGW; ++t) gv[t] = __uint_as_float(v[t]) * f;
                    }
                    shift_down<kGW, kGB>(gv, qw);
                    if constexpr (SW > 0) {
#pragma unroll
                        for (int u = 0; u < SW / 2; ++u) sam_rw_h2[u] = __floats2half2_rn(gv[SW - 1 - 2 * u], gv[SW - 2 - 2 * u]);
                    } else {
#pragma unroll
                        for (int u = 0; u < kSamMaxSide; ++u)
                            if (u < p.s_w) sam_rw[u * kBlockM + r] = gv[u];
                    }
                    // G_h row: rel_h for key row kh is G_h[qh + s_h - 1 - kh]
                    {
                        uint32_t v[kGW];
                        tmem_ld_cols<kGW>(kGinP ? tP + 32 : tO, v);
#pragma unroll
                        for (int t = 0; t < kGW; ++t) gv[t] = __uint_as_float(v[t]) * f;
                    }
                    shift_down<kGW, kGB>(gv, qh);
#pragma unroll
                    for (int u = 0; u < (kSamMaxSide < kGW ? kSamMaxSide : kGW); ++u)
                        if (u < p.s_h) sam_rh[u * kBlockM + r] = gv[u];
                    tc_fence_before();
                    warp_arrive(&bar_gdone[x]);
                    }
                }

                // ------------------------------------------------------ key tiles
                float m_run = -INFINITY;
                for (int j = 0; j < jr.n_kv; ++j) {
                    __syncwarp();
                    if (!__all_sync(0xffffffffu, mbar_wait(&bar_s[x], cnt_s & 1, abort_flag, kStatusWaitS))) { ok = false; break; }
                    ++cnt_s;
                    tc_fence_after();
                    if (kBulkOut && j == 0) release_q();  // the last job's Q tile, once its output copy has read it
                    float xs[kCols];
                    {
                        uint32_t v[kCols];
                        tmem_ld_cols<kCols>(tS, v);
#pragma unroll
                        for (int t = 0; t < kCols; ++t) xs[t] = __uint_as_float(v[t]);
                    }
                    if constexpr (kSepP) {
                        // S_x may now be overwritten by the next tile's scores
                        tc_fence_before();
                        warp_arrive(&bar_sfree[x]);
                    }
                    const int key0 = j * p.kv_w;
                    const int hi = min(p.kv_w, jr.nk - key0);  // valid key columns [0, hi)
                    float m_tile;  // log2 units
                    float sc;      // multiplier applied to xs in the exponent
                    if (BIAS == kBiasNone && !DBG) {
                        // no bias: max on raw scores, p = 2^(s*scale*log2e - m)
                        if (NS && !(p.scale_log2 > 0.f)) {
                            // a scale <= 0: scale first, then mask the keys past the
                            // sequence with -inf (-inf times the scale would not stay -inf)
                            const float2 s2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
                            for (int c = 0; c < kCols; c += 2) {
                                const float2 y = __fmul2_rn(make_float2(xs[c], xs[c + 1]), s2);
                                xs[c] = c < hi ? y.x : -INFINITY;
                                xs[c + 1] = c + 1 < hi ? y.y : -INFINITY;
                            }
                            m_tile = row_max<kCols>(xs);
                            sc = 1.0f;
                        } else {
                            if (hi < kCols) {
#pragma unroll
                                for (int c0 = 0; c0 < kCols; c0 += 16)
                                    if (c0 + 16 > hi)
#pragma unroll
                                        for (int t = 0; t < 16; ++t)
                                            if (c0 + t >= hi) xs[c0 + t] = -INFINITY;
                            }
                            m_tile = row_max<kCols>(xs) * p.scale_log2;
                            sc = p.scale_log2;
                        }
                    } else {
                        constexpr int kRows = (BIAS == kBiasSam && SW > 0) ? (128 + (SW > 0 ? SW : 1) - 1) / (SW > 0 ? SW : 1) : 1;
                        float rh_tile[kRows];
                        if constexpr (BIAS == kBiasSam && SW > 0) {
                            // key rows of this tile; the tile starts at a multiple of SW
                            const int kh0 = key0 / SW;
#pragma unroll
                            for (int rr = 0; rr < kRows; ++rr) {
                                const int kh = min(kh0 + rr, p.k_h - 1);
                                rh_tile[rr] = sam_rh[(p.k_h - 1 - kh) * kBlockM + r];
                            }
                        }
#pragma unroll
                        for (int c = 0; c < kCols; c += 2) {
                            float b0 = 0.f, b1 = 0.f;
                            if constexpr (BIAS == kBiasSam) {
                                if constexpr (SW > 0) {
                                    const float2 rw = __half22float2(sam_rw_h2[(c % SW) / 2]);
                                    b0 = rh_tile[c / SW] + rw.x;
                                    b1 = rh_tile[c / SW] + rw.y;
                                } else {
                                    const int k0 = sam_kt[min(key0 + c, p.Nk - 1)];
                                    const int k1 = sam_kt[min(key0 + c + 1, p.Nk - 1)];
                                    b0 = sam_rh[(k0 & 0xFFFF) * kBlockM + r] + sam_rw[(k0 >> 16) * kBlockM + r];
                                    b1 = sam_rh[(k1 & 0xFFFF) * kBlockM + r] + sam_rw[(k1 >> 16) * kBlockM + r];
                                }
                            }
                            if constexpr (DBG) {
                                if (row_ok) {
                                    float* dst = p.dbg + ((size_t)my_slice * p.Nq + my_tok) * p.Nk + key0;
                                    if (c < hi) dst[c] = b0;
                                    if (c + 1 < hi) dst[c + 1] = b1;
                                }
                            }
                            float2 bv = make_float2(b0, b1);
                            if constexpr (DBG) bv = __fmul2_rn(bv, make_float2(kLog2e, kLog2e));
                            const float2 y = __ffma2_rn(make_float2(xs[c], xs[c + 1]), scale2, bv);
                            xs[c] = y.x;
                            xs[c + 1] = y.y;
                        }
                        if (hi < kCols) {
#pragma unroll
                            for (int c0 = 0; c0 < kCols; c0 += 16)
                                if (c0 + 16 > hi)
#pragma unroll
                                    for (int t = 0; t < 16; ++t)
                                        if (c0 + t >= hi) xs[c0 + t] = -INFINITY;
                        }
                        m_tile = row_max<kCols>(xs);
                        sc = 1.0f;
                    }
                    // With separate P buffers the previous P.V may still be running:
                    // it must be done before O is rescaled or P_x rewritten.
                    bool pv_waited = !(kSepP && j > 0);
                    auto wait_pv = [&]() -> bool {
                        if (pv_waited) return true;
                        pv_waited = true;
                        __syncwarp();
                        if (!__all_sync(0xffffffffu, mbar_wait(&bar_pvd[x], pvd_cnt & 1, abort_flag, kStatusWaitO))) return false;
                        ++pvd_cnt;
                        tc_fence_after();
                        return true;
                    };
                    const float m_new = fmaxf(m_run, m_tile);
                    const bool need = m_new > m_run + kRescaleThreshold;
                    const bool any_rescale = __any_sync(0xffffffffu, need && j > 0);
                    if (any_rescale && !wait_pv()) { ok = false; break; }
                    if (any_rescale) {
                        // O holds the earlier tiles' P.V, complete (with a shared P/S
                        // buffer this score tile was committed after it)
                        const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
                        // 16 columns at a time: the score row is live in registers
#pragma unroll
                        for (int c0 = 0; c0 < DPAD; c0 += 16) {
                            uint32_t w16[16];
                            tmem_ld16(tO + c0, w16);
#pragma unroll
                            for (int t = 0; t < 16; ++t) w16[t] = __float_as_uint(__uint_as_float(w16[t]) * alpha);
                            tmem_st16(tO + c0, w16);
                        }
                    }
                    if (need) {
                        l_run *= ex2_approx(m_run - m_new);
                        m_run = m_new;
                    }
                    const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
                    uint32_t pk[kCols / 2];
                    l_run += exp_pack<kCols>(xs, sc, -m_use, bf, pk);
                    if (!wait_pv()) { ok = false; break; }
                    if constexpr (kShDbl) {
                        // the previous job's output, while this job's P waits in
                        // registers: its P.V ran during this softmax (and P_x
                        // is free once it has)
                        if (ju > 0) {
                            __syncwarp();
                            if (!__all_sync(0xffffffffu, mbar_wait(&bar_o[x], (ju - 1) & 1, abort_flag, kStatusWaitO))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            epilogue(tO + ((ju - 1) & 1) * DPAD, pv_l, pv_m, pv_slice, pv_tok, pv_ok, 0);
                        }
                    }
                    tmem_st_cols<kCols / 2>(tP, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    warp_arrive(&bar_p[x]);
                }
                if (!ok) break;
                m_fin = (m_run == -INFINITY) ? 0.f : m_run;
            }

            // -------------------------------------------------------- epilogue
            if constexpr (kShDbl) {  // written during the next job (or after the last)
                pv_l = l_run;
                pv_m = m_fin;
                pv_slice = my_slice;
                pv_tok = my_tok;
                pv_ok = row_ok;
                continue;
            }
            __syncwarp();
            uint64_t* ob = &bar_o[x];
            if constexpr (kVP) ob = &bar_og[x][my_sl];  // the P.V of this row's slice
            if (!__all_sync(0xffffffffu, mbar_wait(ob, ju & 1, abort_flag, kStatusWaitO))) { ok = false; break; }
            tc_fence_after();
            if constexpr (kVP) {
                vp_hand = my_sl < kBlockM / SL - 1;
                epilogue(tO, l_run, m_fin, 0, vp_orow, row_ok, 0);
            } else if constexpr (VL)  // output rows counted from the buffer start
                epilogue(tO, l_run, m_fin, 0, jr.out_row0 + my_tok, row_ok, ju % p.nq);
            else
                epilogue(tO, l_run, m_fin, my_slice, my_tok, row_ok, MODE == kModeShared ? ju % p.nq : 0);
        }
        if constexpr (kDblO || kShDbl) {
            if (ok && ju > 0) {
                __syncwarp();
                if (__all_sync(0xffffffffu, mbar_wait(&bar_o[x], (ju - 1) & 1, abort_flag, kStatusWaitO))) {
                    tc_fence_after();
                    epilogue(tO + ((ju - 1) & 1) * DPAD, pv_l, pv_m, pv_slice, pv_tok, pv_ok, 0);
                }
            }
        }
        if constexpr (kBulkOut) {
            release_q();
            // the output copies have completed before the CTA retires
            if (lane == 0) bulk_wait0();
            __syncwarp();
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
