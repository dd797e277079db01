// sdpa09_api.cu -- the C ABI declared in include/sdpa09.h: argument
// validation, TMA tensor-map encoding, tiling choice and launch.
//
// The call never allocates, copies host<->device or synchronises: the
// bias arguments are read from the host struct and passed by value in the
// kernel parameters ("PyTorch团队重写「分割一切」模型，比原始实现快8倍", bf16 section:
// host-side index coordinates forced a copy plus a blocking stream
// synchronisation; the boundary is built so that cannot happen here).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/sdpa09.h"
#include "attn_bwd_long.cuh"
#include "attn_bwd_sam.cuh"
#include "attn_launch.cuh"

namespace sdpa09 {

cudaError_t launch_bwd_win(int dpad, bool swin, const BwdMaps& tm, const BwdTcParams& p, int grid, size_t smem,
                           cudaStream_t stream);
cudaError_t launch_bwd_long(int dpad, int mode, int sw, const BwdMaps& tm, const BwdLongParams& p, int grid,
                            size_t smem, cudaStream_t stream);
namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

// Status word written by kernels whose bounded waits ran out.
__device__ int g_status_word;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Exercises the failure path of the bounded waits: one warp waits on an
// mbarrier that nothing ever arrives on, through the same mbar_wait the
// attention kernel uses but with a short limit; the wait gives up, records
// its code in the CTA abort word, and the kernel reports it in the status
// word exactly as the attention kernel's teardown does.
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_sh;
    if (threadIdx.x == 0) {
        abort_sh = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    volatile int* abort_flag = &abort_sh;
    const bool ok = mbar_wait(&bar, 0, abort_flag, kStatusWaitSelfTest, limit_ns);
    __syncwarp();
    if (threadIdx.x == 0 && !ok && abort_sh != 0) atomicCAS(status, 0, abort_sh);
}

int* status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    static int* ptrs[64] = {nullptr};
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return nullptr;
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

// Scratch of attn_bwd_noalloc: the per-row D of the long-sequence backward
// (4 MiB, rows B * H * Nq <= 2^20).  Every GPU that loads the library holds it
// until the process exits; all calls share it.
constexpr int kNoAllocRows = 1 << 20;
static __device__ __align__(256) float g_bwd_scratch[kNoAllocRows];

// Device address of g_bwd_scratch on the current device, looked up once per
// device (the host-side name of the array is only a stand-in for it).
float* noalloc_scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    static float* ptrs[64] = {nullptr};
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return nullptr;
    if (!ptrs[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<float*>(ptr);
    }
    return ptrs[dev];
}

// Generic tiled map with 32-byte swizzle over 16-bit elements.
int encode(CUtensorMap* m, const void* base, bool bf16, int rank, const uint64_t* dims,
           const uint64_t* strides_bytes, const uint32_t* box) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    CUresult r = enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ATTN_OK;
}

// Maps of a [slices][rows][d] tensor (slices = 0: a plain [rows][d] table).
// The full map is (16 elements, row, slice, column block) with a box of
// (16, box_rows, box_slices, atoms - part): one copy lands every 16-column
// block of the tile as [block][row][16]; blocks and rows past the data are
// zero-filled.  When d is not a multiple of 16 the partial map covers the
// last block: (d mod 16 elements, row, slice), box (16, box_rows, box_slices).
int encode_operand(CUtensorMap* full, CUtensorMap* partial, const void* base, bool bf16, int d,
                   int64_t rows, int64_t slices, int atoms, int box_rows, int box_slices) {
    const int fa = d / 16, rem = d % 16;
    const int part = (fa > 0 && rem) ? 1 : 0;
    const bool table = slices == 0;
    const uint64_t row_b = (uint64_t)d * 2, slice_b = (uint64_t)rows * d * 2;
    {
        uint64_t dims[4], str[3];
        uint32_t box[4];
        int rk = 0;
        dims[rk] = fa > 0 ? 16 : (uint64_t)d;
        box[rk++] = 16;
        dims[rk] = (uint64_t)rows;
        box[rk++] = (uint32_t)box_rows;
        if (!table) {
            dims[rk] = (uint64_t)slices;
            box[rk++] = (uint32_t)box_slices;
        }
        dims[rk] = (uint64_t)(fa > 0 ? fa : 1);
        box[rk++] = (uint32_t)(atoms - part);
        int si = 0;
        str[si++] = row_b;
        if (!table) str[si++] = slice_b;
        str[si++] = 32;
        int rc = encode(full, base, bf16, rk, dims, str, box);
        if (rc) return rc;
    }
    if (part) {
        uint64_t dims[3], str[2];
        uint32_t box[3];
        int rk = 0;
        dims[rk] = (uint64_t)rem;
        box[rk++] = 16;
        dims[rk] = (uint64_t)rows;
        box[rk++] = (uint32_t)box_rows;
        if (!table) {
            dims[rk] = (uint64_t)slices;
            box[rk++] = (uint32_t)box_slices;
        }
        str[0] = row_b;
        str[1] = slice_b;
        const void* pb = static_cast<const unsigned char*>(base) + fa * 32;
        int rc = encode(partial, pb, bf16, rk, dims, str, box);
        if (rc) return rc;
    } else {
        *partial = *full;
    }
    return ATTN_OK;
}

// Magic number and shift for fast_div (unsigned division by an invariant d,
// Granlund and Montgomery 1994): l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1.
void fast_div_params(uint32_t d, uint32_t out[2]) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    out[0] = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << l) - d)) / d + 1);
    out[1] = l;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int dpad_for(int d) {
    const int r = (d + 15) / 16 * 16;
    if (r <= 32) return 32;
    if (r == 112) return 128;
    return r;
}

template <int DPAD>
cudaError_t dispatch_bias(int bias, const LaunchArgs& a) {
    switch (bias) {
        case kBiasNone: return launch_attn<DPAD, kBiasNone>(a);
        case kBiasSwin: return launch_attn<DPAD, kBiasSwin>(a);
        case kBiasSam: return launch_attn<DPAD, kBiasSam>(a);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t dispatch(int dpad, int bias, const LaunchArgs& a) {
    switch (dpad) {
        case 32: return dispatch_bias<32>(bias, a);
        case 48: return dispatch_bias<48>(bias, a);
        case 64: return dispatch_bias<64>(bias, a);
        case 80: return dispatch_bias<80>(bias, a);
        case 96: return dispatch_bias<96>(bias, a);
        case 128: return dispatch_bias<128>(bias, a);
        default: return cudaErrorInvalidValue;
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static int cache[64] = {0};
    if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// Dynamic shared memory left for the kernel's buffers after the 1 KB
// alignment pad and its static barriers.
constexpr size_t kSmemBudget = 227 * 1024 - 1024 - 1024;
// largest Swin bias-row area (per-head fp32 matrices + region bits)
constexpr size_t kSwinRowsMax = 96 * 1024;

// vt: a variable-length batch (no bias): B = 1, Nq / Nk = total query / key
// tokens of all sequences, the operands viewed as [H * total][d] rows.
// vp_sl: with vt, its sequences (each at most vp_sl query and key tokens)
// packed vp_sl rows per (sequence, head) slice; 0: shared tiling.
int run(const void* q, const void* k, const void* v, void* out, float* dbg, int B, int H, int Nq,
        int Nk, int d, float scale, attn_dtype dtype, attn_bias_kind bias_kind,
        const void* bias_args, void* stream, const VarlenTable* vt = nullptr, float* lse = nullptr,
        int vp_sl = 0) {
    g_last_error.clear();
    if (!q || !k || !v || !(out || dbg)) return fail(ATTN_ERR_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out ? out : (void*)dbg))
        return fail(ATTN_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return fail(ATTN_ERR_ARG, "B, H, Nq, Nk must be >= 1");
    if (d < 8 || d % 8 != 0) return fail(ATTN_ERR_ARG, "d must be a positive multiple of 8 (got %d)", d);
    if (d > 128) return fail(ATTN_ERR_UNSUPPORTED, "d > 128 is not supported (got %d)", d);
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return fail(ATTN_ERR_ARG, "unknown dtype %d", (int)dtype);
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return fail(ATTN_ERR_ARG, "scale must be finite");
    const int64_t BH = (int64_t)B * H;
    if (BH * Nq >= (int64_t(1) << 31) || BH * Nk >= (int64_t(1) << 31))
        return fail(ATTN_ERR_UNSUPPORTED, "B*H*N must stay below 2^31 rows");
    if (!vt && Nk > (1 << 20)) return fail(ATTN_ERR_UNSUPPORTED, "Nk > 2^20");
    const size_t q_bytes = (size_t)BH * Nq * d * 2, kv_bytes = (size_t)BH * Nk * d * 2;
    if (out && (overlaps(out, q_bytes, q, q_bytes) || overlaps(out, q_bytes, k, kv_bytes) ||
                overlaps(out, q_bytes, v, kv_bytes)))
        return fail(ATTN_ERR_ARG, "out must not alias q, k or v");

    AttnParams p;
    memset(&p, 0, sizeof(p));
    p.out = out;
    p.dbg = dbg;
    p.lse = lse;
    p.BH = (int)BH;
    p.H = H;
    p.Nq = Nq;
    p.Nk = Nk;
    p.d = d;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.is_bf16 = dtype == ATTN_BF16;
    p.q = q;
    p.k = k;
    p.v = v;
    const int dpad = dpad_for(d);
    const size_t tile_bytes = (size_t)(dpad / 16) * kBlockM * 32;
    size_t extra = 0;
    int bias = kBiasNone, sw_spec = 0;
    const void* rel_h = nullptr;
    const void* rel_w = nullptr;

    if (bias_kind == ATTN_BIAS_SWIN) {
        const attn_swin_args* a = static_cast<const attn_swin_args*>(bias_args);
        if (!a || !a->table) return fail(ATTN_ERR_ARG, "SWIN bias needs attn_swin_args with a table");
        const int M = a->win;
        if (M < 1 || M * M != Nq || Nk != Nq) return fail(ATTN_ERR_ARG, "SWIN needs Nq == Nk == win*win");
        if (M * M > kBlockM) return fail(ATTN_ERR_UNSUPPORTED, "SWIN windows above 128 tokens");
        if (a->grid_h < M || a->grid_w < M || a->grid_h % M || a->grid_w % M)
            return fail(ATTN_ERR_ARG, "grid_h and grid_w must be positive multiples of win");
        if (a->shift < 0 || a->shift >= M) return fail(ATTN_ERR_ARG, "shift must lie in [0, win)");
        if (a->layout != ATTN_SWIN_WINDOWS && a->layout != ATTN_SWIN_IMAGE)
            return fail(ATTN_ERR_ARG, "unknown Swin token layout %d", a->layout);
        const int nW = (a->grid_h / M) * (a->grid_w / M);
        if (B % nW) return fail(ATTN_ERR_ARG, "B (windows) must be a multiple of the windows per image");
        if (dpad > 64) return fail(ATTN_ERR_UNSUPPORTED, "SWIN with d > 64 is not supported");
        p.table = a->table;
        p.win = M;
        p.grid_h = a->grid_h;
        p.grid_w = a->grid_w;
        p.shift = a->shift;
        p.n_w = nW;
        p.n_ww = a->grid_w / M;
        p.n_wh = a->grid_h / M;
        fast_div_params((uint32_t)H, p.fd_h);
        fast_div_params((uint32_t)nW, p.fd_w);
        fast_div_params((uint32_t)p.n_ww, p.fd_ww);
        fast_div_params((uint32_t)M, p.fd_m);
        p.swin_image = a->layout == ATTN_SWIN_IMAGE ? 1 : 0;
        bias = kBiasSwin;
    } else if (bias_kind == ATTN_BIAS_SAM_RELPOS) {
        const attn_sam_args* a = static_cast<const attn_sam_args*>(bias_args);
        if (!a || !a->rel_h || !a->rel_w) return fail(ATTN_ERR_ARG, "SAM bias needs attn_sam_args with rel_h, rel_w");
        if (a->q_h < 1 || a->q_w < 1 || a->k_h < 1 || a->k_w < 1) return fail(ATTN_ERR_ARG, "SAM grid sizes must be >= 1");
        if (a->q_h * a->q_w != Nq || a->k_h * a->k_w != Nk)
            return fail(ATTN_ERR_ARG, "SAM needs Nq == q_h*q_w and Nk == k_h*k_w");
        if (a->q_h > kSamMaxSide || a->q_w > kSamMaxSide || a->k_h > kSamMaxSide || a->k_w > kSamMaxSide)
            return fail(ATTN_ERR_UNSUPPORTED, "SAM grid sides above %d", kSamMaxSide);
        // table lengths as given (0: 2*max(q, k)-1, the length the index addresses)
        const int lout_h = 2 * std::max(a->q_h, a->k_h) - 1, lout_w = 2 * std::max(a->q_w, a->k_w) - 1;
        const int lin_h = a->rel_h_len ? a->rel_h_len : lout_h, lin_w = a->rel_w_len ? a->rel_w_len : lout_w;
        if (lin_h < 1 || lin_w < 1) return fail(ATTN_ERR_ARG, "SAM table lengths must be >= 1");
        if (lin_h > kBlockN || lin_w > kBlockN)
            return fail(ATTN_ERR_UNSUPPORTED, "SAM tables longer than %d rows", kBlockN);
        if (!aligned16(a->rel_h) || !aligned16(a->rel_w)) return fail(ATTN_ERR_ARG, "rel_h/rel_w must be 16-byte aligned");
        rel_h = a->rel_h;
        rel_w = a->rel_w;
        p.s_h = a->q_h;
        p.s_w = a->q_w;
        p.k_h = a->k_h;
        p.k_w = a->k_w;
        p.sam_lin_h = lin_h;
        p.sam_lin_w = lin_w;
        p.sam_lout_h = lout_h;
        p.sam_lout_w = lout_w;
        p.rel_h = a->rel_h;
        p.rel_w = a->rel_w;
        // Unequal grids: rows through the coordinate scalers (float32, as the
        // published code computes them), resampled from G when the tables
        // have another length.  Equal grids with such tables: each CTA
        // resamples the tables once into shared memory (G then has the
        // addressed length and the row is a plain shift).
        p.sam_general = (a->q_h != a->k_h || a->q_w != a->k_w) ? 1 : 0;
        p.sam_resample = (!p.sam_general && (lin_h != lout_h || lin_w != lout_w)) ? 1 : 0;
        p.n_rh = ((p.sam_resample ? lout_h : lin_h) + 15) / 16 * 16;
        p.n_rw = ((p.sam_resample ? lout_w : lin_w) + 15) / 16 * 16;
        p.sam_qs_h = (float)std::max((double)a->k_h / a->q_h, 1.0);
        p.sam_ks_h = (float)std::max((double)a->q_h / a->k_h, 1.0);
        p.sam_off_h = (float)((a->k_h - 1) * std::max((double)a->q_h / a->k_h, 1.0));
        p.sam_qs_w = (float)std::max((double)a->k_w / a->q_w, 1.0);
        p.sam_ks_w = (float)std::max((double)a->q_w / a->k_w, 1.0);
        p.sam_off_w = (float)((a->k_w - 1) * std::max((double)a->q_w / a->k_w, 1.0));
        // square 14x14, 48x48 and 64x64 grids have specialised kernels (the
        // row of G that a query needs is then short and its shift has few
        // bits; key tiles start on grid rows), also with resampled tables
        const bool square = a->q_h == a->q_w && a->k_h == a->q_h && a->k_w == a->q_w;
        sw_spec = (square && (a->q_w == 64 || a->q_w == 48 || a->q_w == 14)) ? a->q_w : 0;
        extra = (size_t)sam_extra_floats(sw_spec == 0, a->k_h, a->k_w, Nk) * 4;
        if ((sw_spec == 64 || sw_spec == 48) && dpad <= 96) {
            // one grid row of keys per score tile, two score buffers per slot;
            // rel_h rows as fp16 [2 slots][64][128].  The tables pass through
            // two ring stages per job (64 rows per K or V tile), or, resampled,
            // are staged once per CTA.
            extra = kSamDbsExtra;
        }
        if (p.sam_resample) {
            // the resampled tables after the bias rows, 1 KB aligned (swizzled operands)
            extra = (extra + 1023) / 1024 * 1024;
            p.off_rtab = (uint32_t)extra;  // relative to the extra area until its offset is known
            extra += 2 * tile_bytes;
        }
        bias = kBiasSam;
    } else if (bias_kind != ATTN_BIAS_NONE) {
        return fail(ATTN_ERR_ARG, "unknown bias kind %d", (int)bias_kind);
    }

    // ---- job layout
    const int nmax = std::max(Nq, Nk);
    const int sl = vp_sl ? vp_sl : (nmax <= 32 ? 32 : (nmax <= 64 ? 64 : 128));
    const bool separate = vt ? (vp_sl != 0) : (bias == kBiasSwin || (bias == kBiasNone && sl <= 64 && dpad <= 64));
    if (vt && vp_sl && (bias != kBiasNone || dpad > 64 || (vp_sl != 32 && vp_sl != 64)))
        return fail(ATTN_ERR_UNSUPPORTED, "packed variable-length tiling: no bias, d <= 64, 32- or 64-row slices");
    int mode;
    if (separate) {
        mode = kModeSeparate;
        // 7x7 windows (49 tokens in 64-row slots) have a softmax specialised
        // for that key count
        if (bias == kBiasSwin && Nk == 49 && sl == 64) sw_spec = 49;
        p.g = kBlockM / sl;
        // packed variable-length batch: one slice per (sequence, head)
        if (vt) p.BH = H * vt->n_seq;
        const int64_t n_tiles = ((int64_t)p.BH + p.g - 1) / p.g;
        p.n_jobs = (int)((n_tiles + 1) / 2);
        p.n_kv = 1;
        p.kv_w = kBlockN;
        p.kv_cols = kBlockN;
        p.box_q = sl;
        p.box_kv = sl;
        p.nq = 0;
        p.ring_stage_bytes = (uint32_t)(3 * tile_bytes);
        if (bias == kBiasSwin) {
            // bias rows read by the softmax for windows up to 64 tokens when they
            // fit (and the table fits the first two ring stages, where it is
            // staged), else bias MMAs
            const size_t rows = swin_rows_extra_bytes(sl, H);
            const size_t table = (size_t)(2 * p.win - 1) * (2 * p.win - 1) * H * 4;
            p.swin_rows = (sl <= 64 && rows <= kSwinRowsMax && table <= 2 * (size_t)p.ring_stage_bytes) ? 1 : 0;
            extra = p.swin_rows ? rows : swin_extra_bytes(sl, H);
            // The bias-MMA variant holds table / scale and -100 / scale as
            // 16-bit MMA operands: a zero scale, or one so small that the
            // mask term leaves the operand type's range, cannot be
            // represented there.
            const double max16 = p.is_bf16 ? 3.3e38 : 65504.0;
            if (!p.swin_rows && (scale == 0.0f || 100.0 / std::fabs((double)scale) > max16))
                return fail(ATTN_ERR_UNSUPPORTED,
                            "SWIN windows of this size fold the bias into 16-bit MMA operands as bias / scale; "
                            "|scale| must be at least %g here (got %g)", 100.0 / max16, (double)scale);
        }
        const size_t avail = kSmemBudget > extra ? kSmemBudget - extra : 0;
        p.nst = (int)std::min<size_t>(kMaxStages, avail / p.ring_stage_bytes);
        if (p.nst < 2) return fail(ATTN_ERR_UNSUPPORTED, "shared memory too small for the packed tiling (H=%d)", H);
        p.off_q = 0;
        p.off_ring = 0;
        p.off_extra = (uint32_t)(p.nst * p.ring_stage_bytes);
    } else {
        mode = kModeShared;
        p.g = 1;
        // no bias and every key in one tile of at most 80 (e.g. 77 text tokens):
        // 80-column score tiles, P.V over 80 keys
        if (!vt && bias == kBiasNone && Nk <= 80 && dpad <= 64) sw_spec = 80;
        // with head dims up to 48 that kernel pipelines its jobs (two O buffers
        // per slot in tensor memory) and stages each slot's 128 output rows in
        // an area of its own
        if (sw_spec == 80 && 2 * 80 + 128 + 4 * dpad <= 512 && !dbg) extra = 2 * (size_t)kBlockM * d * 2;
        // SAM key tiles start on grid rows: 112 keys (8 rows) on the 14-wide
        // grid, 128 (2 rows) on the 64-wide one
        // (head dims up to 96: O and P then share 128 tensor-memory columns)
        const bool tiles64 = bias == kBiasSam && (sw_spec == 64 || sw_spec == 48) && dpad <= 96;
        p.kv_w = tiles64 ? sw_spec : (bias == kBiasSam && sw_spec) ? (sw_spec == 14 ? 112 : (kBlockN / sw_spec) * sw_spec)
                                                                   : kBlockN;
        p.kv_cols = kBlockN;  // unused by the kernel: its key-tile width is a compile-time constant
        p.n_kv = (Nk + p.kv_w - 1) / p.kv_w;
        p.q_jobs = (Nq + 2 * kBlockM - 1) / (2 * kBlockM);
        // a variable-length batch has H * ceil(Lq_s / 256) jobs per sequence
        const int64_t nj = vt ? (int64_t)vt->jobs_end[vt->n_seq - 1] : BH * p.q_jobs;
        if (nj > 0x7fffffff) return fail(ATTN_ERR_UNSUPPORTED, "too many jobs");
        p.n_jobs = (int)nj;
        p.box_q = kBlockM;
        // K/V tiles of one grid row for SAM on the 64 x 64 and 48 x 48 grids, else 128
        p.box_kv = tiles64 ? sw_spec : kBlockN;
        p.ring_stage_bytes = (uint32_t)(2 * (size_t)(dpad / 16) * p.box_kv * 32);
        // prefer >= 3 K/V stages, then double-buffered Q (the 64-key tiles
        // of the 64 x 64 SAM grid want >= 5: their scores run two tiles ahead)
        int nq = 0, nst = 0;
        const int tries[6][2] = {{2, tiles64 ? 5 : 3}, {1, tiles64 ? 5 : 3}, {2, 3}, {1, 3}, {2, 2}, {1, 2}};
        for (auto& t : tries) {
            const size_t fixed = 2 * (size_t)t[0] * tile_bytes + extra;
            if (fixed >= kSmemBudget) continue;
            const int s = (int)std::min<size_t>(kMaxStages, (kSmemBudget - fixed) / p.ring_stage_bytes);
            if (s >= t[1]) {
                nq = t[0];
                nst = s;
                break;
            }
        }
        if (!nst) return fail(ATTN_ERR_UNSUPPORTED, "shared memory too small for d=%d with this bias", d);
        p.nq = nq;
        p.nst = nst;
        p.off_q = 0;
        p.off_ring = (uint32_t)(2 * nq * tile_bytes);
        p.off_extra = (uint32_t)(p.off_ring + nst * p.ring_stage_bytes);
        if (p.sam_resample) p.off_rtab += p.off_extra;
    }
    const size_t smem = p.off_extra + extra + 1024;
    const int nsm = sm_count();
    if (nsm <= 0) return fail(ATTN_ERR_CUDA, "no CUDA device");
    const int grid = std::min(p.n_jobs, nsm);

    TmaMaps tm;
    const bool bf = p.is_bf16 != 0;
    const int atoms = dpad / 16;
    p.full_atoms = d / 16;
    p.part = (d / 16 > 0 && d % 16) ? 1 : 0;
    int rc;
    if (separate) {
        if ((rc = encode_operand(&tm.q, &tm.qp, q, bf, d, Nq, BH, atoms, sl, p.g))) return rc;
        if ((rc = encode_operand(&tm.k, &tm.kp, k, bf, d, Nk, BH, atoms, sl, p.g))) return rc;
        if ((rc = encode_operand(&tm.v, &tm.vp, v, bf, d, Nk, BH, atoms, sl, p.g))) return rc;
    } else if (vt) {
        // one slice of H * total rows: a job addresses its sequence's rows
        if ((rc = encode_operand(&tm.q, &tm.qp, q, bf, d, BH * Nq, 1, atoms, kBlockM, 1))) return rc;
        if ((rc = encode_operand(&tm.k, &tm.kp, k, bf, d, BH * Nk, 1, atoms, kBlockN, 1))) return rc;
        if ((rc = encode_operand(&tm.v, &tm.vp, v, bf, d, BH * Nk, 1, atoms, kBlockN, 1))) return rc;
    } else {
        if ((rc = encode_operand(&tm.q, &tm.qp, q, bf, d, Nq, BH, atoms, kBlockM, 1))) return rc;
        if ((rc = encode_operand(&tm.k, &tm.kp, k, bf, d, Nk, BH, atoms, p.box_kv, 1))) return rc;
        if ((rc = encode_operand(&tm.v, &tm.vp, v, bf, d, Nk, BH, atoms, p.box_kv, 1))) return rc;
    }
    if (bias == kBiasSam) {
        // table copies land in K/V ring tiles: box_kv rows at a time
        const int tb = separate ? kBlockN : p.box_kv;
        if ((rc = encode_operand(&tm.rh, &tm.rhp, rel_h, bf, d, p.sam_lin_h, 0, atoms, tb, 1))) return rc;
        if ((rc = encode_operand(&tm.rw, &tm.rwp, rel_w, bf, d, p.sam_lin_w, 0, atoms, tb, 1))) return rc;
    } else {
        tm.rh = tm.rhp = tm.rw = tm.rwp = tm.q;
    }
    p.status = status_ptr();
    if (!p.status) return fail(ATTN_ERR_CUDA, "no CUDA device / status word unavailable");

    LaunchArgs la;
    la.tm = &tm;
    la.p = &p;
    la.mode = mode;
    la.sw = sw_spec;
    la.sl = sl;
    la.dbg = dbg != nullptr;
    la.grid = grid;
    la.smem = smem;
    la.stream = static_cast<cudaStream_t>(stream);
    la.vt = vt;
    cudaError_t e = dispatch(dpad, bias, la);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    static const bool debug_env = getenv("SDPA09_DEBUG") && getenv("SDPA09_DEBUG")[0] == '1';
    if (debug_env) return attn_device_status(stream);
    return ATTN_OK;
}

// ------------------------------------------------------------------ backward

// Workspace of the backward pass for sequences longer than one 128-key tile
// (none is needed for windows of up to 128 tokens).
// Layout of the long-sequence backward's workspace (byte offsets, each
// 256-byte aligned): D [rows] fp32; for SAM also the rel terms [rows][stride]
// fp16, scale dS.K [rows][d] fp32, dRelH [rows][k_h] fp32 and dRelW
// [2][rows][k_w] fp32, one array per column half (rows = B * H * Nq); with
// tables of another length than 2 S - 1 rows also their resampled 16-bit
// copies [2][2S-1][d] and the fp32 gradients of those [2][2S-1][d].
struct BwdWs {
    size_t d, rel, dq32, drh, drw, rtab, drr, total;
};
static size_t al256(size_t x) { return (x + 255) / 256 * 256; }
static BwdWs bwd_ws_layout(int64_t rows, int d, bool sam, int s_h, int s_w, int rel_stride, bool resample) {
    BwdWs w{};
    size_t o = 0;
    w.d = o;
    o += al256((size_t)rows * 4);
    if (sam) {
        w.rel = o;
        o += al256((size_t)rows * rel_stride * 2);
        w.dq32 = o;
        o += al256((size_t)rows * d * 4);
        w.drh = o;
        o += al256((size_t)rows * s_h * 4);
        w.drw = o;
        o += al256((size_t)2 * rows * s_w * 4);
        if (resample) {
            const size_t nt = (size_t)(2 * s_w - 1);
            w.rtab = o;
            o += al256(2 * nt * d * 2);
            w.drr = o;
            o += al256(2 * nt * d * 4);
        }
    }
    w.total = o;
    return w;
}
// table lengths of a SAM bias as given (0: 2 * side - 1) and whether the
// backward resamples them
static bool sam_bwd_resample(const attn_sam_args* a, int* lh, int* lw) {
    *lh = a->rel_h_len ? a->rel_h_len : 2 * a->q_h - 1;
    *lw = a->rel_w_len ? a->rel_w_len : 2 * a->q_w - 1;
    return *lh != 2 * a->q_h - 1 || *lw != 2 * a->q_w - 1;
}
static bool bwd_is_windows(int Nq, int Nk, int d) { return Nq <= kBlockM && Nk <= kBlockN && dpad_for(d) <= 64; }
static int sam_rel_stride(int s_h, int s_w, int* rw0) {
    *rw0 = (s_h + 7) / 8 * 8;
    return *rw0 + (s_w + 7) / 8 * 8;
}

size_t bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d, attn_bias_kind bias_kind, const void* bias_args) {
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return 0;
    if (bias_kind != ATTN_BIAS_SAM_RELPOS && bwd_is_windows(Nq, Nk, d)) return 0;
    const int64_t rows = (int64_t)B * H * Nq;
    bool sam = false, resample = false;
    int s_h = 0, s_w = 0, stride = 0, rw0 = 0;
    if (bias_kind == ATTN_BIAS_SAM_RELPOS && bias_args) {
        const attn_sam_args* a = static_cast<const attn_sam_args*>(bias_args);
        sam = true;
        s_h = a->q_h;
        s_w = a->q_w;
        stride = sam_rel_stride(s_h, s_w, &rw0);
        int lh = 0, lw = 0;
        resample = sam_bwd_resample(a, &lh, &lw);
    }
    return bwd_ws_layout(rows, d, sam, s_h, s_w, stride, resample).total;
}

// Sequences longer than one 128-key tile (or d > 64): pre-pass for D, then
// the key pass (dK, dV) and the query pass (dQ) on the tensor cores.
int run_bwd_long(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, attn_dtype dtype,
                 const attn_sam_args* sam, float* d_bias, void* workspace, size_t workspace_bytes, void* stream) {
    const int dpad = dpad_for(d);
    if (dpad > 80) return fail(ATTN_ERR_UNSUPPORTED, "backward for sequences over 128 tokens needs d <= 80");
    if (!lse)
        return fail(ATTN_ERR_ARG, "sequences over 128 tokens (or d > 64) need the forward's lse (attn_fwd_train)");
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return fail(ATTN_ERR_ARG, "lse must be 4-byte aligned");
    const int64_t BH = (int64_t)B * H, rows = BH * Nq;
    int rw0 = 0, stride = 0, lin_h = 0, lin_w = 0;
    bool resample = false;
    if (sam) {
        stride = sam_rel_stride(sam->q_h, sam->q_w, &rw0);
        resample = sam_bwd_resample(sam, &lin_h, &lin_w);
    }
    const BwdWs ws = bwd_ws_layout(rows, d, sam != nullptr, sam ? sam->q_h : 0, sam ? sam->q_w : 0, stride, resample);
    if (!workspace || workspace_bytes < ws.total)
        return fail(ATTN_ERR_ARG, "workspace of %zu bytes needed (attn_bwd_workspace_size), %zu given", ws.total,
                    workspace_bytes);
    if (!aligned16(workspace)) return fail(ATTN_ERR_ARG, "workspace must be 16-byte aligned");
    unsigned char* wsb = static_cast<unsigned char*>(workspace);
    const int nsm = sm_count();
    if (nsm <= 0) return fail(ATTN_ERR_CUDA, "no CUDA device");
    int* status = status_ptr();
    if (!status) return fail(ATTN_ERR_CUDA, "no CUDA device / status word unavailable");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = dtype == ATTN_BF16;

    BwdPrepParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.o = out;
    pp.dout = dout;
    pp.Dws = reinterpret_cast<float*>(wsb + ws.d);
    pp.rows = (int)rows;
    pp.d = d;
    pp.is_bf16 = bf;
    cudaError_t e = launch_bwd_prep(pp, nsm, st);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    const int sw = sam ? sam->q_w : 0;
    SamBwdParams sp;
    memset(&sp, 0, sizeof(sp));
    if (sam) {
        sp.q = q;
        sp.rel_h = sam->rel_h;
        sp.rel_w = sam->rel_w;
        sp.rel = reinterpret_cast<__half*>(wsb + ws.rel);
        sp.dq32 = reinterpret_cast<float*>(wsb + ws.dq32);
        sp.d_relh = reinterpret_cast<float*>(wsb + ws.drh);
        sp.d_relw = reinterpret_cast<float*>(wsb + ws.drw);
        sp.dq = dq;
        sp.d_bias = d_bias;
        sp.BH = (int)BH;
        sp.Nq = Nq;
        sp.d = d;
        sp.rel_stride = stride;
        sp.rw0 = rw0;
        sp.groups = sam_bwd_groups(sw, (int)BH, nsm);
        sp.status = status;
        if (resample) {
            // the tables resampled to 2 S - 1 rows as the forward does; the post
            // passes add the gradients of those rows to a cleared area, which
            // the transposed resampling returns to d_bias at the end
            const int nt = 2 * sw - 1;
            uint16_t* rt = reinterpret_cast<uint16_t*>(wsb + ws.rtab);
            float* drr = reinterpret_cast<float*>(wsb + ws.drr);
            e = launch_bwd_sam_resample(sam->rel_h, rt, lin_h, nt, d, bf, drr, 2 * nt * d, st);
            if (e == cudaSuccess) e = launch_bwd_sam_resample(sam->rel_w, rt + (size_t)nt * d, lin_w, nt, d, bf, nullptr, 0, st);
            if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
            sp.rel_h = rt;
            sp.rel_w = rt + (size_t)nt * d;
            sp.d_bias = drr;
        }
        e = launch_bwd_sam_rel_tc(sp, sw, bf, nsm, st);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    }

    BwdLongParams p;
    memset(&p, 0, sizeof(p));
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.lse = lse;
    p.Dws = pp.Dws;
    p.status = status;
    p.BH = (int)BH;
    p.Nq = Nq;
    p.Nk = Nk;
    p.d = d;
    // key tiles start on grid rows: 112 keys (8 rows) on the 14-wide grid, 96
    // (2 rows) on the 48-wide one
    p.kv_w = sw == 14 ? 112 : (sw == 48 ? 96 : kBlockN);
    if (sam) {
        p.rel = sp.rel;
        p.rel_stride = stride;
        p.rw0 = rw0;
        p.k_h = sam->k_h;
        p.k_w = sam->k_w;
        p.dq32 = const_cast<float*>(sp.dq32);
        p.d_relh = sp.d_relh;
        p.d_relw = const_cast<float*>(sp.d_relw);
    }
    p.n_qb = (Nq + kBlockM - 1) / kBlockM;
    p.n_kb = (Nk + p.kv_w - 1) / p.kv_w;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.is_bf16 = bf;
    p.full_atoms = d / 16;
    p.part = (d / 16 > 0 && d % 16) ? 1 : 0;
    const size_t tile = (size_t)(dpad / 16) * kBlockM * 32;
    p.stage_bytes = (uint32_t)(2 * tile);
    const int atoms = dpad / 16;
    BwdMaps tm;
    int rc;
    if ((rc = encode_operand(&tm.q, &tm.qp, q, bf, d, Nq, BH, atoms, kBlockM, 1))) return rc;
    if ((rc = encode_operand(&tm.k, &tm.kp, k, bf, d, Nk, BH, atoms, kBlockN, 1))) return rc;
    if ((rc = encode_operand(&tm.v, &tm.vp, v, bf, d, Nk, BH, atoms, kBlockN, 1))) return rc;
    if ((rc = encode_operand(&tm.dout, &tm.dop, dout, bf, d, Nq, BH, atoms, kBlockM, 1))) return rc;
    for (int mode = 0; mode < 2; ++mode) {
        const size_t pds = mode == kBwdKeyPass ? 2 * (size_t)8 * kBlockM * 32 : (size_t)8 * kBlockM * 32;
        const size_t fixed = 2 * tile + pds;
        if (fixed + 2 * p.stage_bytes > kSmemBudget) return fail(ATTN_ERR_UNSUPPORTED, "shared memory too small (d=%d)", d);
        p.nst = (int)std::min<size_t>(kMaxStages, (kSmemBudget - fixed) / p.stage_bytes);
        p.off_res = 0;
        p.off_ring = (uint32_t)(2 * tile);
        p.off_p = p.off_ring + (uint32_t)(p.nst * p.stage_bytes);
        p.off_ds = p.off_p + (mode == kBwdKeyPass ? (uint32_t)(8 * kBlockM * 32) : 0u);
        const size_t smem = p.off_ds + (size_t)8 * kBlockM * 32 + 1024;
        p.n_jobs = (int)(BH * (mode == kBwdKeyPass ? p.n_kb : p.n_qb));
        const int grid = std::min(p.n_jobs, nsm);
        e = launch_bwd_long(dpad, mode, sw, tm, p, grid, smem, st);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    }
    if (sam) {
        e = launch_bwd_sam_post(sp, sw, bf, nsm, st);
        if (e == cudaSuccess && resample) {
            const int nt = 2 * sw - 1;
            e = launch_bwd_sam_unresample(sp.d_bias, d_bias, lin_h, nt, d, st);
            if (e == cudaSuccess)
                e = launch_bwd_sam_unresample(sp.d_bias + (size_t)nt * d, d_bias + (size_t)lin_h * d, lin_w, nt, d, st);
        }
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    }
    static const bool debug_env = getenv("SDPA09_DEBUG") && getenv("SDPA09_DEBUG")[0] == '1';
    if (debug_env) return attn_device_status(stream);
    return ATTN_OK;
}

int run_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, attn_dtype dtype,
            attn_bias_kind bias_kind, const void* bias_args, float* d_bias, void* workspace, size_t workspace_bytes,
            void* stream) {
    g_last_error.clear();
    (void)lse; (void)workspace; (void)workspace_bytes;
    const void* ptrs[8] = {q, k, v, out, dout, dq, dk, dv};
    for (const void* x : ptrs) {
        if (!x) return fail(ATTN_ERR_ARG, "null tensor pointer");
        if (!aligned16(x)) return fail(ATTN_ERR_ARG, "tensor pointers must be 16-byte aligned");
    }
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return fail(ATTN_ERR_ARG, "B, H, Nq, Nk must be >= 1");
    if (d < 8 || d % 8 != 0) return fail(ATTN_ERR_ARG, "d must be a positive multiple of 8 (got %d)", d);
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return fail(ATTN_ERR_ARG, "unknown dtype %d", (int)dtype);
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return fail(ATTN_ERR_ARG, "scale must be finite");
    const int64_t BH = (int64_t)B * H;
    if (BH * Nq >= (int64_t(1) << 31) || BH * Nk >= (int64_t(1) << 31))
        return fail(ATTN_ERR_UNSUPPORTED, "B*H*N must stay below 2^31 rows");
    const int dpad = dpad_for(d);
    BwdTcParams p;
    memset(&p, 0, sizeof(p));
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.o = out;
    p.BH = (int)BH;
    p.H = H;
    p.Nq = Nq;
    p.Nk = Nk;
    p.d = d;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.is_bf16 = dtype == ATTN_BF16;
    bool swin = false;
    if (bias_kind == ATTN_BIAS_SWIN) {
        const attn_swin_args* a = static_cast<const attn_swin_args*>(bias_args);
        if (!a || !a->table) return fail(ATTN_ERR_ARG, "SWIN bias needs attn_swin_args with a table");
        if (!d_bias) return fail(ATTN_ERR_ARG, "SWIN backward needs d_bias (the table gradient)");
        const int M = a->win;
        if (M < 1 || Nq != M * M || Nk != M * M) return fail(ATTN_ERR_ARG, "SWIN needs Nq == Nk == win*win");
        if (a->grid_h < M || a->grid_w < M || a->grid_h % M || a->grid_w % M)
            return fail(ATTN_ERR_ARG, "grid_h and grid_w must be positive multiples of win");
        if (a->shift < 0 || a->shift >= M) return fail(ATTN_ERR_ARG, "shift must lie in [0, win)");
        if (a->layout != ATTN_SWIN_WINDOWS && a->layout != ATTN_SWIN_IMAGE)
            return fail(ATTN_ERR_ARG, "unknown Swin token layout %d", (int)a->layout);
        const int nW = (a->grid_h / M) * (a->grid_w / M);
        if (B % nW) return fail(ATTN_ERR_ARG, "B (windows) must be a multiple of the windows per image");
        swin = true;
        if (a->layout == ATTN_SWIN_IMAGE) {
            // the kernel gathers the windows' rows and scatters the gradients
            p.swin_image = 1;
            fast_div_params((uint32_t)M, p.fd_m);
            p.q = q;
            p.k = k;
            p.v = v;
            p.dout = dout;
        }
        p.table = a->table;
        p.d_table = d_bias;
        p.win = M;
        p.grid_h = a->grid_h;
        p.grid_w = a->grid_w;
        p.shift = a->shift;
        p.n_w = nW;
        p.n_ww = a->grid_w / M;
        p.n_wh = a->grid_h / M;
        fast_div_params((uint32_t)H, p.fd_h);
        fast_div_params((uint32_t)nW, p.fd_w);
        fast_div_params((uint32_t)p.n_ww, p.fd_ww);
    } else if (bias_kind == ATTN_BIAS_SAM_RELPOS) {
        const attn_sam_args* a = static_cast<const attn_sam_args*>(bias_args);
        if (!a || !a->rel_h || !a->rel_w) return fail(ATTN_ERR_ARG, "SAM bias needs attn_sam_args with rel_h, rel_w");
        if (!d_bias) return fail(ATTN_ERR_ARG, "SAM backward needs d_bias (the rel_h and rel_w gradients)");
        if (a->q_h * a->q_w != Nq || a->k_h * a->k_w != Nk)
            return fail(ATTN_ERR_ARG, "SAM needs Nq == q_h*q_w and Nk == k_h*k_w");
        const int S = a->q_w;
        int lh = 0, lw = 0;
        sam_bwd_resample(a, &lh, &lw);
        if (a->q_h != S || a->k_h != S || a->k_w != S || (S != 14 && S != 48 && S != 64))
            return fail(ATTN_ERR_UNSUPPORTED, "the SAM backward takes square 14 x 14, 48 x 48 or 64 x 64 grids");
        if (lh < 1 || lw < 1 || lh > kBlockN || lw > kBlockN)
            return fail(ATTN_ERR_UNSUPPORTED, "SAM tables of 1 to %d rows", kBlockN);
        if (dpad != 64 && dpad != 80) return fail(ATTN_ERR_UNSUPPORTED, "the SAM backward takes 48 < d <= 80");
        if (!aligned16(a->rel_h) || !aligned16(a->rel_w)) return fail(ATTN_ERR_ARG, "rel_h/rel_w must be 16-byte aligned");
        if ((reinterpret_cast<uintptr_t>(d_bias) & 3u) != 0) return fail(ATTN_ERR_ARG, "d_bias must be 4-byte aligned");
        return run_bwd_long(q, k, v, out, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, dtype, a, d_bias, workspace,
                            workspace_bytes, stream);
    } else if (bias_kind != ATTN_BIAS_NONE) {
        return fail(ATTN_ERR_ARG, "unknown bias kind %d", (int)bias_kind);
    }
    if (!bwd_is_windows(Nq, Nk, d)) {
        if (swin) return fail(ATTN_ERR_UNSUPPORTED, "SWIN backward with d > 64");
        return run_bwd_long(q, k, v, out, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, dtype, nullptr, nullptr,
                            workspace, workspace_bytes, stream);
    }
    // packed windows: g slices of up to SL tokens share a 128-row tile
    const int nmax = std::max(Nq, Nk);
    const int sl = nmax <= 32 ? 32 : (nmax <= 64 ? 64 : 128);
    p.sl = sl;
    p.g = kBlockM / sl;
    p.n_jobs = (int)((BH + p.g - 1) / p.g);
    const size_t tile_bytes = (size_t)(dpad / 16) * kBlockM * 32;
    p.stage_bytes = (uint32_t)(4 * tile_bytes);
    const size_t pds = 2 * (size_t)8 * kBlockM * 32;
    size_t extra = swin ? (2 * (size_t)(2 * p.win - 1) * (2 * p.win - 1) * H * 4 + 1023) / 1024 * 1024 : 0;
    if (pds + extra + 2 * p.stage_bytes > kSmemBudget)
        return fail(ATTN_ERR_UNSUPPORTED, "shared memory too small for this backward (H=%d)", H);
    // Swin: the table gradient sums dS per (head, key token, query token) in
    // shared memory when that fits (else one shared-memory atomic per pair,
    // by relative offset), and per-CTA fp16 bias rows are used when they fit
    // next to >= 3 stages (2 for the widest tiles), else per-element gathers
    // from the table
    if (swin) {
        const size_t acc = ((size_t)H * Nq * Nk * 4 + 1023) / 1024 * 1024;
        const int want = p.stage_bytes > 40 * 1024 ? 2 : 3;
        p.swin_acc = (pds + extra + acc + 2 * (size_t)p.stage_bytes <= kSmemBudget) ? 1 : 0;
        p.swin_acc_atomic = p.g > H ? 1 : 0;
        p.off_acc = (uint32_t)extra;  // relative to the extra area until its offset is known
        if (p.swin_acc) extra += acc;
        const size_t rows = ((size_t)H * sl * sl * 2 + 3 * (size_t)sl * (sl / 32) * 4 + 1023) / 1024 * 1024;
        p.swin_rows = (sl <= 64 && pds + extra + rows + want * (size_t)p.stage_bytes <= kSmemBudget) ? 1 : 0;
        p.off_rows = (uint32_t)extra;
        if (p.swin_rows) extra += rows;
    }
    p.nst = (int)std::min<size_t>(kMaxStages, (kSmemBudget - pds - extra) / p.stage_bytes);
    p.off_ring = 0;
    p.off_p = (uint32_t)(p.nst * p.stage_bytes);
    p.off_ds = p.off_p + (uint32_t)(pds / 2);
    p.off_extra = p.off_ds + (uint32_t)(pds / 2);
    p.off_rows += p.off_extra;
    p.off_acc += p.off_extra;
    const size_t smem = p.off_extra + extra + 1024;
    p.full_atoms = d / 16;
    p.part = (d / 16 > 0 && d % 16) ? 1 : 0;
    const int atoms = dpad / 16;
    const bool bf = p.is_bf16 != 0;
    BwdMaps tm;
    int rc;
    if ((rc = encode_operand(&tm.q, &tm.qp, q, bf, d, Nq, BH, atoms, sl, p.g))) return rc;
    if ((rc = encode_operand(&tm.k, &tm.kp, k, bf, d, Nk, BH, atoms, sl, p.g))) return rc;
    if ((rc = encode_operand(&tm.v, &tm.vp, v, bf, d, Nk, BH, atoms, sl, p.g))) return rc;
    if ((rc = encode_operand(&tm.dout, &tm.dop, dout, bf, d, Nq, BH, atoms, sl, p.g))) return rc;
    const int nsm = sm_count();
    if (nsm <= 0) return fail(ATTN_ERR_CUDA, "no CUDA device");
    p.status = status_ptr();
    if (!p.status) return fail(ATTN_ERR_CUDA, "no CUDA device / status word unavailable");
    const int grid = std::min(p.n_jobs, nsm);
    cudaError_t e = launch_bwd_win(dpad, swin, tm, p, grid, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    static const bool debug_env = getenv("SDPA09_DEBUG") && getenv("SDPA09_DEBUG")[0] == '1';
    if (debug_env) return attn_device_status(stream);
    return ATTN_OK;
}

}  // namespace
}  // namespace sdpa09

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int H, int Nq, int Nk,
             int d, float scale, attn_dtype dtype, attn_bias_kind bias_kind, const void* bias_args,
             void* stream) {
    if (!out) return sdpa09::fail(ATTN_ERR_ARG, "null output pointer");
    return sdpa09::run(q, k, v, out, nullptr, B, H, Nq, Nk, d, scale, dtype, bias_kind, bias_args,
                       stream);
}

int attn_fwd_train(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H, int Nq,
                   int Nk, int d, float scale, attn_dtype dtype, attn_bias_kind bias_kind, const void* bias_args,
                   void* stream) {
    if (!out) return sdpa09::fail(ATTN_ERR_ARG, "null output pointer");
    if (!lse) return sdpa09::fail(ATTN_ERR_ARG, "null lse pointer");
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return sdpa09::fail(ATTN_ERR_ARG, "lse must be 4-byte aligned");
    return sdpa09::run(q, k, v, out, nullptr, B, H, Nq, Nk, d, scale, dtype, bias_kind, bias_args, stream, nullptr,
                       lse);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* out, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int n_seq, int H, int d, float scale, attn_dtype dtype,
                    void* stream) {
    using sdpa09::fail;
    static_assert(ATTN_VARLEN_MAX_SEQ == sdpa09::kVarlenMaxSeq, "header and kernel table sizes");
    sdpa09::g_last_error.clear();
    if (!cu_seqlens_q || !cu_seqlens_k) return fail(ATTN_ERR_ARG, "null cu_seqlens pointer");
    if (n_seq < 1) return fail(ATTN_ERR_ARG, "n_seq must be >= 1");
    if (n_seq > sdpa09::kVarlenMaxSeq)
        return fail(ATTN_ERR_UNSUPPORTED, "more than %d sequences", sdpa09::kVarlenMaxSeq);
    if (H < 1) return fail(ATTN_ERR_ARG, "H must be >= 1");
    if (cu_seqlens_q[0] != 0 || cu_seqlens_k[0] != 0) return fail(ATTN_ERR_ARG, "cu_seqlens must start at 0");
    // Sequences of at most 32 (64) query and key tokens, with d <= 64, are
    // packed four (two) (sequence, head) slices per 128-row tile; the others
    // take the shared tiling, longest key range first (the CTAs take jobs
    // round-robin, and this order evens out their totals).
    int order[sdpa09::kVarlenMaxSeq];
    int n_q = 0;  // sequences with queries in the shared tiling
    sdpa09::VarlenTable packed[2];  // slices of 32 and of 64 rows
    memset(packed, 0, sizeof(packed));
    for (int s = 0; s < n_seq; ++s) {
        const int lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s], lk = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
        if (lq < 0 || lk < 0) return fail(ATTN_ERR_ARG, "cu_seqlens must be nondecreasing (sequence %d)", s);
        if (lq > 0 && lk == 0) return fail(ATTN_ERR_ARG, "sequence %d has queries but no keys", s);
        if (lk > (1 << 20)) return fail(ATTN_ERR_UNSUPPORTED, "sequence %d has more than 2^20 keys", s);
        if (lq == 0) continue;
        const int n = std::max(lq, lk);
        if (d <= 64 && n <= 64) {
            sdpa09::VarlenTable& t = packed[n <= 32 ? 0 : 1];
            t.q_off[t.n_seq] = cu_seqlens_q[s];
            t.q_len[t.n_seq] = lq;
            t.k_off[t.n_seq] = cu_seqlens_k[s];
            t.k_len[t.n_seq] = lk;
            ++t.n_seq;
        } else {
            order[n_q++] = s;
        }
    }
    std::stable_sort(order, order + n_q, [&](int a, int b) {
        return cu_seqlens_k[a + 1] - cu_seqlens_k[a] > cu_seqlens_k[b + 1] - cu_seqlens_k[b];
    });
    sdpa09::VarlenTable vt;
    memset(&vt, 0, sizeof(vt));
    vt.n_seq = n_q;
    int64_t jobs = 0;
    for (int e = 0; e < n_q; ++e) {
        const int s = order[e];
        vt.q_off[e] = cu_seqlens_q[s];
        vt.q_len[e] = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        vt.k_off[e] = cu_seqlens_k[s];
        vt.k_len[e] = cu_seqlens_k[s + 1] - cu_seqlens_k[s];
        jobs += (int64_t)H * ((vt.q_len[e] + 2 * sdpa09::kBlockM - 1) / (2 * sdpa09::kBlockM));
        if (jobs > 0x7fffffff) return fail(ATTN_ERR_UNSUPPORTED, "too many jobs");
        vt.jobs_end[e] = (int)jobs;
    }
    const int tq = cu_seqlens_q[n_seq], tk = cu_seqlens_k[n_seq];
    int rc = ATTN_OK;
    if (jobs > 0)
        rc = sdpa09::run(q, k, v, out, nullptr, 1, H, tq, tk, d, scale, dtype, ATTN_BIAS_NONE, nullptr, stream, &vt);
    for (int i = 0; i < 2 && rc == ATTN_OK; ++i)
        if (packed[i].n_seq > 0)
            rc = sdpa09::run(q, k, v, out, nullptr, 1, H, tq, tk, d, scale, dtype, ATTN_BIAS_NONE, nullptr, stream,
                             &packed[i], nullptr, i == 0 ? 32 : 64);
    return rc;  // (no sequence with a query: nothing to do, the tensors may be empty)
}

size_t attn_bwd_workspace_size(int B, int H, int Nq, int Nk, int d, attn_bias_kind bias_kind, const void* bias_args) {
    return sdpa09::bwd_workspace_bytes(B, H, Nq, Nk, d, bias_kind, bias_args);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, attn_dtype dtype,
             attn_bias_kind bias_kind, const void* bias_args, float* d_bias, void* workspace, size_t workspace_bytes,
             void* stream) {
    return sdpa09::run_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, dtype, bias_kind, bias_args,
                           d_bias, workspace, workspace_bytes, stream);
}

int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale,
                     attn_dtype dtype, void* stream) {
    using sdpa09::fail;
    sdpa09::g_last_error.clear();
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return fail(ATTN_ERR_ARG, "B, H, Nq, Nk must be >= 1");
    const size_t need = sdpa09::bwd_workspace_bytes(B, H, Nq, Nk, d, ATTN_BIAS_NONE, nullptr);
    if ((int64_t)B * H * Nq > sdpa09::kNoAllocRows || need > sizeof(float) * (size_t)sdpa09::kNoAllocRows)
        return fail(ATTN_ERR_UNSUPPORTED,
                    "attn_bwd_noalloc holds scratch for at most %d query rows (B*H*Nq = %lld); use attn_bwd with a "
                    "workspace", sdpa09::kNoAllocRows, (long long)B * H * Nq);
    float* scratch = nullptr;
    if (need > 0) {
        scratch = sdpa09::noalloc_scratch_ptr();
        if (!scratch) return fail(ATTN_ERR_CUDA, "no CUDA device / scratch address unavailable");
    }
    return sdpa09::run_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, dtype, ATTN_BIAS_NONE,
                           nullptr, nullptr, scratch, need, stream);
}

int attn_debug_bias(const void* q, const void* k, const void* v, float* bias_out, int B, int H,
                    int Nq, int Nk, int d, float scale, attn_dtype dtype, attn_bias_kind bias_kind,
                    const void* bias_args, void* stream) {
    if (!bias_out) return sdpa09::fail(ATTN_ERR_ARG, "null bias_out pointer");
    return sdpa09::run(q, k, v, nullptr, bias_out, B, H, Nq, Nk, d, scale, dtype, bias_kind,
                       bias_args, stream);
}

int attn_device_status(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return sdpa09::fail(ATTN_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, sdpa09::g_status_word, sizeof(int));
    if (e != cudaSuccess) return sdpa09::fail(ATTN_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(sdpa09::g_status_word, &zero, sizeof(int));
        return sdpa09::fail(ATTN_ERR_DEVICE_TIMEOUT, "a kernel wait ran out of time (code %d)", v);
    }
    return ATTN_OK;
}

int attn_selftest_wait_timeout(unsigned limit_us, void* stream) {
    if (limit_us == 0 || limit_us > 2000000u)
        return sdpa09::fail(ATTN_ERR_ARG, "limit_us must lie in [1, 2000000] (got %u)", limit_us);
    int* status = sdpa09::status_ptr();
    if (!status) return sdpa09::fail(ATTN_ERR_CUDA, "no CUDA device / status word unavailable");
    sdpa09::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status,
                                                                                  (uint64_t)limit_us * 1000u);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return sdpa09::fail(ATTN_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

const char* attn_last_error(void) { return sdpa09::g_last_error.c_str(); }

int attn_abi_version(void) { return SDPA09_ABI_VERSION; }

}  // extern "C"
