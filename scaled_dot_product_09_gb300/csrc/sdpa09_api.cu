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

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <string>

#include "../../include/sdpa09.h"
#include "attn_launch.cuh"

namespace sdpa09 {
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

// Rank-2 or rank-3 tiled map over a [outer][rows][d] half tensor with a
// box of 16 elements x box_rows rows, 32-byte swizzle.
int encode_map(CUtensorMap* m, const void* base, bool bf16, int d, int64_t rows, int64_t outer,
               int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {16, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    const cuuint32_t rank = outer > 0 ? 3 : 2;
    CUresult r = enc(m, dt, rank, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ATTN_OK;
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

size_t tiles_bytes(int dpad) {
    const int stages = dpad <= 64 ? 4 : (dpad <= 96 ? 3 : 2);
    return (size_t)(dpad / 16) * kBlockM * 32 * (1 + 2 * stages);
}

cudaError_t dispatch(int dpad, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const AttnParams& p, int bias, bool dbg, int grid, size_t smem,
                     cudaStream_t st) {
    switch (dpad) {
        case 32: return launch_attn<32>(tq, tk, tv, p, bias, dbg, grid, smem, st);
        case 48: return launch_attn<48>(tq, tk, tv, p, bias, dbg, grid, smem, st);
        case 64: return launch_attn<64>(tq, tk, tv, p, bias, dbg, grid, smem, st);
        case 80: return launch_attn<80>(tq, tk, tv, p, bias, dbg, grid, smem, st);
        case 96: return launch_attn<96>(tq, tk, tv, p, bias, dbg, grid, smem, st);
        case 128: return launch_attn<128>(tq, tk, tv, p, bias, dbg, grid, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

constexpr size_t kMaxSmem = 227 * 1024;
constexpr int kMaxSwinTable = 4096;  // floats of (2M-1)^2 * H kept in shared memory
constexpr int kMaxSamKeys = 4096;

int run(const void* q, const void* k, const void* v, void* out, float* dbg, int B, int H, int Nq,
        int Nk, int d, float scale, attn_dtype dtype, attn_bias_kind bias_kind,
        const void* bias_args, void* stream) {
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
    if (Nk > (1 << 20)) return fail(ATTN_ERR_UNSUPPORTED, "Nk > 2^20");
    const size_t q_bytes = (size_t)BH * Nq * d * 2, kv_bytes = (size_t)BH * Nk * d * 2;
    if (out && (overlaps(out, q_bytes, q, q_bytes) || overlaps(out, q_bytes, k, kv_bytes) ||
                overlaps(out, q_bytes, v, kv_bytes)))
        return fail(ATTN_ERR_ARG, "out must not alias q, k or v");

    AttnParams p;
    memset(&p, 0, sizeof(p));
    p.out = out;
    p.dbg = dbg;
    p.BH = (int)BH;
    p.H = H;
    p.Nq = Nq;
    p.Nk = Nk;
    p.d = d;
    p.scale_log2 = scale * kLog2e;
    p.is_bf16 = dtype == ATTN_BF16;
    p.q = q;
    const int dpad = dpad_for(d);
    size_t extra = 0;
    int bias = kBiasNone;

    if (bias_kind == ATTN_BIAS_SWIN) {
        const attn_swin_args* a = static_cast<const attn_swin_args*>(bias_args);
        if (!a || !a->table) return fail(ATTN_ERR_ARG, "SWIN bias needs attn_swin_args with a table");
        const int M = a->win;
        if (M < 1 || M * M != Nq || Nk != Nq) return fail(ATTN_ERR_ARG, "SWIN needs Nq == Nk == win*win");
        if (M * M > kBlockM) return fail(ATTN_ERR_UNSUPPORTED, "SWIN windows above 128 tokens");
        if (a->grid_h < M || a->grid_w < M || a->grid_h % M || a->grid_w % M)
            return fail(ATTN_ERR_ARG, "grid_h and grid_w must be positive multiples of win");
        if (a->shift < 0 || a->shift >= M) return fail(ATTN_ERR_ARG, "shift must lie in [0, win)");
        const int nW = (a->grid_h / M) * (a->grid_w / M);
        if (B % nW) return fail(ATTN_ERR_ARG, "B (windows) must be a multiple of the windows per image");
        const int tl = (2 * M - 1) * (2 * M - 1);
        if (tl * H > kMaxSwinTable) return fail(ATTN_ERR_UNSUPPORTED, "Swin table larger than %d floats", kMaxSwinTable);
        p.table = a->table;
        p.win = M;
        p.grid_h = a->grid_h;
        p.grid_w = a->grid_w;
        p.shift = a->shift;
        p.n_w = nW;
        p.n_ww = a->grid_w / M;
        extra = swin_extra_bytes(tl * H);
        bias = kBiasSwin;
    } else if (bias_kind == ATTN_BIAS_SAM_RELPOS) {
        const attn_sam_args* a = static_cast<const attn_sam_args*>(bias_args);
        if (!a || !a->rel_h || !a->rel_w) return fail(ATTN_ERR_ARG, "SAM bias needs attn_sam_args with rel_h, rel_w");
        if (a->q_h < 1 || a->q_w < 1 || a->k_h < 1 || a->k_w < 1) return fail(ATTN_ERR_ARG, "SAM grid sizes must be >= 1");
        if (a->q_h != a->k_h || a->q_w != a->k_w)
            return fail(ATTN_ERR_UNSUPPORTED, "SAM with different query and key grids");
        if (a->q_h * a->q_w != Nq || Nk != Nq) return fail(ATTN_ERR_ARG, "SAM needs Nq == Nk == q_h*q_w");
        if (a->q_h + a->q_w > kBlockM || Nk > kMaxSamKeys)
            return fail(ATTN_ERR_UNSUPPORTED, "SAM grid too large (q_h+q_w <= 128, N <= 4096)");
        p.rel_h = a->rel_h;
        p.rel_w = a->rel_w;
        p.s_h = a->q_h;
        p.s_w = a->q_w;
        extra = sam_extra_bytes(a->q_h, a->q_w, Nk);
        bias = kBiasSam;
    } else if (bias_kind != ATTN_BIAS_NONE) {
        return fail(ATTN_ERR_ARG, "unknown bias kind %d", (int)bias_kind);
    }

    // Tiling.
    int g = std::min(kBlockM / Nq, kBlockN / Nk);
    const bool packed = bias == kBiasSwin || (bias == kBiasNone && g >= 2);
    if (bias == kBiasSwin) g = std::max(g, 1);
    int grid;
    if (packed) {
        p.packed = 1;
        p.g = g;
        p.n_q_tiles = 1;
        p.n_kv_tiles = 1;
        p.kv_cols = (g * Nk + 15) / 16 * 16;
        p.box_rows_q = g * Nq;
        p.box_rows_kv = g * Nk;
        grid = (int)((BH + g - 1) / g);
    } else {
        p.packed = 0;
        p.g = 1;
        p.n_q_tiles = (Nq + kBlockM - 1) / kBlockM;
        p.n_kv_tiles = (Nk + kBlockN - 1) / kBlockN;
        p.kv_cols = kBlockN;
        p.box_rows_q = kBlockM;
        p.box_rows_kv = kBlockN;
        const int64_t nt = BH * p.n_q_tiles;
        if (nt > 0x7fffffff) return fail(ATTN_ERR_UNSUPPORTED, "too many tiles");
        grid = (int)nt;
    }
    const size_t smem = tiles_bytes(dpad) + extra + 1024;
    if (smem > kMaxSmem)
        return fail(ATTN_ERR_UNSUPPORTED, "shared memory %zu B exceeds the per-CTA limit", smem);

    CUtensorMap tq, tk, tv;
    const bool bf = p.is_bf16 != 0;
    int rc;
    if (packed) {
        if ((rc = encode_map(&tq, q, bf, d, BH * Nq, 0, p.box_rows_q))) return rc;
        if ((rc = encode_map(&tk, k, bf, d, BH * Nk, 0, p.box_rows_kv))) return rc;
        if ((rc = encode_map(&tv, v, bf, d, BH * Nk, 0, p.box_rows_kv))) return rc;
    } else {
        if ((rc = encode_map(&tq, q, bf, d, Nq, BH, kBlockM))) return rc;
        if ((rc = encode_map(&tk, k, bf, d, Nk, BH, kBlockN))) return rc;
        if ((rc = encode_map(&tv, v, bf, d, Nk, BH, kBlockN))) return rc;
    }
    p.status = status_ptr();
    if (!p.status) return fail(ATTN_ERR_CUDA, "no CUDA device / status word unavailable");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = dispatch(dpad, tq, tk, tv, p, bias, dbg != nullptr, grid, smem, st);
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

const char* attn_last_error(void) { return sdpa09::g_last_error.c_str(); }

int attn_abi_version(void) { return SDPA09_ABI_VERSION; }

}  // extern "C"
