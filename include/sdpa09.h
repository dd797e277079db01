/*
 * sdpa09.h -- C ABI of the GB300 (sm_103a) fused scaled-dot-product
 * attention library, libsdpa09.so: the forward pass (attn_fwd,
 * attn_fwd_varlen, attn_fwd_train) and its backward (attn_bwd).
 *
 * The operation (per batch-head slice):
 *
 *     O = softmax(scale * Q . K^T + bias) . V
 *
 * "视觉大模型训练和推理加速" (NVIDIA Swin talk), section 一 Swin Transformer简介:
 * attention takes query, key and value; query and key with a softmax give
 * the attention map that weights the values; multi-head attention repeats
 * this per head.  "Accelerated Diffusers with PyTorch 2.0", section 加速
 * Transformer 块: the scaled-dot-product-attention function takes
 * (query, key, value) and every backend computes the same result.  The
 * bias kinds are described at attn_bias_kind.
 *
 * Conventions shared by the attention calls:
 *  - All tensors are device pointers owned by the caller.  The library
 *    never allocates per call, never copies host<->device and never
 *    synchronises the stream (attn_device_status, a status read, does) ("PyTorch团队重写「分割一切」模型，比原始实现快8倍",
 *    section on the bf16 baseline: an index operation whose host-side
 *    coordinates forced a copy and a blocking cudaStreamSynchronize was the
 *    first bottleneck removed).  Bias arguments are read from the host
 *    struct at call time and passed by value to the kernel.
 *  - Layout: Q and O are [B][H][Nq][d], K and V are [B][H][Nk][d], all
 *    contiguous with d innermost, in the dtype given (bf16 or fp16); the
 *    Swin image layout and attn_fwd_varlen document their own.  Each
 *    pointer must be 16-byte aligned and d a multiple of 8 (the row pitch
 *    must be a multiple of 16 bytes for the tensor-memory-access engine).
 *  - Work runs on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream).  The call returns once the kernel is enqueued.
 *  - Return value 0 on success, a negative ATTN_ERR_* code otherwise;
 *    attn_last_error() then describes the failure.  No exception or abort
 *    crosses the ABI.  Arguments are validated before any CUDA call.
 */
#ifndef SDPA09_H
#define SDPA09_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDPA09_ABI_VERSION 6

typedef enum {
    ATTN_BF16 = 0, /* bfloat16 Q/K/V/O ("model.to(torch.bfloat16)" in the SAM rewrite) */
    ATTN_FP16 = 1  /* float16 Q/K/V/O (torch.cuda.amp in the Swin talk, fp16 diffusers) */
} attn_dtype;

/* Bias added to scale * Q.K^T before the softmax.
 *
 * ATTN_BIAS_NONE: no bias -- the diffusion UNet self- and cross-attention
 *   of "Accelerated Diffusers with PyTorch 2.0", section 在 diffusers 中使用缩放点积注意力机制.
 *
 * ATTN_BIAS_SWIN: Swin window attention with relative position bias and the
 *   shifted-window mask ("视觉大模型训练和推理加速", section 一: window
 *   attention, window shift, relative position bias).  Each slice is one
 *   M x M window (Nq = Nk = M*M, tokens row-major in the window); the
 *   batch index b counts windows, b = image * nW + w with window w
 *   row-major over the (grid_h/M) x (grid_w/M) window grid.  For query
 *   token (ri,ci) and key token (rj,cj) of head h the bias is
 *       table[((ri-rj+M-1)*(2M-1) + (ci-cj+M-1)) * H + h]
 *   plus -100 when, after a cyclic shift by `shift`, the two tokens lie in
 *   different regions (strips [0,G-M), [G-M,G-shift), [G-shift,G) along
 *   each axis); shift = 0 means no mask.  The cyclic shift and window
 *   partition themselves happen before this call.
 *
 * ATTN_BIAS_SAM_RELPOS: SAM image-encoder decomposed relative position
 *   ("Accelerating Generative AI (part 1), Segment Anything", section
 *   Bfloat16 半精度: the encoder indexes rel_pos_resized with q_coords /
 *   k_coords).  Tokens are row-major on a q_h x q_w grid; for query
 *   i = (qh,qw) and key j = (kh,kw)
 *       bias = Q_i . R_h[qh-kh+q_h-1] + Q_i . R_w[qw-kw+q_w-1]
 *   with the unscaled Q, on equal query and key grids.  Unequal grids (keys
 *   on a k_h x k_w grid) and tables of another length are accepted too: the
 *   row index then goes through the coordinate scalers and the tables are
 *   resampled, as attn_sam_args describes.
 */
typedef enum {
    ATTN_BIAS_NONE = 0,
    ATTN_BIAS_SWIN = 1,
    ATTN_BIAS_SAM_RELPOS = 2
} attn_bias_kind;

typedef struct {
    const float* table; /* device, [(2*win-1)^2][H] row-major fp32 */
    int win;            /* M, window side in tokens (7 for Swin-T) */
    int grid_h, grid_w; /* tokens per image side, multiples of win (56, 56) */
    int shift;          /* cyclic shift, 0 <= shift < win; 0 = no mask */
    int layout;         /* ATTN_SWIN_WINDOWS or ATTN_SWIN_IMAGE, see below */
} attn_swin_args;

/* Token layouts of q, k, v and out under the Swin bias.
 *   ATTN_SWIN_WINDOWS: [B windows][H][win*win][d] -- already cyclically
 *     shifted and partitioned, windows row-major within each image.
 *   ATTN_SWIN_IMAGE:   [B / nW images][grid_h][grid_w][H][d] -- the natural
 *     token layout of the feature map; the call applies the cyclic shift by
 *     -shift and the window partition while loading ("视觉大模型训练和推理加速"
 *     section 一, window attention on the shifted map; section 二, both are
 *     index mapping) and their inverse while storing, so no rolled or
 *     partitioned copy is made.  B still counts windows. */
enum { ATTN_SWIN_WINDOWS = 0, ATTN_SWIN_IMAGE = 1 };

/* SAM decomposed relative position ("Accelerating Generative AI (part 1),
 * Segment Anything", section Bfloat16 半精度: the image encoder's rel-pos term,
 * q_coords / k_coords indexing rel_pos_resized).  For query (qh, qw) and key
 * (kh, kw) the bias is Q . R_h'[ih] + Q . R_w'[iw] with the unscaled Q, where
 * R' is the table resampled linearly to 2*max(q, k)-1 rows when its length
 * differs (half-pixel centres, no corner alignment) and, per axis,
 * i = trunc(q_i * max(k/q, 1) - k_j * max(q/k, 1) + (k-1) * max(q/k, 1)) in
 * float32 -- on equal grids simply qh - kh + q_h - 1. */
typedef struct {
    const void* rel_h;  /* device, [rel_h_len][d], same dtype as Q */
    const void* rel_w;  /* device, [rel_w_len][d], same dtype as Q */
    int q_h, q_w;       /* query grid; Nq = q_h * q_w (sides <= 64) */
    int k_h, k_w;       /* key grid; Nk = k_h * k_w (sides <= 64) */
    int rel_h_len;      /* rows of rel_h, 1..128; 0 = 2*max(q_h, k_h)-1 */
    int rel_w_len;      /* rows of rel_w, 1..128; 0 = 2*max(q_w, k_w)-1 */
} attn_sam_args;

enum {
    ATTN_OK = 0,
    ATTN_ERR_ARG = -1,            /* null/misaligned pointer, bad size, bad bias args */
    ATTN_ERR_UNSUPPORTED = -2,    /* valid but not implemented (e.g. d > 128, SAM grid sides > 64) */
    ATTN_ERR_CUDA = -3,           /* a CUDA runtime/driver call or the launch failed */
    ATTN_ERR_DEVICE_TIMEOUT = -4  /* a kernel wait ran out of time (attn_device_status) */
};

/* attn_fwd -- the fused forward pass O = softmax(scale*Q.K^T + bias).V.
 *
 *  q, k, v    device inputs, layout above; not modified.
 *  out        device output [B][H][Nq][d]; fully overwritten; must not
 *             alias q, k or v.
 *  B, H       batch (or window count) and heads, >= 1.
 *  Nq, Nk     query and key lengths, >= 1 (Nk <= 2^20).
 *  d          head dim: a multiple of 8, 8 <= d <= 128.
 *  scale      multiplies Q.K^T only (usually 1/sqrt(d)).
 *  dtype      element type of q, k, v, out (and SAM tables).
 *  bias_kind  see attn_bias_kind; bias_args points to attn_swin_args or
 *             attn_sam_args (host memory, read during the call), or NULL
 *             for ATTN_BIAS_NONE.
 *  stream     cudaStream_t to enqueue on.
 *
 * Accumulation is fp32 (scores, softmax, P.V); P is rounded to the input
 * dtype before the second product; O is rounded to nearest even.
 *
 * Swin windows whose bias rows do not fit shared memory (more than 64
 * tokens, or many heads) add the bias through the tensor core, as 16-bit
 * operands holding table / scale and -100 / scale.  There a zero scale, or
 * |scale| < 100 / 65504 for fp16 (100 / 3.3e38 for bf16), returns
 * ATTN_ERR_UNSUPPORTED, and table entries must satisfy
 * |table / scale| <= 65504 for fp16 (beyond it they saturate to infinity).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int H, int Nq,
             int Nk, int d, float scale, attn_dtype dtype, attn_bias_kind bias_kind,
             const void* bias_args, void* stream);

/* attn_fwd_train -- attn_fwd that also writes each query row's log-sum-exp,
 * the statistic the backward pass (attn_bwd) recomputes the probabilities
 * from: the Swin talk ("视觉大模型训练和推理加速" section 二) builds the forward
 * and the backward computation of its attention operators alike, for
 * training.  For row i of slice b,
 *     lse[b * Nq + i] = log sum_j exp(scale * Q_i . K_j + bias_ij)
 * (natural logarithm, fp32), so that P_ij = exp(scale * Q_i . K_j + bias_ij
 * - lse_i).  With the Swin image layout the rows are still counted in the
 * windows order (b a window-head slice, i a token of the window).
 *
 *  lse        device fp32 [B][H][Nq], fully overwritten, 4-byte aligned; must
 *             not alias the other tensors.
 *  the rest   as for attn_fwd; out is written exactly as attn_fwd writes it.
 * Returns as attn_fwd (ATTN_ERR_ARG also for a null lse).
 */
int attn_fwd_train(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                   int Nq, int Nk, int d, float scale, attn_dtype dtype, attn_bias_kind bias_kind,
                   const void* bias_args, void* stream);

/* attn_fwd_varlen -- attention over a batch of sequences of different
 * lengths packed in one buffer, each sequence attending only to itself: a
 * nested tensor ("PyTorch团队重写「分割一切」模型" and its translations: Nested
 * Tensor batches data of non-uniform size, such as images of different
 * sizes, in one tensor, packing {tensor, mask}).  For sequence s with
 * Lq_s = cu_seqlens_q[s+1] - cu_seqlens_q[s] queries and Lk_s keys,
 * O_s = softmax(scale * Q_s.K_s^T) . V_s per head, no bias -- the same as a
 * padded batch whose padded keys are masked out.
 *
 *  q, out     device, the concatenation over s of [H][Lq_s][d]: the buffer of
 *             a contiguous (n_seq, H, Lq*, d) nested tensor; out is fully
 *             overwritten and must not alias q, k or v.
 *  k, v       device, the concatenation over s of [H][Lk_s][d].
 *  cu_seqlens_q, cu_seqlens_k
 *             HOST int32 [n_seq + 1]: token offsets, starting at 0 and
 *             nondecreasing; read during the call.  Lk_s >= 1 wherever
 *             Lq_s >= 1; Lk_s <= 2^20.
 *  n_seq      1 .. ATTN_VARLEN_MAX_SEQ sequences.
 *  H, d, scale, dtype, stream   as for attn_fwd.
 *
 * Returns ATTN_OK (also when no sequence has a query: then nothing is
 * launched and the tensor pointers may be null), ATTN_ERR_ARG,
 * ATTN_ERR_UNSUPPORTED (more than ATTN_VARLEN_MAX_SEQ sequences, d > 128)
 * or ATTN_ERR_CUDA.  Sequences never interact: the rows of a neighbouring
 * sequence that a tile holds are masked (keys) or cleared (values) before
 * use, so even non-finite values there leave a sequence's output unchanged.
 *
 * With d <= 64, sequences of at most 32 (64) query and key tokens are
 * packed: four (two) (sequence, head) slices share one 128-row tile, the way
 * the Swin windows of attn_fwd do, but each slice's P.V reads only its own
 * values, so packed sequences stay apart in the same sense.  The call then
 * makes up to three launches on the stream (longer sequences, slices of 32,
 * slices of 64 rows); an error stops at the first failing one.
 */
#define ATTN_VARLEN_MAX_SEQ 128
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* out, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int n_seq, int H, int d, float scale, attn_dtype dtype,
                    void* stream);

/* attn_bwd -- gradients of attn_fwd for training: the Swin talk
 * ("视觉大模型训练和推理加速" section 二) builds the forward and the backward
 * computation of its window operators alike.  With
 * P = softmax(scale*Q.K^T + bias), O = P.V and dO = dout:
 *   dV = P^T dO,  dS = P * (dO V^T - rowsum(dO * O)),
 *   dQ = scale dS K,  dK = scale dS^T Q,
 * and the bias gradients: Swin, dS summed into the table row of each
 * (query, key) pair of each head (the mask is constant); SAM
 * ("Accelerating Generative AI (part 1), Segment Anything", Bfloat16
 * section: the decomposed rel-pos terms rel_h[q][kh] = Q_q . R_h[qh-kh+S-1],
 * rel_w alike), dRelH[q][kh] = sum over kw of dS[q][(kh,kw)] (dRelW alike),
 * then dQ_q += sum_kh dRelH[q][kh] R_h[qh-kh+S-1] + the same over kw, and
 * dR_h[j] = sum of dRelH[q][kh] Q_q over the (q, kh) with qh-kh+S-1 = j.
 *
 *  q, k, v    device inputs of the forward call, layout [B][H][N][d];
 *  out        device O of the forward call (rowsum(dO * O) is taken from it);
 *  dout       device gradient of the loss with respect to O, like out;
 *  lse        device fp32 [B][H][Nq], the row log-sum-exp attn_fwd_train
 *             wrote; may be NULL when Nq <= 128 and Nk <= 128 (each row then
 *             fits one key tile and its softmax is recomputed exactly);
 *  dq, dk, dv device outputs, like q, k, v; fully overwritten.
 *  B, H, Nq, Nk, d, scale, dtype as for attn_fwd.
 *  bias_kind  ATTN_BIAS_NONE, ATTN_BIAS_SWIN (bias_args as for attn_fwd,
 *             either token layout: with ATTN_SWIN_IMAGE, q, k, v, out, dout
 *             and dq, dk, dv are [images][grid_h][grid_w][H][d] and the
 *             kernel folds the shift and the window partition into its loads
 *             and their inverse into its stores) or ATTN_BIAS_SAM_RELPOS (bias_args as for
 *             attn_fwd, with equal square query and key grids of side
 *             S = 14, 48 or 64 and tables of 1 to 128 rows; tables of another
 *             length than 2*S-1 are resampled to 2*S-1 rows as the forward
 *             resamples them, and their gradients returned through the
 *             transposed resampling).
 *  d_bias     device fp32 bias gradient, ADDED to (the caller zeroes it
 *             first): ATTN_BIAS_SWIN: [(2*win-1)^2][H]; ATTN_BIAS_SAM_RELPOS:
 *             [rel_h rows][d] for R_h followed by [rel_w rows][d] for R_w
 *             (the tables' lengths as given); NULL otherwise.
 *  workspace, workspace_bytes
 *             device scratch of at least attn_bwd_workspace_size(...) bytes,
 *             16-byte aligned, owned by the caller (NULL when that size is
 *             0); its contents on entry do not matter.
 *  stream     cudaStream_t to enqueue on.
 * Products run on the tensor cores with fp32 accumulation from 16-bit
 * operands (P and dS rounded to the input type); the SAM row sums of dS and
 * their products with Q and the tables stay in fp32 (CUDA cores); outputs
 * are rounded to nearest even.  Windows (Nq, Nk <= 128, d <= 64, no SAM
 * bias) take one kernel and no workspace; longer sequences, d > 64 or the
 * SAM bias take a pre-pass, a key pass (dK, dV), a query pass (dQ) and, for
 * SAM, two post-passes, with lse and the workspace.  Returns ATTN_OK,
 * ATTN_ERR_ARG, ATTN_ERR_UNSUPPORTED (see the limits) or ATTN_ERR_CUDA.
 * Limits: d <= 80 (d <= 64 with the Swin bias, 48 < d <= 80 with the SAM
 * bias); B*H*N < 2^31.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale,
             attn_dtype dtype, attn_bias_kind bias_kind, const void* bias_args, float* d_bias,
             void* workspace, size_t workspace_bytes, void* stream);

/* attn_bwd_workspace_size -- bytes of device scratch attn_bwd needs for these
 * arguments (0 when none is needed).  Reads only its arguments (and the host
 * struct bias_args points to). */
size_t attn_bwd_workspace_size(int B, int H, int Nq, int Nk, int d, attn_bias_kind bias_kind,
                               const void* bias_args);

/* attn_bwd_noalloc -- attn_bwd without a bias and without a caller
 * workspace: the same gradients, for callers that cannot allocate device
 * memory at the point where they run the backward pass -- code whose device
 * memory all belongs to a pool or fixed budget set up by someone else (an
 * engine with a preallocated arena, a plugin whose host forbids allocation
 * while it runs), or code with no allocator at hand.  It allocates nothing:
 * its scratch (one fp32 value per query row) is a fixed array inside the
 * library, 4 MiB on every GPU that loads the library, held until the process
 * exits.  The reference pages have no counterpart to this call.
 *
 *  Arguments as for attn_bwd with bias_kind ATTN_BIAS_NONE, no d_bias and no
 *  workspace.  B * H * Nq must not exceed 2^20 (1048576) query rows; larger
 *  calls return ATTN_ERR_UNSUPPORTED before any CUDA call.
 *  The first call on a device looks up the array's device address (with that
 *  device current); make that first call before any stream capture.
 *  Every call uses the same array and leaves its last contents there (nothing
 *  in it needs to start at zero: each call writes what it reads).  Calls
 *  whose kernels overlap on the GPU -- on different streams, or from several
 *  threads -- race on the array; order them on one stream.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                     float scale, attn_dtype dtype, void* stream);

/* attn_debug_bias -- test hook for the in-kernel bias builders.
 *
 * Runs the same kernel as attn_fwd with the same arguments but, instead
 * of O, writes the bias value the builder adds to each score (in natural
 * units, before the softmax; masked-out key padding excluded) to
 * bias_out [B][H][Nq][Nk] fp32 (device).  Meant for small shapes.
 */
int attn_debug_bias(const void* q, const void* k, const void* v, float* bias_out, int B, int H,
                    int Nq, int Nk, int d, float scale, attn_dtype dtype,
                    attn_bias_kind bias_kind, const void* bias_args, void* stream);

/* attn_device_status -- synchronises `stream`, then reads and clears the
 * library's device status word.  Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT
 * when some kernel wait ran out of time since the last call (the kernel
 * then stopped early and its output is invalid), or ATTN_ERR_CUDA. */
int attn_device_status(void* stream);

/* attn_selftest_wait_timeout -- test hook for the failure path of the
 * kernels' bounded waits; the pages have no counterpart.  Launches on
 * `stream` one warp that waits on a shared-memory barrier nothing arrives
 * on, through the same bounded wait the attention kernel uses but with a
 * limit of `limit_us` microseconds (1 .. 2000000).  The wait gives up, the
 * kernel stores its code (9) in the device status word and returns, so the
 * context stays usable; attn_device_status then reports
 * ATTN_ERR_DEVICE_TIMEOUT.  Returns ATTN_OK once launched, ATTN_ERR_ARG for a
 * limit out of range (before any CUDA call), ATTN_ERR_CUDA otherwise. */
int attn_selftest_wait_timeout(unsigned limit_us, void* stream);

/* attn_last_error -- text of the last failure on the calling thread
 * (empty string when none).  The pointer stays valid until the next call
 * on the same thread. */
const char* attn_last_error(void);

/* attn_abi_version -- SDPA09_ABI_VERSION of the built library. */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SDPA09_H */
