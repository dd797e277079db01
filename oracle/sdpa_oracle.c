/*
 * sdpa_oracle.c -- plain, slow fp64 CPU oracle for the fused
 * scaled-dot-product attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA path and must never be used as a
 * fallback for it.
 *
 * What it computes, per (batch, head) slice, written out as the definition:
 *
 *   S[i,j] = scale * sum_c Q[i,c] K[j,c] + bias[i,j]          (fp64)
 *   P[i,j] = exp(S[i,j] - max_j S[i,:]) / sum_j exp(...)
 *   O[i,c] = sum_j P[i,j] V[j,c]
 *
 * Sources:
 *  - "视觉大模型训练和推理加速" (NVIDIA Swin talk), section 一 Swin
 *    Transformer简介: attention takes query, key and value; query and key
 *    with a softmax give the attention map, which weights the values.
 *  - "Accelerated Diffusers with PyTorch 2.0", section 加速 Transformer 块:
 *    every scaled-dot-product-attention backend (FlashAttention,
 *    memory-efficient, native C++) computes the same function; the native
 *    C++ one is the high-precision path.  This oracle plays that role.
 *  - Bias kinds:
 *    * SWIN: "视觉大模型训练和推理加速" section 一 names window attention,
 *      window shift and the relative position bias.  The concrete form (a
 *      (2M-1)^2 x H table gathered by relative (row, column) offset, and a
 *      -100 mask between tokens of different regions after the cyclic
 *      shift) is the published Swin definition, restated here.
 *    * SAM_RELPOS: "Accelerating Generative AI (part 1), Segment Anything"
 *      section Bfloat16 半精度 names the image encoder's relative position
 *      term indexed through q_coords / k_coords into rel_pos_resized.  The
 *      concrete form (decomposed rel_h = Q . R_h[idx_h(qh, kh)],
 *      rel_w = Q . R_w[idx_w(qw, kw)] with the unscaled Q, broadcast-added;
 *      idx = qh - kh + S_h - 1 on equal grids) is the published SAM
 *      definition, restated here.  For unequal query and key grids the
 *      caller passes the resized tables and the coordinate-scaled index
 *      tables (oracle/__init__.py computes both from the definition).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - scale multiplies Q.K^T only; the bias is added after scaling.
 *  - the Swin mask adds the finite value -100 (not -inf).
 *  - Swin relative index uses (query - key) offsets; table row-major
 *    [(2M-1)^2][H], fp32 values.
 *  - slice b' of a Swin batch is image * nW + w, windows row-major.
 *  - SAM indices on unequal grids are computed in float32, as the
 *    published code's coordinate scalers are.
 *
 * Everything is double precision.  Inputs arrive as fp64 arrays that the
 * caller converted exactly from the half-precision tensors.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BIAS_NONE = 0, OR_BIAS_SWIN = 1, OR_BIAS_SAM = 2 };

/* Bias description.  Field meanings follow the attention call's arguments. */
typedef struct {
    int kind;
    /* SWIN */
    const double* table; /* [(2M-1)^2][H] */
    int win;             /* M */
    int grid_h, grid_w;  /* tokens per image side (multiples of M) */
    int shift;           /* 0 = no mask */
    /* SAM */
    const double* rel_h; /* [L_h][d], L_h = 2*max(S_h, K_h)-1 (resized if needed) */
    const double* rel_w; /* [L_w][d] */
    int s_h, s_w;        /* query grid s_h x s_w */
    int k_h, k_w;        /* key grid (0, 0: the query grid) */
    const int* idx_h;    /* [s_h][k_h] table row of (qh, kh), or NULL: qh - kh + s_h - 1 */
    const int* idx_w;    /* [s_w][k_w] */
} oracle_bias_t;

/* ---------------------------------------------------------------- Swin -- */

/* Relative position index of query token (ri,ci) and key token (rj,cj)
 * inside one M x M window: row offset and column offset, each shifted to
 * be non-negative, combined row-major over the (2M-1) x (2M-1) table. */
int oracle_swin_index(int M, int ri, int ci, int rj, int cj)
{
    int dr = ri - rj + (M - 1);
    int dc = ci - cj + (M - 1);
    return dr * (2 * M - 1) + dc;
}

/* Region label along one axis of the cyclically shifted map.  After the
 * shift by s, the last s rows (columns) came from the start of the map and
 * the M-s before them are the old tail: three strips
 *   [0, G-M)  [G-M, G-s)  [G-s, G). */
static int swin_strip(int pos, int G, int M, int s)
{
    if (pos < G - M) return 0;
    if (pos < G - s) return 1;
    return 2;
}

/* Mask value between token ti and token tj (both 0..M*M-1, row-major in
 * the window) of window w of one image.  0 inside one region, -100
 * across regions, 0 everywhere when shift == 0. */
double oracle_swin_mask(int M, int Gh, int Gw, int shift, int w, int ti, int tj)
{
    if (shift == 0) return 0.0;
    int nww = Gw / M;
    int wr = w / nww, wc = w % nww;
    int yi = wr * M + ti / M, xi = wc * M + ti % M;
    int yj = wr * M + tj / M, xj = wc * M + tj % M;
    int same = swin_strip(yi, Gh, M, shift) == swin_strip(yj, Gh, M, shift) &&
               swin_strip(xi, Gw, M, shift) == swin_strip(xj, Gw, M, shift);
    return same ? 0.0 : -100.0;
}

/* Full Swin bias for slice (bp, h): table gather + mask. */
static double swin_bias(const oracle_bias_t* a, int H, int bp, int h, int i, int j)
{
    int M = a->win;
    int nW = (a->grid_h / M) * (a->grid_w / M);
    int w = bp % nW;
    int idx = oracle_swin_index(M, i / M, i % M, j / M, j % M);
    return a->table[(size_t)idx * H + h] +
           oracle_swin_mask(M, a->grid_h, a->grid_w, a->shift, w, i, j);
}

/* ----------------------------------------------------------------- SAM -- */

/* Decomposed relative position term for query row i (vector q_i of length
 * d, unscaled) of the s_h x s_w query grid against key j of the key grid
 * (row-major tokens on both). */
static double sam_bias(const oracle_bias_t* a, const double* qi, int d, int i, int j)
{
    int kgh = a->k_h ? a->k_h : a->s_h, kgw = a->k_w ? a->k_w : a->s_w;
    int qh = i / a->s_w, qw = i % a->s_w;
    int kh = j / kgw, kw = j % kgw;
    int ih = a->idx_h ? a->idx_h[qh * kgh + kh] : qh - kh + a->s_h - 1;
    int iw = a->idx_w ? a->idx_w[qw * kgw + kw] : qw - kw + a->s_w - 1;
    const double* rh = a->rel_h + (size_t)ih * d;
    const double* rw = a->rel_w + (size_t)iw * d;
    double h = 0.0, w = 0.0;
    for (int c = 0; c < d; ++c) {
        h += qi[c] * rh[c];
        w += qi[c] * rw[c];
    }
    return h + w;
}

/* ------------------------------------------------------------ generic -- */

static double bias_value(const oracle_bias_t* a, int H, int slice, const double* qi,
                         int d, int i, int j)
{
    if (!a || a->kind == OR_BIAS_NONE) return 0.0;
    if (a->kind == OR_BIAS_SWIN) return swin_bias(a, H, slice / H, slice % H, i, j);
    return sam_bias(a, qi, d, i, j);
}

/* Bias matrix of one slice, Nq x Nk, for the pins. */
int oracle_bias_matrix(const double* q, int H, int slice, int Nq, int Nk, int d,
                       const oracle_bias_t* a, double* bias)
{
    if (Nq <= 0 || Nk <= 0 || d <= 0) return -1;
    const double* qs = q + (size_t)slice * Nq * d;
    for (int i = 0; i < Nq; ++i)
        for (int j = 0; j < Nk; ++j)
            bias[(size_t)i * Nk + j] = bias_value(a, H, slice, qs + (size_t)i * d, d, i, j);
    return 0;
}

/* One output row: row i of slice `slice`.  Writes the d outputs and, when
 * probs != NULL, the Nk probabilities.  `srow` is caller scratch of Nk. */
static void attn_row(const double* q, const double* k, const double* v, int H, int slice,
                     int Nq, int Nk, int d, double scale, const oracle_bias_t* a, int i,
                     double* srow, double* orow, double* probs)
{
    const double* qi = q + ((size_t)slice * Nq + i) * d;
    const double* ks = k + (size_t)slice * Nk * d;
    const double* vs = v + (size_t)slice * Nk * d;
    double m = -INFINITY;
    for (int j = 0; j < Nk; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qi[c] * ks[(size_t)j * d + c];
        srow[j] = scale * dot + bias_value(a, H, slice, qi, d, i, j);
        if (srow[j] > m) m = srow[j];
    }
    double l = 0.0;
    for (int j = 0; j < Nk; ++j) {
        srow[j] = exp(srow[j] - m);
        l += srow[j];
    }
    for (int j = 0; j < Nk; ++j) srow[j] /= l;
    if (probs) memcpy(probs, srow, sizeof(double) * (size_t)Nk);
    for (int c = 0; c < d; ++c) orow[c] = 0.0;
    for (int j = 0; j < Nk; ++j) {
        double p = srow[j];
        for (int c = 0; c < d; ++c) orow[c] += p * vs[(size_t)j * d + c];
    }
}

static int check_args(int BH, int H, int Nq, int Nk, int d, const oracle_bias_t* a)
{
    if (BH <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || BH % H) return -1;
    if (a && a->kind == OR_BIAS_SWIN) {
        int M = a->win;
        if (M <= 0 || Nq != M * M || Nk != M * M || !a->table) return -1;
        if (a->grid_h % M || a->grid_w % M || a->shift < 0 || a->shift >= M) return -1;
    }
    if (a && a->kind == OR_BIAS_SAM) {
        int kgh = a->k_h ? a->k_h : a->s_h, kgw = a->k_w ? a->k_w : a->s_w;
        if (a->s_h <= 0 || a->s_w <= 0 || kgh <= 0 || kgw <= 0 || Nq != a->s_h * a->s_w || Nk != kgh * kgw)
            return -1;
        if ((kgh != a->s_h || kgw != a->s_w) && (!a->idx_h || !a->idx_w)) return -1;
        if (!a->rel_h || !a->rel_w) return -1;
    }
    return 0;
}

/* Whole tensor: q [BH][Nq][d], k, v [BH][Nk][d], out [BH][Nq][d].
 * nthreads <= 0 uses the OpenMP default.  Returns the thread count used. */
int oracle_attn_fwd(const double* q, const double* k, const double* v, double* out, int BH,
                    int H, int Nq, int Nk, int d, double scale, const oracle_bias_t* a,
                    int nthreads)
{
    if (check_args(BH, H, Nq, Nk, d, a)) return -1;
    int used = 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    used = omp_get_max_threads();
#endif
    long long rows = (long long)BH * Nq;
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)Nk);
#pragma omp for schedule(dynamic, 16)
        for (long long r = 0; r < rows; ++r) {
            int slice = (int)(r / Nq), i = (int)(r % Nq);
            attn_row(q, k, v, H, slice, Nq, Nk, d, scale, a, i, srow, out + (size_t)r * d, NULL);
        }
        free(srow);
    }
    return used;
}

/* Selected rows only: row_ids[n] = slice * Nq + i.  out [n][d]. */
int oracle_attn_rows(const double* q, const double* k, const double* v, double* out, int BH,
                     int H, int Nq, int Nk, int d, double scale, const oracle_bias_t* a,
                     const int64_t* row_ids, int64_t n, int nthreads)
{
    if (check_args(BH, H, Nq, Nk, d, a)) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (row_ids[t] < 0 || row_ids[t] >= (int64_t)BH * Nq) return -1;
    int used = 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    used = omp_get_max_threads();
#endif
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)Nk);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n; ++t) {
            int slice = (int)(row_ids[t] / Nq), i = (int)(row_ids[t] % Nq);
            attn_row(q, k, v, H, slice, Nq, Nk, d, scale, a, i, srow, out + (size_t)t * d, NULL);
        }
        free(srow);
    }
    return used;
}

/* Probability matrix of one slice (Nq x Nk) for the softmax pins. */
int oracle_attn_probs(const double* q, const double* k, const double* v, int BH, int H,
                      int Nq, int Nk, int d, double scale, const oracle_bias_t* a, int slice,
                      double* probs, double* out)
{
    if (check_args(BH, H, Nq, Nk, d, a) || slice < 0 || slice >= BH) return -1;
    double* srow = (double*)malloc(sizeof(double) * (size_t)Nk);
    for (int i = 0; i < Nq; ++i)
        attn_row(q, k, v, H, slice, Nq, Nk, d, scale, a, i, srow, out + (size_t)i * d,
                 probs + (size_t)i * Nk);
    free(srow);
    return 0;
}
