// attn_bwd_window.cuh -- parameters and launcher of the short-sequence
// backward kernel (attn_bwd_window.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

namespace sdpa09 {

struct BwdParams {
    const void *q, *k, *v, *o, *dout;  // [BH][N][d] 16-bit
    void *dq, *dk, *dv;                // outputs, same layouts
    int BH, H, Nq, Nk, d;
    float scale;
    int is_bf16;
    // Swin bias (windows layout)
    int swin;
    const float* table;  // [(2M-1)^2][H]
    float* d_table;      // gradient of table, accumulated (+=)
    int win, grid_h, grid_w, shift, n_w, n_ww;
};

// Dynamic shared memory of one CTA: the slice's Q, K, V, O, dO (16-bit), the
// padded score matrix and row terms (fp32), the Swin table gradient (fp32).
size_t bwd_window_smem_bytes(int Nq, int Nk, int d, int win, int H, bool swin);

cudaError_t launch_bwd_window(const BwdParams& p, int grid, size_t smem, cudaStream_t stream);

}  // namespace sdpa09
