// attn_bwd_sam.cuh -- parameters and launchers of the SAM rel-pos parts of the
// long-sequence backward (attn_bwd_sam_rel.cu, attn_bwd_sam.cu).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace sdpa09 {

struct SamBwdParams {
    const void* q;              // [BH][Nq][d] 16-bit
    const void *rel_h, *rel_w;  // [2S-1][d] 16-bit tables
    __half* rel;                // pre-pass output: [BH*Nq][rel_stride] fp16, rel_h at 0, rel_w at rw0 (log2 units)
    const float* dq32;          // [BH*Nq][d] scale dS.K from the query pass
    float* d_relh;              // [BH*Nq][S] dRelH (on 14-wide grids cleared by the pre-pass, then added to)
    const float* d_relw;        // [2][BH*Nq][S] dRelW, one array per column half of the query pass
    void* dq;                   // [BH*Nq][d] 16-bit output
    float* d_bias;              // [2S-1][d] gradient of R_h, then [2S-1][d] of R_w (added to)
    int BH, Nq, d, rel_stride, rw0;
    int groups;                 // slice groups of the table pass (sam_bwd_groups)
    int* status;                // device status word (a bounded wait that gave up)
};

// Row layout of the pre-pass output for a grid of side S: rel_h at
// [0, S), rel_w at [kRw0, kRw0 + S), each part padded to a multiple of 8.
template <int S>
struct RelLayout {
    static constexpr int kRw0 = (S + 7) / 8 * 8;
    static constexpr int kStride = 2 * kRw0;
};

int sam_bwd_groups(int S, int BH, int nsm);
// rel pre-pass on the tensor cores (attn_bwd_sam_rel.cu): rel_h, rel_w per
// query row into p.rel; on 14-wide grids also clears p.d_relh
cudaError_t launch_bwd_sam_rel_tc(const SamBwdParams& p, int S, bool bf, int nsm, cudaStream_t st);
cudaError_t launch_bwd_sam_post(const SamBwdParams& p, int S, bool bf, int nsm, cudaStream_t st);
// tables of another length: the resampled 16-bit copy [lout][d] of a table
// [lin][d] (also clears n floats at dz), and the transposed resampling of the
// gradient of that copy added to the table's gradient
cudaError_t launch_bwd_sam_resample(const void* src, void* dst, int lin, int lout, int d, bool bf, float* dz, int n,
                                    cudaStream_t st);
cudaError_t launch_bwd_sam_unresample(const float* dRr, float* dR, int lin, int lout, int d, cudaStream_t st);

}  // namespace sdpa09
