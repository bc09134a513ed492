// Launchers of the MXFP8 quantisers (mx_quant.cu).
#pragma once
#include "moe_common.cuh"

namespace moe {

// bf16 rows [nrows, C] -> E4M3 rows [nrows, C] + E8M0 scale atoms (K = C), in place
// order: the weight copies whose contraction axis is the stored row.
struct MxRowsArgs {
    const bf16 *src;
    uint8_t *codes, *scales;
    int nrows, C;
};
cudaError_t launch_mx_rows(const MxRowsArgs &a, int max_rows, int num_sms, cudaStream_t s);

// batch x bf16 [R][C] -> batch x E4M3 [C][R] + scale atoms (K = R).
// R and C multiples of 128. Input rows >= *r_limit_ptr (if set) are
// treated as zeros and their 128-row blocks skipped.
// Gather mode (row_slot != null, batch 1): input row r is token row_slot[r] / k
// of src (zeros when row_slot[r] < 0), so expert-sorted rows are quantised
// along the token axis straight from the token-ordered tensor.
// Interleaved order (offp != null, batch 1): the rows form ilv_nseg runs of
// 128-row multiples, [offp[s], offp[s + 1]), ilv_E per macrobatch, each at most
// ilv_jb blocks of 128 rows; block j of every expert of a macrobatch is taken
// before block j + 1 of any, so the copies of one token taken by different
// experts are read close together in time and the source leaves HBM about once.
// r_limit_ptr is unused.
// Row-wise copy as well (rcodes != null, batch 1): the same input rows quantised
// along C into rcodes [R][C] + scale atoms rscales (K = C), destination row =
// input row; the fused form of an mx_rows pass over the same gathered rows.
struct MxTransposeArgs {
    const bf16 *src;
    uint8_t *codes, *scales;
    int R, C;
    const int32_t *r_limit_ptr;
    const int32_t *row_slot;
    int k;
    const int32_t *offp;
    int ilv_E, ilv_nseg, ilv_jb;
    uint8_t *rcodes, *rscales;
    int nslots;     // gather mode: a row's slot lies in [-1, nslots); one outside raises
    int *status;    // MOE_ERR_INTERNAL here and the row is read as zeros
};
cudaError_t launch_mx_transpose(const MxTransposeArgs &a, int batch, cudaStream_t s);

}  // namespace moe
