// Launchers of the MXFP8 quantisers (mx_quant.cu).
#pragma once
#include "moe_common.cuh"

namespace moe {

// bf16 rows [*, C] -> E4M3 rows [*, C] + E8M0 scale atoms (K = C).
// Gather mode (row_slot != null): rows r in [offp[beg], offp[end]) take source
// token row_slot[r] / k (zeros when row_slot[r] < 0). Identity mode
// (row_slot == null): rows [0, nrows), or [offp[beg], offp[end]) when offp is set.
// Destination row = dst_row0 + r - first row.
struct MxRowsArgs {
    const bf16 *src;
    uint8_t *codes, *scales;
    const int32_t *row_slot, *offp;
    int beg, end, nrows;
    int dst_row0, C, k;
};
cudaError_t launch_mx_rows(const MxRowsArgs &a, int max_rows, int num_sms, cudaStream_t s);

// batch x bf16 [R][C] -> batch x E4M3 [C][R] + scale atoms (K = R).
// R multiple of 128, C multiple of 64. Input rows >= *r_limit_ptr (if set) are
// treated as zeros and their 128-row blocks skipped.
// Gather mode (row_slot != null, batch 1): input row r is token row_slot[r] / k
// of src (zeros when row_slot[r] < 0), so expert-sorted rows are quantised
// along the token axis straight from the token-ordered tensor.
struct MxTransposeArgs {
    const bf16 *src;
    uint8_t *codes, *scales;
    int R, C;
    const int32_t *r_limit_ptr;
    const int32_t *row_slot;
    int k;
};
cudaError_t launch_mx_transpose(const MxTransposeArgs &a, int batch, cudaStream_t s);

}  // namespace moe
