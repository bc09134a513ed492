// One work item of the combine (article "O MoK do Cursor ...", section 03: Combine and the
// final weighted fusion): out[t] = bf16( sum_{j=0}^{k-1} w[t,j] * Y[row(t,j)] ) for 512
// columns of one token, fp32 accumulation in fixed slot order j, one rounding. Shared by the
// combine kernel and the persistent forward so that both give the same bytes.
#pragma once
#include "route_kernels.cuh"

namespace moe {

// it: item index within [t0, t1) x (H / 512 column chunks); nch = column chunks per token;
// shift: ring row - padded row; [lo, hi): the padded rows of the macrobatch, the only rows
// its slots may name (a slot row outside them raises MOE_ERR_INTERNAL and the slot is left
// out, so no load leaves the ring). Y is read with plain (coherent) loads: in the persistent
// forward it was written earlier in the same kernel.
__device__ __forceinline__ void combine_item(const CombineArgs &a, int it, int nch, int shift, int lo, int hi,
                                             int lane) {
    const int vecs = a.H / 8;   // a multiple of 32
    const int t = a.t0 + it / nch;
    // two vectors per lane, rows in batches of 4: 8 loads of 16 B per lane in flight
    const int v0 = (it % nch) * 64 + lane;
    const bool two = v0 + 32 < vecs;
    float acc[2][8];
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[p][i] = 0.0f;
    for (int j0 = 0; j0 < a.k; j0 += 4) {
        const int nj = min(4, a.k - j0);
        int rows[4];
        float ws[4];
        uint4 y[2][4];
        bool ok[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            ok[j] = false;
            if (j < nj) {
                const int prow = a.slot_row[(size_t)t * a.k + j0 + j];
                ok[j] = prow >= lo && prow < hi;
                if (!ok[j] && lane == 0) raise_status(a.status, kStatusInternal);
                rows[j] = ok[j] ? prow + shift : 0;
                ws[j] = ok[j] ? a.w[(size_t)t * a.k + j0 + j] : 0.0f;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (j < nj) {
                y[0][j] = ok[j] ? ld_v4(a.Y + (size_t)rows[j] * a.H + v0 * 8) : make_uint4(0, 0, 0, 0);
                if (two) y[1][j] = ok[j] ? ld_v4(a.Y + (size_t)rows[j] * a.H + (v0 + 32) * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (j < nj && (p == 0 || two)) {
                    const uint32_t q[4] = {y[p][j].x, y[p][j].y, y[p][j].z, y[p][j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[p][2 * i] = fmaf(ws[j], bf16lo(q[i]), acc[p][2 * i]);
                        acc[p][2 * i + 1] = fmaf(ws[j], bf16hi(q[i]), acc[p][2 * i + 1]);
                    }
                }
    }
#pragma unroll
    for (int p = 0; p < 2; ++p)
        if (p == 0 || two)
            st_v4(a.out + (size_t)t * a.H + (v0 + 32 * p) * 8,
                  make_uint4(pack_bf16x2(acc[p][0], acc[p][1]), pack_bf16x2(acc[p][2], acc[p][3]),
                             pack_bf16x2(acc[p][4], acc[p][5]), pack_bf16x2(acc[p][6], acc[p][7])));
}

}  // namespace moe
