// Argument blocks and launchers of the router / schedule / dispatch / combine
// kernels and of the token-side backward (route_kernels.cu).
#pragma once
#include "moe_common.cuh"

namespace moe {

struct RouterArgs {
    const bf16 *x, *Wr;
    const float *bias;      // may be null
    bf16 *WrT;              // scratch [EP, H]
    int T, H, E, k;
    float *probs;           // [T, E]
    int32_t *ids;           // [T, k]
    float *w;               // [T, k]
    int32_t *ids2;          // optional second copy (saved buffer)
    float *w2;
};
cudaError_t launch_router(const RouterArgs &a, cudaStream_t s);

struct SchedArgs {
    const int32_t *ids;     // [T*k]
    int T, k, E, Mb, nM, chunks_per_mb, nchunks;
    int *chunk_counts, *chunk_base;   // [nchunks * E]
    int32_t *counts;        // [nM*E]
    int32_t *offsets;       // [nM*(E+1)]
    int32_t *offp;          // [nM*E + 1] padded run starts
    int32_t *sorted_to_slot, *slot_to_sorted;   // [T*k]
    int32_t *slot_row;      // optional [T*k] padded row of each slot
    int32_t *row_slot;      // optional [rows_pad_max] slot of each padded row
    int *ready;             // optional [ready_n] GEMM1 minibatch counters, zeroed by the scan
    int ready_n;
    // optional further counter ranges the scan zeroes (the decode kernel's, the persistent
    // forward's), so that no memset breaks the chain of programmatic launches
    int *zero[2];
    int zero_n[2];
    int *status;
};
cudaError_t launch_schedule(const SchedArgs &a, cudaStream_t s);

struct DispatchArgs {
    const bf16 *src;        // [T, H]
    bf16 *dst;
    const int32_t *row_slot, *offp;
    int beg, end;           // rows [offp[beg], offp[end])
    int dst_row0;
    int H, k;
    int nslots;             // T * k: a row's slot lies in [-1, nslots) (-1 = padding)
    int *status;            // MOE_ERR_INTERNAL on an index outside its range (the row is zeroed)
};
cudaError_t launch_dispatch(const DispatchArgs &a, int max_rows, int num_sms, cudaStream_t s);

struct CombineArgs {
    const bf16 *Y;          // ring rows
    const int32_t *slot_row, *offp;
    const float *w;
    bf16 *out;
    int t0, t1, k, H, E, m, ring_base;
    int *status;            // MOE_ERR_INTERNAL on a slot row outside macrobatch m (the slot is skipped)
};
cudaError_t launch_combine(const CombineArgs &a, int num_sms, cudaStream_t s);

struct RouterBwdArgs {
    const float *dw_part;   // [rows, nparts]
    int nparts;
    const int32_t *slot_row, *ids;
    const float *w, *probs;
    float *dlogits;         // [T, E]
    int T, k, E;
    int rows;               // padded rows: a slot's row lies in [0, rows)
    int *status;            // MOE_ERR_INTERNAL on a row outside it (the slot's dw is taken as 0)
};
struct RevDispatchArgs {
    const bf16 *dXs;        // [rows, H]
    const int32_t *slot_row;
    const float *dlogits;
    const bf16 *Wr;
    bf16 *dx;
    int T, k, E, H;
    int rows;               // padded rows: a slot's row lies in [0, rows)
    int *status;            // MOE_ERR_INTERNAL on a row outside it (the row is skipped)
};
struct RouterWgradArgs {
    const bf16 *x;
    const float *dlogits;
    float *part;            // [splits, E, H]
    float *dWr;
    int T, H, E, splits, accumulate;
};
cudaError_t launch_router_bwd_dlogits(const RouterBwdArgs &rb, cudaStream_t s);
cudaError_t launch_reverse_dispatch(const RevDispatchArgs &rd, cudaStream_t s);
cudaError_t launch_router_wgrad(const RouterWgradArgs &rw, cudaStream_t s);

}  // namespace moe
