// Shared definitions of the MoE layer kernels: sizes, buffer layouts inside
// the caller's workspace / saved buffers, and small device helpers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx_sm103.cuh"

namespace moe {

constexpr int kMaxExperts = 64;
constexpr int kRowPad = 128;          // each (macrobatch, expert) run of sorted rows is padded to this
constexpr int kSchedChunk = 1024;     // routed slots per schedule block
constexpr int kSchedWarps = 8;
constexpr int kMxBlock = 32;          // MXFP8 block along the contraction axis

// status codes written to the device status word (values of moe_status_t)
constexpr int kStatusTimeout = 5;
constexpr int kStatusInternal = 6;

typedef __nv_bfloat16 bf16;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Host-computed layout of every buffer; identical for the forward and the
// backward of one configuration. All offsets are in bytes from the buffer base.
struct Layout {
    // shape
    int T, H, F, E, k, R;
    int precision;
    int Mb, nM;             // macrobatch tokens / count
    int rows_pad_max;       // bound on padded sorted rows (all macrobatches)
    int half_rows;          // bound on padded rows of one macrobatch (one ring half)
    int ring_halves;        // 1 or 2
    int nchunks;            // schedule blocks
    int chunks_per_mb;
    int minibatch_rows;
    int num_sms;
    int dwr_splits;         // token splits of the router-weight gradient
    // saved buffer
    size_t s_ids, s_w, s_probs, s_counts, s_offsets, s_offp, s_s2sorted, s_sorted2s, s_slot_row,
        s_row_slot, s_a, s_b, saved_bytes;
    // workspace (header first, then a region shared by forward and backward)
    size_t w_status, w_chunk_counts, w_chunk_base, w_wrt, w_offp;
    size_t w_ringX, w_ringXs, w_ringH, w_ringHs, w_ringY, ring_bytes;   // forward
    size_t w_Xs, w_Gin, w_da, w_db, w_hw, w_dXs, w_dwpart, w_dlogits, w_dwr_part;   // backward
    size_t workspace_bytes;
};

__device__ __forceinline__ float bf2f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ bf16 f2bf(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ld_v4(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ void st_v4(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

}  // namespace moe
