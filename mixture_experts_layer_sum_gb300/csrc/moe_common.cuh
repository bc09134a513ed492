// Shared definitions of the MoE layer kernels: sizes, buffer layouts inside
// the caller's workspace / saved buffers, and small device helpers.
#pragma once
#include <utility>
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx_sm103.cuh"

namespace moe {

constexpr int kMaxExperts = 64;
constexpr int kRowPad = 128;          // each (macrobatch, expert) run of sorted rows is padded to this
constexpr int kSchedChunk = 256;      // routed slots per schedule block
constexpr int kSchedWarps = 8;       // one 32-slot group per warp: every id load of a chunk in flight at once
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
    int ring_halves;        // 1 (the ring holds one macrobatch)
    int nchunks;            // schedule blocks
    int chunks_per_mb;
    int minibatch_rows;
    int num_sms;
    int dwr_splits;         // token splits of the router-weight gradient
    // saved buffer
    size_t s_ids, s_w, s_probs, s_counts, s_offsets, s_offp, s_s2sorted, s_sorted2s, s_slot_row,
        s_row_slot, s_a, s_b, s_xs, saved_bytes;
    // bf16 with one macrobatch: the forward's dispatched X rows live in the saved
    // buffer (s_xs) and the backward's weight gradient reads them there (no replay)
    bool keep_x;
    // workspace (header first, then a region shared by forward and backward)
    size_t w_status, w_chunk_counts, w_chunk_base, w_wrt, w_offp, w_ready;
    size_t w_tiles128, w_tiles256, w_tile_counts;   // backward M-tile lists (several macrobatches)
    size_t w_decode;        // decode forward: work-item counter + per-expert h counters
    size_t w_mega_list, w_mega_meta, w_mega_count, w_mega_cnt, w_mega_hready;   // persistent forward
    size_t mega_list_max, mega_zero_bytes;   // list entries; bytes of counters zeroed per call
    bool decode;            // bf16 forward of few tokens through the decode kernel
    int tile_list_max;                              // entries each list can hold
    int mb_rows;            // minibatch rows used by the fused dispatch (multiple of 128)
    size_t w_ringX, w_ringXs, w_ringH, w_ringHs, w_ringY, ring_bytes;   // forward
    size_t w_Gin, w_da, w_db, w_hw, w_dXs, w_dwpart, w_dlogits, w_dwr_part;   // backward
    // backward, MXFP8 only: quantised operands (codes, scale atoms)
    size_t w_Ginq, w_Ginq_s, w_daq, w_daq_s, w_dbq, w_dbq_s;       // along H / F (row-wise)
    size_t w_GinT, w_GinT_s, w_XsT, w_XsT_s, w_hwT, w_hwT_s, w_daT, w_daT_s, w_dbT, w_dbT_s;   // along rows
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
// Saved a, b (GEMM1 outputs read back by the GEMM2 dgrad epilogue) are stored in
// 32 x 32 blocks of 2 KB: block (row / 32, col / 32) of a [rows][C] matrix starts at
// element ((row / 32) * (C / 32) + col / 32) * 1024; inside it, element (r, c) sits at
// ((c / 8) * 32 + r) * 8 + c % 8, so the 16-byte vector j of the 32 rows of a block is
// 512 contiguous bytes and a warp (lane = row) reads or writes it in one instruction.
__host__ __device__ __forceinline__ size_t blk32_offset(int row, int col, int C) {
    return ((size_t)(row >> 5) * (size_t)(C >> 5) + (size_t)(col >> 5)) * 1024;
}

// Programmatic dependent launch: every kernel of the layer is launched with
// programmatic stream serialisation, so it may start while its predecessor on the
// stream finishes. pdl_wait() (every thread, before the first read of anything an
// earlier kernel wrote) blocks until the predecessor grid has completed and its memory
// is visible; pdl_trigger() lets the successor launch (it then waits in its own
// pdl_wait). Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_v4(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ void st_v4(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------- MXFP8
// E4M3 element codes with one E8M0 scale byte per 32 consecutive elements of a
// row along the contraction axis K. Scales are stored in 512-byte atoms that
// cover 128 rows x 128 elements (4 blocks): atom (r/128, k/128) in row-major
// order, byte (r%32)*16 + ((r/32)%4)*4 + (k/32)%4 inside it. This is the order
// tcgen05.cp.32x128b.warpx4 moves into tensor memory for the block-scaled MMA.
__host__ __device__ __forceinline__ size_t mx_sf_offset(size_t r, size_t k, size_t K) {
    return ((r >> 7) * (K >> 7) + (k >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + ((k >> 5) & 3);
}

// Shared exponent of a block: the smallest s with amax <= 448 * 2^s (the
// block's largest element never saturates), clamped to [-127, 127]; zero and
// subnormal maxima give -127.
__device__ __forceinline__ int mx_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int e = (int)((b >> 23) & 0xFF);
    if (e == 0) return -127;
    const int s = e - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// 2^-s for s in [-127, 126] (finite fp32 maxima give s <= 120)
__device__ __forceinline__ float mx_inv_scale(int s) { return __uint_as_float((uint32_t)(127 - s) << 23); }

// four floats -> four E4M3 bytes (round to nearest even, saturate finite), element 0 in the low byte
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(lo) : "f"(a), "f"(b));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(hi) : "f"(c), "f"(d));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// One 32-byte global store (a whole sector); p 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void *p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Quantises 32 values held by one thread: 8 words of codes, returns the scale byte.
__device__ __forceinline__ uint32_t mx_quant32(const float (&v)[32], uint32_t (&codes)[8]) {
    // block maximum as a pairwise tree (depth 5, not a chain of 32 dependent steps)
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
#pragma unroll
    for (int n = 8; n >= 1; n /= 2)
#pragma unroll
        for (int i = 0; i < n; ++i) m[i] = fmaxf(m[i], m[i + n]);
    const float amax = m[0];
    const int s = mx_exponent(amax);
    const float inv = mx_inv_scale(s);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        codes[i] = cvt_e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    return (uint32_t)(s + 127);
}

// Launch with programmatic stream serialisation (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
