// MXFP8 quantisers (article "O MoK do Cursor ...", section 02: MXFP8 activation
// quantisation fused into dispatch, grouped GEMM and SwiGLU, with no separate
// quantisation pass over HBM for the dispatched rows).
//
//   mx_rows_kernel       bf16 rows -> E4M3 rows + E8M0 scales along the row.
//                        Gather mode is the quantising dispatch: destination
//                        row r takes token row_slot[r] / k of the source (zero
//                        for padding rows), so x is read once and written once
//                        in MXFP8. Identity mode quantises a matrix in place
//                        order (weights along their K, gathered dY rows).
//   mx_transpose_kernel  bf16 [R][C] -> E4M3 [C][R] + scales along R: operands
//                        whose contraction axis is the row axis (weights for the
//                        other GEMM orientation, token-axis operands of the
//                        weight gradients).
#include "mx_quant.cuh"

namespace moe {

// Warp per destination row; lane handles 8 consecutive elements (one 16-byte
// load), a quad of lanes forms one 32-element block.
__global__ void __launch_bounds__(256) mx_rows_kernel(MxRowsArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    const int lane = threadIdx.x % 32;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int nw = gridDim.x * blockDim.x / 32;
    int r0 = 0, r1 = a.nrows;
    if (a.offp) { r0 = a.offp[a.beg]; r1 = a.offp[a.end]; }
    const int vecs = a.C / 8;
    for (int r = r0 + gw; r < r1; r += nw) {
        const bf16 *src = nullptr;
        if (a.row_slot) {
            const int slot = a.row_slot[r];
            if (slot >= 0) src = a.src + (size_t)(slot / a.k) * a.C;
        } else {
            src = a.src + (size_t)r * a.C;
        }
        const size_t drow = (size_t)(a.dst_row0 + r - r0);
        uint8_t *dst = a.codes + drow * a.C;
        for (int v = lane; v < vecs; v += 32) {
            float f[8];
            if (src) {
                const uint4 q = ld_nc_v4(src + v * 8);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) { f[2 * i] = bf16lo(w[i]); f[2 * i + 1] = bf16hi(w[i]); }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = 0.0f;
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int s = mx_exponent(amax);
            const float inv = mx_inv_scale(s);
            uint2 c;
            c.x = cvt_e4m3x4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
            c.y = cvt_e4m3x4(f[4] * inv, f[5] * inv, f[6] * inv, f[7] * inv);
            *reinterpret_cast<uint2 *>(dst + v * 8) = c;
            if ((lane & 3) == 0) a.scales[mx_sf_offset(drow, (size_t)v * 8, a.C)] = (uint8_t)(s + 127);
        }
    }
}

cudaError_t launch_mx_rows(const MxRowsArgs &a, int max_rows, int num_sms, cudaStream_t s) {
    if (max_rows <= 0) return cudaSuccess;
    const int blocks = min(ceil_div(max_rows, 8), num_sms * 8);
    cudaError_t e = launch_pdl(mx_rows_kernel, dim3(blocks), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Block: 128 input rows x 64 input columns of one batch item, staged in shared
// memory; thread (c, b) quantises input rows [32b, 32b+32) of column c into one
// 32-byte run of output row c.
__global__ void __launch_bounds__(256) mx_transpose_kernel(MxTransposeArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ __align__(16) bf16 tile[128][64 + 8];
    const int c0 = blockIdx.x * 64, rb0 = blockIdx.y * 128;
    const size_t bi = blockIdx.z;
    const int r_limit = a.r_limit_ptr ? *a.r_limit_ptr : a.R;
    if (rb0 >= r_limit) return;
    const bf16 *src = a.src + bi * (size_t)a.R * a.C;
    for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
        const int rr = i / 8, v = i % 8;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (rb0 + rr < r_limit) {
            if (a.row_slot) {
                const int slot = a.row_slot[rb0 + rr];
                if (slot >= 0) q = ld_nc_v4(src + (size_t)(slot / a.k) * a.C + c0 + v * 8);
            } else {
                q = ld_nc_v4(src + (size_t)(rb0 + rr) * a.C + c0 + v * 8);
            }
        }
        *reinterpret_cast<uint4 *>(&tile[rr][v * 8]) = q;
    }
    __syncthreads();
    const int c = threadIdx.x % 64, b = threadIdx.x / 64;
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = bf2f(tile[b * 32 + i][c]);
    uint32_t codes[8];
    const uint32_t sbyte = mx_quant32(f, codes);
    const size_t orow = (size_t)(c0 + c);
    uint8_t *dst = a.codes + bi * (size_t)a.C * a.R + orow * a.R + rb0 + b * 32;
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
    a.scales[bi * ((size_t)a.C * a.R / kMxBlock) + mx_sf_offset(orow, (size_t)rb0 + b * 32, a.R)] = (uint8_t)sbyte;
}

cudaError_t launch_mx_transpose(const MxTransposeArgs &a, int batch, cudaStream_t s) {
    if (a.R <= 0 || batch <= 0) return cudaSuccess;
    dim3 grid(a.C / 64, ceil_div(a.R, 128), batch);
    cudaError_t e = launch_pdl(mx_transpose_kernel, grid, dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
