// MXFP8 quantisers (article "O MoK do Cursor ...", section 02: MXFP8 activation
// quantisation fused into dispatch, grouped GEMM and SwiGLU, with no separate
// quantisation pass over HBM for the dispatched rows; the forward's quantising
// dispatch itself runs inside GEMM1).
//
//   mx_rows_kernel       bf16 rows -> E4M3 rows + E8M0 scales along the row
//                        (weight copies along their stored rows).
//   mx_transpose_kernel  bf16 [R][C] -> E4M3 [C][R] + scales along R: operands
//                        whose contraction axis is the row axis (weights for the
//                        other GEMM orientation, token-axis operands of the
//                        weight gradients, gathered straight from x and dout);
//                        optionally also the row-wise copy of the same rows
//                        (dY along H for the GEMM2 dgrad).
#include "mx_quant.cuh"

namespace moe {

// ---------------------------------------------------------------- helpers
// Halfwise max(|a|, |b|) of two bf16 pairs; the result's sign bits carry no
// magnitude (mask them with 0x7fff7fff at the end of a reduction).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Shared exponent from the 15-bit magnitude of a bf16 block maximum: the same
// rule as mx_exponent (smallest s with amax <= 448 * 2^s; 448 = 1.75 * 2^8, so
// one more when the mantissa exceeds 0.75), zero and subnormal maxima give -127.
// A finite or infinite bf16 maximum gives s <= 121.
__device__ __forceinline__ int mx_exponent_bf16(uint32_t m) {
    const int e = (int)(m >> 7);
    if (e == 0) return -127;
    const int s = e - 135 + ((m & 127u) > 96u ? 1 : 0);
    return s < -127 ? -127 : s;
}

// 2^-s as bf16 bits, s in [-127, 121] (a normal number).
__device__ __forceinline__ uint16_t mx_inv_bf16(int s) { return (uint16_t)((127 - s) << 7); }

// E4M3 codes of (lo(a), lo(b)) scaled by inv_lo and of (hi(a), hi(b)) scaled by
// inv_hi; the first element of each pair in the low byte. The mixed-precision
// FMA multiplies bf16 by a power of two exactly into fp32 (adding -0 keeps the
// sign of zero), then the pair is rounded to nearest even with saturation.
__device__ __forceinline__ void e4m3_pairs(uint32_t a, uint32_t b, uint16_t inv_lo, uint16_t inv_hi, uint16_t &clo,
                                           uint16_t &chi) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 fa, fb, ga, gb;\n\t"
        "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 fa, al, %4, 0f80000000;\n\tfma.rn.f32.bf16 fb, bl, %4, 0f80000000;\n\t"
        "fma.rn.f32.bf16 ga, ah, %5, 0f80000000;\n\tfma.rn.f32.bf16 gb, bh, %5, 0f80000000;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 %0, fb, fa;\n\tcvt.rn.satfinite.e4m3x2.f32 %1, gb, ga;\n\t}"
        : "=h"(clo), "=h"(chi)
        : "r"(a), "r"(b), "h"(inv_lo), "h"(inv_hi));
}

// E4M3 codes of the four bf16 of (w0, w1), in order, all scaled by inv.
__device__ __forceinline__ uint32_t e4m3x4_row(uint32_t w0, uint32_t w1, uint16_t inv) {
    uint32_t d;
    asm("{\n\t.reg .b16 a0, a1, b0, b1, c0, c1;\n\t.reg .f32 f0, f1, f2, f3;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.bf16 f0, a0, %3, 0f80000000;\n\tfma.rn.f32.bf16 f1, a1, %3, 0f80000000;\n\t"
        "fma.rn.f32.bf16 f2, b0, %3, 0f80000000;\n\tfma.rn.f32.bf16 f3, b1, %3, 0f80000000;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 c0, f1, f0;\n\tcvt.rn.satfinite.e4m3x2.f32 c1, f3, f2;\n\t"
        "mov.b32 %0, {c0, c1};\n\t}"
        : "=r"(d)
        : "r"(w0), "r"(w1), "h"(inv));
    return d;
}

// ---------------------------------------------------------------- rows
// Warp per destination row, in chunks of 1024 elements (32 blocks). The warp
// loads a chunk with coalesced 16-byte vectors (the next chunk's loads go out
// before the current one is quantised), passes it through a per-warp 2 KB
// buffer, and lane l then holds block l whole: its maximum, exponent and codes
// need no cross-lane step; codes leave as one 32-byte store per lane and the
// four scale bytes of lanes 4q..4q+3 (adjacent in the atom row) as one word.
constexpr int kRowsWarps = 8;

// Slot of 16-byte vector v of a chunk in the staging buffer: the XOR of bits
// 3.. into bits 0..2 keeps both the store pattern (lane l writes v = l + 32u)
// and the load pattern (lane l reads v = 4l + j) free of bank conflicts.
__device__ __forceinline__ int mx_stage_slot(int v) { return (v & ~7) | ((v ^ (v >> 3)) & 7); }

__global__ void __launch_bounds__(kRowsWarps * 32) mx_rows_kernel(MxRowsArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ __align__(16) uint4 stage[kRowsWarps][128];
    const int lane = threadIdx.x % 32, wib = threadIdx.x / 32;
    uint4 *wb = stage[wib];
    const int gw = blockIdx.x * kRowsWarps + wib, nw = gridDim.x * kRowsWarps;
    const int nchunk = (a.C + 1023) / 1024;
    for (int r = gw; r < a.nrows; r += nw) {
        const bf16 *src = a.src + (size_t)r * a.C;
        const size_t drow = (size_t)r;
        uint8_t *dst = a.codes + drow * a.C;
        uint4 q[4];
        auto load = [&](int ch) {
            const int e0 = ch * 1024, nvec = min(128, (a.C - e0) / 8);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = lane + 32 * u;
                q[u] = v < nvec ? ld_nc_v4(src + e0 + v * 8) : make_uint4(0, 0, 0, 0);
            }
        };
        load(0);
        for (int ch = 0; ch < nchunk; ++ch) {
            const int e0 = ch * 1024, nvec = min(128, (a.C - e0) / 8);
#pragma unroll
            for (int u = 0; u < 4; ++u) wb[mx_stage_slot(lane + 32 * u)] = q[u];
            __syncwarp();
            if (ch + 1 < nchunk) load(ch + 1);
            const bool active = lane * 4 < nvec;   // nvec % 32 == 0: whole quads in or out
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 t = active ? wb[mx_stage_slot(4 * lane + j)] : make_uint4(0, 0, 0, 0);
                w[4 * j] = t.x; w[4 * j + 1] = t.y; w[4 * j + 2] = t.z; w[4 * j + 3] = t.w;
            }
            __syncwarp();
            uint32_t m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = absmax_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
            for (int i = 0; i < 4; ++i) m[i] = absmax_bf16x2(m[2 * i], m[2 * i + 1]);
            m[0] = absmax_bf16x2(absmax_bf16x2(m[0], m[1]), absmax_bf16x2(m[2], m[3]));
            const uint32_t mag = max(m[0] & 0x7fffu, (m[0] >> 16) & 0x7fffu);
            const int sx = mx_exponent_bf16(mag);
            const uint16_t inv = mx_inv_bf16(sx);
            uint32_t c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = e4m3x4_row(w[2 * i], w[2 * i + 1], inv);
            if (active) st_global_32B(dst + e0 + 32 * lane, c);
            uint32_t sb = (uint32_t)(sx + 127);
            sb |= __shfl_down_sync(0xffffffffu, sb, 1) << 8;
            sb |= __shfl_down_sync(0xffffffffu, sb, 2) << 16;
            if (active && (lane & 3) == 0)
                *reinterpret_cast<uint32_t *>(a.scales + mx_sf_offset(drow, (size_t)(e0 + 32 * lane), a.C)) = sb;
        }
    }
}

cudaError_t launch_mx_rows(const MxRowsArgs &a, int max_rows, int num_sms, cudaStream_t s) {
    if (max_rows <= 0) return cudaSuccess;
    const int blocks = min(ceil_div(max_rows, kRowsWarps), num_sms * 8);
    cudaError_t e = launch_pdl(mx_rows_kernel, dim3(blocks), dim3(kRowsWarps * 32), 0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------- transpose
// Block: 128 input rows x 128 input columns of one batch item, staged in shared
// memory with coalesced 16-byte loads (gathered rows resolve their token index
// once, into shared memory). Warp w then takes input rows 32w..32w+31 (one
// 32-element block of each output row) and lane l input columns 4l..4l+3 with
// 8-byte shared loads: two packed maxima over 32 rows give the four column
// maxima; each output row gets one 32-byte store of codes. The block's 512
// scale bytes are exactly one atom (output rows c0..c0+127, K block rb0/128):
// built in shared memory, stored as 32 x 16 bytes.
constexpr int kMxtRows = 128, kMxtCols = 128;
__global__ void __launch_bounds__(128) mx_transpose_kernel(MxTransposeArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ __align__(16) bf16 tile[kMxtRows][kMxtCols + 8];
    __shared__ int tok[kMxtRows];
    __shared__ __align__(16) uint8_t atom[512];
    const size_t bi = blockIdx.z;
    int cb = blockIdx.x, rb0 = blockIdx.y * kMxtRows, r_limit;
    if (a.offp) {
        const int ncb = a.C / kMxtCols, yb = blockIdx.x / ncb;
        cb = blockIdx.x - yb * ncb;
        const int per_m = a.ilv_E * a.ilv_jb;
        const int m = yb / per_m, rem = yb - m * per_m, j = rem / a.ilv_E, e = rem - j * a.ilv_E;
        const int seg = m * a.ilv_E + e;
        rb0 = a.offp[seg] + j * kMxtRows;
        r_limit = a.offp[seg + 1];
    } else {
        r_limit = a.r_limit_ptr ? *a.r_limit_ptr : a.R;
    }
    if (rb0 >= r_limit) return;
    const int c0 = cb * kMxtCols;
    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const bf16 *src = a.src + bi * (size_t)a.R * a.C;
    {
        const int r = rb0 + t;
        int tk = -1;
        if (r < r_limit) {
            if (a.row_slot) {
                const int slot = a.row_slot[r];
                if (slot >= a.nslots || slot < -1) raise_status(a.status, kStatusInternal);
                else if (slot >= 0) tk = slot / a.k;
            } else {
                tk = r;
            }
        }
        tok[t] = tk;
    }
    __syncthreads();
    // 128 rows x 16 vectors of 16 B: 16 loads per thread, issued together
    uint4 q[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int i = t + 128 * j, rr = i >> 4, v = i & 15;
        const int tk = tok[rr];
        q[j] = tk >= 0 ? ld_nc_v4(src + (size_t)tk * a.C + c0 + v * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int i = t + 128 * j, rr = i >> 4, v = i & 15;
        *reinterpret_cast<uint4 *>(&tile[rr][v * 8]) = q[j];
    }
    __syncthreads();
    uint2 d[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) d[r] = *reinterpret_cast<const uint2 *>(&tile[warp * 32 + r][lane * 4]);
    uint32_t mx[16], my[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        mx[r] = absmax_bf16x2(d[2 * r].x, d[2 * r + 1].x);
        my[r] = absmax_bf16x2(d[2 * r].y, d[2 * r + 1].y);
    }
#pragma unroll
    for (int n = 8; n >= 1; n /= 2)
#pragma unroll
        for (int r = 0; r < n; ++r) {
            mx[r] = absmax_bf16x2(mx[r], mx[r + n]);
            my[r] = absmax_bf16x2(my[r], my[r + n]);
        }
    const uint32_t mag[4] = {mx[0] & 0x7fffu, (mx[0] >> 16) & 0x7fffu, my[0] & 0x7fffu, (my[0] >> 16) & 0x7fffu};
    int sx[4];
    uint16_t inv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) { sx[i] = mx_exponent_bf16(mag[i]); inv[i] = mx_inv_bf16(sx[i]); }
    uint8_t *dst = a.codes + bi * (size_t)a.C * a.R + (size_t)(c0 + lane * 4) * a.R + rb0 + warp * 32;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        uint32_t clo[8], chi[8];
#pragma unroll
        for (int r = 0; r < 32; r += 4) {
            uint16_t l01, h01, l23, h23;
            const uint32_t a0 = p ? d[r].y : d[r].x, a1 = p ? d[r + 1].y : d[r + 1].x;
            const uint32_t a2 = p ? d[r + 2].y : d[r + 2].x, a3 = p ? d[r + 3].y : d[r + 3].x;
            e4m3_pairs(a0, a1, inv[2 * p], inv[2 * p + 1], l01, h01);
            e4m3_pairs(a2, a3, inv[2 * p], inv[2 * p + 1], l23, h23);
            clo[r / 4] = (uint32_t)l01 | ((uint32_t)l23 << 16);
            chi[r / 4] = (uint32_t)h01 | ((uint32_t)h23 << 16);
        }
        st_global_32B(dst + (size_t)(2 * p) * a.R, clo);
        st_global_32B(dst + (size_t)(2 * p + 1) * a.R, chi);
    }
    // scale byte of output row c (local), K block warp: atom byte (c%32)*16 + ((c/32)%4)*4 + warp
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = lane * 4 + i;
        atom[(c & 31) * 16 + ((c >> 5) & 3) * 4 + warp] = (uint8_t)(sx[i] + 127);
    }
    if (a.rcodes && rb0 + t < r_limit) {
        // row-wise copy: thread t quantises tile row t along C (four 32-column blocks)
        // from the same staged tile; 16-byte shared loads at the 272-byte row stride
        // hit distinct banks within each quarter warp
        const size_t grow = (size_t)(rb0 + t);
        uint8_t *rdst = a.rcodes + grow * a.C + c0;
        uint32_t sw = 0;
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 q = *reinterpret_cast<const uint4 *>(&tile[t][b * 32 + j * 8]);
                w[4 * j] = q.x; w[4 * j + 1] = q.y; w[4 * j + 2] = q.z; w[4 * j + 3] = q.w;
            }
            uint32_t m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = absmax_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
            for (int i = 0; i < 4; ++i) m[i] = absmax_bf16x2(m[2 * i], m[2 * i + 1]);
            m[0] = absmax_bf16x2(absmax_bf16x2(m[0], m[1]), absmax_bf16x2(m[2], m[3]));
            const int rs = mx_exponent_bf16(max(m[0] & 0x7fffu, (m[0] >> 16) & 0x7fffu));
            const uint16_t rinv = mx_inv_bf16(rs);
            uint32_t cw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) cw[i] = e4m3x4_row(w[2 * i], w[2 * i + 1], rinv);
            st_global_32B(rdst + b * 32, cw);
            sw |= (uint32_t)(rs + 127) << (8 * b);
        }
        // the four blocks' scale bytes are adjacent in the atom row
        *reinterpret_cast<uint32_t *>(a.rscales + mx_sf_offset(grow, (size_t)c0, a.C)) = sw;
    }
    __syncthreads();
    if (t < 32) {
        uint8_t *sdst = a.scales + bi * ((size_t)a.C * a.R / kMxBlock) +
                        ((size_t)(c0 / 128) * (size_t)(a.R / 128) + (size_t)(rb0 / 128)) * 512;
        reinterpret_cast<uint4 *>(sdst)[t] = reinterpret_cast<const uint4 *>(atom)[t];
    }
}

cudaError_t launch_mx_transpose(const MxTransposeArgs &a, int batch, cudaStream_t s) {
    if (a.R <= 0 || batch <= 0) return cudaSuccess;
    if (a.R % kMxtRows || a.C % kMxtCols) return cudaErrorInvalidValue;
    dim3 grid(a.C / kMxtCols, a.R / kMxtRows, batch);
    if (a.rcodes && batch != 1) return cudaErrorInvalidValue;
    if (a.offp) {
        if (batch != 1 || a.ilv_E <= 0 || a.ilv_nseg % a.ilv_E) return cudaErrorInvalidValue;
        const long long nb = (long long)(a.C / kMxtCols) * a.ilv_nseg * a.ilv_jb;
        if (nb <= 0) return cudaSuccess;
        if (nb > 0x7fffffffLL) return cudaErrorInvalidValue;
        grid = dim3((unsigned)nb, 1, 1);
    }
    cudaError_t e = launch_pdl(mx_transpose_kernel, grid, dim3(128), 0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
