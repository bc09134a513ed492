// NVFP4 copies of the expert weights (a weight-update step, like the MXFP8 copies): the
// format is E2M1 elements, one E4M3 scale per 16 elements along the contraction axis and a
// power-of-two FP32 scale per expert matrix (the smallest g with amax <= 448 * 6 * g, so every
// block scale fits E4M3 and a dequantised weight e2m1 * scale * g is exact in bf16). A block
// scale is the E4M3 value nearest to amax_block / (6 g); an element is the E2M1 value nearest
// (ties to even) to v / (scale * g), saturating at 6 (Cursor's NVFP4 kernels are prior work the
// pages name in "Por que a camada MoE virou o gargalo", noticiai.com.br; they give no format
// details, so this is the plain NVFP4 one). Both roundings use the hardware conversions
// (cvt.rn.satfinite to E4M3 and to E2M1); the quotients they round are IEEE fp32 divisions.
#include "nvfp4.cuh"

namespace moe {

NvLayout nv_layout(int E, int H, int F) {
    NvLayout L{};
    const size_t tiles = (size_t)E * (H / 64) * (F / 128);   // tiles of W1 (or W3, or W2) over all experts
    size_t o = 0;
    L.w13 = o;
    o = align_up(o + 2 * tiles * kNvTile, 1024);
    L.w2 = o;
    o = align_up(o + tiles * kNvTile, 1024);
    L.gscale = o;
    o = align_up(o + 4 * 3 * (size_t)E, 1024);
    L.amax = o;
    o = align_up(o + 4 * 3 * (size_t)E, 1024);
    L.bytes = o;
    return L;
}

namespace {

struct NvSrc {
    const bf16 *w[3];
};

// maxima of |W| per (matrix, expert) as float bits (non-negative floats order like integers)
__global__ void __launch_bounds__(256) nv_amax_kernel(NvSrc src, unsigned *amax, int E, int H, int F) {
    pdl_wait();
    pdl_trigger();
    const int mat = blockIdx.z, e = blockIdx.y;
    const size_t n = (size_t)H * F;   // every matrix of an expert has H * F elements
    const uint4 *p = reinterpret_cast<const uint4 *>(src.w[mat] + (size_t)e * n);
    float m = 0.0f;
    for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < n / 8; v += (size_t)gridDim.x * blockDim.x) {
        const uint4 q = ld_nc_v4(p + v);
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16lo(w4[i])), fabsf(bf16hi(w4[i]))));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    if (threadIdx.x % 32 == 0) atomicMax(amax + mat * E + e, __float_as_uint(m));
}

// smallest power of two g with amax <= 2688 g (1 for zero)
__device__ __forceinline__ float nv_gscale(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    const float r = __fdiv_rn(amax, 2688.0f);
    const uint32_t b = __float_as_uint(r);
    const uint32_t pow2 = b & 0x7F800000u;          // r rounded down to a power of two (r is normal here)
    return (b & 0x007FFFFFu) ? __uint_as_float(pow2 + 0x00800000u) : __uint_as_float(pow2);
}

// value -> E4M3 byte (round to nearest even, saturating) and back
__device__ __forceinline__ uint32_t e4m3_byte(float x) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(h) : "f"(x), "f"(0.0f));
    return h & 0xFFu;
}
__device__ __forceinline__ float e4m3_value(uint32_t byte) {
    uint32_t h2;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(byte));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
// eight floats -> eight E2M1 codes (round to nearest even, saturating at 6); element 2i in the
// low nibble of byte i
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
    uint32_t r;
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// One block per (128-column x 64-K tile, expert, matrix). The tile is staged in shared memory
// [64 K][128 columns]; thread t quantises column t % 128, K blocks 2 (t / 128) and 2 (t / 128) + 1.
__global__ void __launch_bounds__(256) nv_quant_kernel(NvSrc src, uint8_t *base, NvLayout L, int E, int H, int F) {
    pdl_wait();
    pdl_trigger();
    __shared__ __align__(16) bf16 tile[64][128];
    const int mat = blockIdx.z, e = blockIdx.y;
    const int K = mat < 2 ? H : F, N = mat < 2 ? F : H;
    const int ktiles = K / 64;
    const int nt = blockIdx.x / ktiles, kt = blockIdx.x % ktiles;
    const bf16 *w = src.w[mat] + (size_t)e * K * N;
    // 64 rows x 256 B, coalesced 16-byte loads
    for (int i = threadIdx.x; i < 64 * 16; i += blockDim.x) {
        const int r = i / 16, c = i % 16;
        *reinterpret_cast<uint4 *>(&tile[r][c * 8]) = ld_nc_v4(w + (size_t)(kt * 64 + r) * N + nt * 128 + c * 8);
    }
    __syncthreads();
    const float amax = __uint_as_float(reinterpret_cast<const unsigned *>(base + L.amax)[mat * E + e]);
    const float g = nv_gscale(amax);
    const int col = threadIdx.x % 128, half = threadIdx.x / 128;
    uint8_t *t = base + nv_tile_offset(L, mat, e, nt, kt, H, F);
    uint32_t codes[4], sbytes = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int k0 = (2 * half + b) * kNvBlock;
        float v[16], am = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = __bfloat162float(tile[k0 + i][col]);
            am = fmaxf(am, fabsf(v[i]));
        }
        const uint32_t sb = e4m3_byte(__fdiv_rn(am, 6.0f * g));
        const float sg = e4m3_value(sb) * g;        // exact: E4M3 value times a power of two
        float q[2][8];
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i / 8][i % 8] = sg > 0.0f ? __fdiv_rn(v[i], sg) : 0.0f;
        codes[2 * b] = sg > 0.0f ? e2m1x8(q[0]) : 0u;
        codes[2 * b + 1] = sg > 0.0f ? e2m1x8(q[1]) : 0u;
        sbytes |= sb << (8 * b);
    }
    *reinterpret_cast<uint4 *>(t + col * 32 + half * 16) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
    *reinterpret_cast<uint16_t *>(t + 4096 + col * 4 + half * 2) = (uint16_t)sbytes;
    if (blockIdx.x == 0 && threadIdx.x == 0) reinterpret_cast<float *>(base + L.gscale)[mat * E + e] = g;
}

}  // namespace

cudaError_t launch_nv_quantize(const bf16 *W1, const bf16 *W3, const bf16 *W2, uint8_t *base, const NvLayout &L,
                               int E, int H, int F, int num_sms, cudaStream_t s) {
    NvSrc src{{W1, W3, W2}};
    cudaError_t e = cudaMemsetAsync(base + L.amax, 0, 4 * 3 * (size_t)E, s);
    if (e != cudaSuccess) return e;
    const int chunks = std::max(1, std::min(64, (num_sms * 4 + 3 * E - 1) / (3 * E)));
    e = launch_pdl(nv_amax_kernel, dim3(chunks, E, 3), dim3(256), 0, s, src, reinterpret_cast<unsigned *>(base + L.amax),
                   E, H, F);
    if (e != cudaSuccess) return e;
    // W1, W3 have (F/128)(H/64) tiles per expert, W2 (H/128)(F/64): the same count
    e = launch_pdl(nv_quant_kernel, dim3((F / 128) * (H / 64), E, 3), dim3(256), 0, s, src, base, L, E, H, F);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
