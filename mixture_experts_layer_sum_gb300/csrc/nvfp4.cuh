// NVFP4 expert weights for the decode forward (nvfp4.cu): E2M1 elements with one E4M3 scale
// per 16 elements along the contraction axis and a power-of-two FP32 scale per expert matrix.
#pragma once
#include "moe_common.cuh"

namespace moe {

constexpr int kNvBlock = 16;

// Storage of one quantised matrix set (W1, W3 or W2 of every expert), quantised along its
// contraction axis K and tiled for the decode kernel's 128-column x 64-K weight tiles:
//   codes  [E][N/128][K/64][128 rows][32 B]  (row = weight column; byte j holds K elements 2j
//                                             (low nibble) and 2j + 1 (high nibble))
//   scales [E][N/128][K/64][128 rows][4 B]   (byte b: E4M3 scale of K elements 16b .. 16b + 15)
// so one tile is 4 KB of codes and 512 B of scales, each contiguous.
struct NvMatrix {
    size_t codes, scales;   // byte offsets inside the NVFP4 weight buffer
    int K, N;               // contraction length, columns
};
struct NvLayout {
    NvMatrix m[3];          // W1 (K = H, N = F), W3 (K = H, N = F), W2 (K = F, N = H)
    size_t gscale;          // float [3][E]: power-of-two matrix scales
    size_t amax;            // unsigned [3][E]: scratch of the quantiser (matrix maxima as float bits)
    size_t bytes;
};
NvLayout nv_layout(int E, int H, int F);

// Quantises the bf16 masters W1, W3 [E][H][F] and W2 [E][F][H] into the NVFP4 buffer (base
// 1024-byte aligned): a matrix maximum pass, then one block per 128 x 64 tile.
cudaError_t launch_nv_quantize(const bf16 *W1, const bf16 *W3, const bf16 *W2, uint8_t *base, const NvLayout &L,
                               int E, int H, int F, int num_sms, cudaStream_t s);

}  // namespace moe
