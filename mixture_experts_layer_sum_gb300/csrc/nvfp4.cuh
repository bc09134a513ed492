// NVFP4 expert weights for the decode forward (nvfp4.cu): E2M1 elements with one E4M3 scale
// per 16 elements along the contraction axis and a power-of-two FP32 scale per expert matrix.
#pragma once
#include "moe_common.cuh"

namespace moe {

constexpr int kNvBlock = 16;

// Storage of the quantised W1, W3 (contraction axis K = H, N = F columns) and W2 (K = F,
// N = H), in the order the decode kernel streams them. A tile covers 128 weight columns and 64 K
// elements, kNvTile bytes:
//   codes  [128 rows][32 B]  (row = weight column; byte j holds K elements 2j (low nibble) and
//                             2j + 1 (high nibble))
//   scales [128 rows][4 B]   (byte b: E4M3 scale of K elements 16b .. 16b + 15)
// A decode stage covers 128 K elements, and each stage's tiles are one contiguous block:
//   W1 and W3: [E][F/128][H/128][W1 tile k, W1 tile k + 64, W3 tile k, W3 tile k + 64]
//   W2:        [E][H/128][F/128][tile k, tile k + 64]
constexpr uint32_t kNvTile = 4096 + 512;
struct NvLayout {
    size_t w13, w2;         // byte offsets inside the NVFP4 weight buffer
    size_t gscale;          // float [3][E]: power-of-two matrix scales (W1, W3, W2)
    size_t amax;            // unsigned [3][E]: scratch of the quantiser (matrix maxima as float bits)
    size_t bytes;
};
// byte offset of tile (columns 128 nt.., K elements 64 kt..) of matrix mat (0 W1, 1 W3, 2 W2) of expert e
__host__ __device__ inline size_t nv_tile_offset(const NvLayout &L, int mat, int e, int nt, int kt, int H, int F) {
    if (mat < 2)
        return L.w13 + ((((size_t)e * (F / 128) + nt) * (H / 128) + kt / 2) * 4 + mat * 2 + (kt & 1)) * kNvTile;
    return L.w2 + ((((size_t)e * (H / 128) + nt) * (F / 128) + kt / 2) * 2 + (kt & 1)) * kNvTile;
}
NvLayout nv_layout(int E, int H, int F);

// Quantises the bf16 masters W1, W3 [E][H][F] and W2 [E][F][H] into the NVFP4 buffer (base
// 1024-byte aligned): a matrix maximum pass, then one block per 128 x 64 tile.
cudaError_t launch_nv_quantize(const bf16 *W1, const bf16 *W3, const bf16 *W2, uint8_t *base, const NvLayout &L,
                               int E, int H, int F, int num_sms, cudaStream_t s);

}  // namespace moe
