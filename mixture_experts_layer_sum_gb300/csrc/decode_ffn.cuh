// Decode-shaped expert FFN (decode_ffn.cu): the forward of a few tokens, where every expert
// holds at most 128 routed rows and the time goes to streaming the weights from HBM.
#pragma once
#include "moe_common.cuh"

namespace moe {

// Largest token count the decode kernel takes: a token picks an expert at most once, so no
// expert then holds more than this many routed rows (one 128-row N tile).
constexpr int kDecodeMaxTokens = 128;

struct DecodeArgs {
    CUtensorMap w1, w3;   // W1, W3 viewed MN-major: (64 columns, E*H rows, F/64 chunks), box (64, 64, 2)
    CUtensorMap w2;       // W2 viewed MN-major: (64 columns, E*F rows, H/64 chunks), box (64, 64, 2)
    CUtensorMap x;        // dispatched x rows [rows][H] bf16, box (64, 32), 128-byte swizzle
    CUtensorMap h;        // h rows [rows][F] bf16, box (64, 32), 128-byte swizzle
    int nb;               // ceil(T / 32): 32-row boxes the largest expert can need (<= 4)
    const int *offp;      // [E + 1] padded run starts (one macrobatch)
    const int *counts;    // [E] routed rows of each expert
    bf16 *a, *b;          // saved a = x W1, b = x W3 of every padded row (32 x 32 blocks, blk32_offset)
    bf16 *hrows;          // h rows [rows][F] (the same memory as map h)
    bf16 *y;              // expert outputs [rows][H]
    int *claim;           // work-item counter (zeroed before the launch)
    int *hdone;           // [E] GEMM1 epilogue warps finished per expert, 4 per item (zeroed before the launch)
    int E, H, F;
    int *status;
    unsigned long long budget_ns;
    // NVFP4 weights (launch_decode_nv): the nvfp4.cuh stages of W1 and W3 (offset nv_w13) and
    // of W2 (nv_w2) inside nvq, and the matrix scales
    const uint8_t *nvq;
    size_t nv_w13, nv_w2;
    const float *nv_g;    // [3][E]
};

cudaError_t launch_decode_ffn(const DecodeArgs &a, int num_sms, cudaStream_t s);
// The same forward with NVFP4 expert weights (maps w1, w3, w2 unused): compressed tiles stream
// from HBM and are expanded to bf16 in tensor memory, the MMA's A operand. Writes the h rows and
// the expert outputs only (an NVFP4 layer has no backward, so a and b are not saved).
cudaError_t launch_decode_nv(const DecodeArgs &a, int num_sms, cudaStream_t s);

}  // namespace moe
