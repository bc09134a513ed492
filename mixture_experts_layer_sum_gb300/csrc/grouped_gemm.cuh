// Arguments of the persistent tcgen05 grouped GEMM (grouped_gemm.cu).
#pragma once
#include "moe_common.cuh"

namespace moe {

enum GemmOp { OP_FWD1 = 0, OP_FWD2 = 1, OP_BWD2 = 2, OP_BWD1 = 3, OP_WG2 = 4, OP_WG13 = 5 };

// Row spaces: "padded rows" are the expert-sorted routed rows where every
// (macrobatch, expert) run starts at offp[m*E+e] and is padded with zero rows
// to a multiple of 128. Ring buffers hold the rows of one macrobatch:
// ring row = padded row - offp[m*E] + ring_base.
struct GemmArgs {
    CUtensorMap a0, a1, b0, b1;   // TMA maps (bf16, 128-byte swizzle, 64-element inner box)
    CUtensorMap om0, om1, om2;    // output maps for TMA stores: fp32 weight gradients (32 x 32,
                                  // 128B swizzle) or bf16 row outputs (32 x 32, no swizzle)
    int tma_store;                // 1: bf16 variants store epilogue tiles through shared memory + TMA
    const int *offp;              // [nM*E + 1] padded run starts
    int E, nM, m;                 // experts, macrobatches, macrobatch of a grouped-M launch
    int H, F;
    int N, K, Mw;                 // output columns, contraction length (grouped-M), rows of dW (grouped-K)
    int a_ring;                   // A rows are ring rows
    int o_ring;                   // FWD2 output rows are ring rows
    int ring_base;
    bf16 *o0, *o1, *o2;           // bf16 outputs (see each op)
    float *of0, *of1;             // fp32 outputs
    const bf16 *in0, *in1;        // BWD2: saved a, b (2 KB blocks, blk32_offset); FWD1 writes o0, o1 so
    const int *row_slot;          // BWD2: slot of each padded row (-1 = padding)
    const float *wslot;           // BWD2: router weight of each slot
    int accumulate;               // WG ops: add into the fp32 outputs
    // MXFP8 variant: scale atoms of A (a0, a1) and B (b0, b1) operands, the
    // K extent of the stored operand matrices, and quantised epilogue outputs
    const uint8_t *sfa0, *sfa1, *sfb0, *sfb1;
    int kstore;
    uint8_t *q0, *q1, *qs0, *qs1;  // FWD1: h codes/scales (ring); BWD2: da, db codes/scales
    // BWD2, MXFP8: da, db and h.w quantised along the padded rows ([F][tR] codes + scale atoms,
    // 32-row blocks), the weight gradients' operands
    uint8_t *tq[3], *tqs[3];
    int tR;
    // routed slots (T * k): a row's slot in row_slot lies in [-1, nslots); one outside raises
    // MOE_ERR_INTERNAL in the status word and the row is treated as padding
    int nslots;
    // FWD1 with the dispatch fused in (fused = 1): warps 6-9 of every CTA
    // claim 4-row chunks of the macrobatch from a counter, gather them into the
    // ring (bf16, or MXFP8 along H) and add the rows to ready[j] of their
    // minibatch; the TMA producer acquires ready[j] == rows of minibatch j
    // before it loads a tile of it. ready[0..ready_slots) and the claim counter
    // ready[ready_slots] are zeroed before every launch.
    int fused;
    int x_global;                 // bf16: gathered rows go to their global padded row (saved context)
    const bf16 *xsrc;
    bf16 *ringx;
    uint8_t *ringxq, *ringxs;
    int *ready;
    int ready_slots;
    int mb_rows, k;
    // MXFP8 CTA-pair variant: the scale arrays viewed as [bytes / 128][128] bytes (no swizzle),
    // so one 128 x 4 box is one 512-byte atom, loaded by TMA with completion on the pair
    // leader's barrier: A atoms (msa0, msa1) and B atoms (msb0, msb1)
    CUtensorMap msa0, msa1, msb0, msb1;
    // grouped-M ops over every macrobatch in one launch (tiles != nullptr): the M tiles come
    // from a list built on the device by launch_tile_lists, one int4 per tile, in expert-major
    // order (every run of expert 0, then of expert 1, ...) so that the CTAs running at one time
    // share one expert's weights; *tile_count holds the list's length. m stays 0 (only the ring
    // ops use it). 1-CTA kernels read 128-row tiles (first padded row, expert, end of the run,
    // 0), CTA pairs 256-row ones (first row of CTA 0's half, expert, first row of CTA 1's half
    // or -1, 0): two 128-row chunks of one expert, possibly from different runs.
    const int4 *tiles;
    const int *tile_count;
    int *status;
    unsigned long long budget_ns;
};

// pair = true: CTA-pair variant with 256-row tiles (cta_group::2); the B maps of the
// K-major ops then need 128-row boxes (bf16 and MXFP8), MXFP8 also the atom maps above.
cudaError_t launch_grouped_gemm(int op, const GemmArgs &g, int grid, cudaStream_t stream, bool fp8 = false,
                                bool pair = false);

// Persistent forward over every macrobatch (one launch of CTA pairs): the fused dispatch
// (gather warps), GEMM1 + SwiGLU and GEMM2 tiles, and the combine, handed on by device
// counters. Tiles come from a device-built list, macrobatch by macrobatch: GEMM1 tiles of m
// (expert, pair m-tile, n-tile), then GEMM2 tiles of m. One macrobatch is in the ring (h, Y
// rows; x rows too in MXFP8), so a tile that writes ring rows of m waits until the readers of
// m - 1 are done with them.
enum MegaCounter { MEGA_G1_READ = 0, MEGA_G2_READ, MEGA_Y_DONE, MEGA_COMBINED, MEGA_COMBINE_CLAIM, MEGA_NCNT = 8 };
struct MegaArgs {
    GemmArgs g1, g2;              // GEMM1 (fused dispatch) and GEMM2 of the forward (their m is unused)
    const int4 *tiles;            // (first padded row, expert | n-tile << 8 | op << 24, run end, macrobatch)
    const int *tile_count;        // [0]: tiles in the list
    const int *meta;              // [nM][4]: GEMM1 pair tiles, GEMM2 pair tiles, 4 x GEMM2 CTA tiles
                                  //          with rows (one per epilogue warp), combine items
    // hready: per 128-row block, one count per epilogue warp and GEMM1 n-tile (4 F / 128 when full)
    int *cnt;                     // [nM][MEGA_NCNT] counters (zeroed before the launch)
    int *hready;                  // [padded rows / 128]: GEMM1 n-tiles that stored h of the block
    const int32_t *slot_row;      // combine: padded row of each slot
    const float *w;               // combine: router weights [T, k]
    bf16 *out;                    // [T, H]
    int T, Mb, ready_stride;      // tokens, macrobatch tokens, ready ints per macrobatch
};

// Builds the persistent forward's tile list and per-macrobatch counts (one block per
// macrobatch). Entries: at most (rows_pad_max / 256 + nM * E) * (F / 128 + H / 256).
cudaError_t launch_mega_list(const int *offp, int E, int nM, int F, int H, int T, int Mb, int4 *list, int *meta,
                             int *count, cudaStream_t stream);
cudaError_t launch_fwd_mega(const MegaArgs &a, int grid, cudaStream_t stream, bool fp8);

// Writes the M-tile lists of every (macrobatch, expert) run of padded rows, expert-major:
// list128 with the 128-row chunks of each run (1-CTA kernels), list256 with those chunks
// taken two at a time per expert (CTA pairs; an expert's last pair may have one chunk).
// counts[0], counts[1] = their lengths. Each list needs at most offp[nM*E] / 128 + nM*E
// entries; E <= kMaxExperts.
cudaError_t launch_tile_lists(const int *offp, int E, int nM, int4 *list128, int4 *list256, int *counts,
                              cudaStream_t stream);

}  // namespace moe
