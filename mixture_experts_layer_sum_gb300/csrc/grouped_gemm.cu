// Persistent grouped GEMMs of the expert FFN on tcgen05 tensor cores.
//
// One kernel template serves the six contractions of the layer (article
// "O MoK do Cursor ...", section 01: the grouped GEMM needs each expert's
// tokens grouped; section 02: SwiGLU and the quantisation sit in the GEMM's
// data path):
//   FWD1  [a|b] = X_e [W1_e|W3_e]; epilogue stores bf16 a, b and h = silu(a)*b
//   FWD2  Y = h_e W2_e
//   BWD2  G = dY_e W2_e^T; epilogue: dw partials <G,h>, dh = w G, SwiGLU
//         backward -> da, db, and hw = w*h for the W2 weight gradient
//   BWD1  dX = da W1_e^T + db W3_e^T            (contraction over 2F)
//   WG2   dW2_e = (w h)_e^T dY_e                (contraction over the expert's rows)
//   WG13  [dW1_e|dW3_e] = X_e^T [da_e|db_e]      (contraction over the expert's rows)
//
// Structure (one CTA per SM, 192 threads; 320 for GEMM1 with the fused dispatch):
//   warp 0     TMA producer: 128B-swizzled tiles of A (128 x 64) and B
//              (256 x 64) into a 4-stage shared-memory ring
//   warp 1     TMEM allocator and single-thread tcgen05.mma issuer
//              (M=128, N=256, K=16 per instruction); accumulators in TMEM,
//              double buffered (2 x 256 columns)
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, fused elementwise
//              work, stores to global memory
//   warps 6-9  (GEMM1 only) dispatch: gather/quantise token rows into the ring
//              minibatch by minibatch, publish per-minibatch ready row counts
// MXFP8 variant (FP8 = true): every operand is K-major E4M3 with E8M0 scale
// atoms (moe_common.cuh); a stage holds 128 elements of K (A 128x128 B,
// B 256x128 B) plus the 512-byte scale atoms of A and of both 128-row halves
// of B (1-D bulk copies). The MMA thread moves the atoms into tensor memory
// with tcgen05.cp.32x128b.warpx4 (4 columns per 128 rows) and issues
// tcgen05.mma.kind::mxf8f6f4.block_scale.scale_vec::1X (K=32) with the scale
// byte selected by k-block. The scale columns take TMEM columns 256..319, so
// the fp32 accumulator is single-buffered in this variant.
// Every mbarrier wait is bounded; when a wait gives up the status word is set
// and all roles leave their loops, drain their in-flight copies/MMAs and free
// TMEM before exiting.
#include <algorithm>
#include <atomic>

#include "grouped_gemm.cuh"
#include "combine_item.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KiB (bf16 128x64, or e4m3 128x128)
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t CHUNK_BYTES = 64 * 64 * 2;   // one 64x64 bf16 box, 8 KiB
constexpr uint32_t SF_BYTES = 3 * 512;          // scale atoms: A, B rows 0-127, B rows 128-255
constexpr uint32_t STAGE_STRIDE_FP8 = 51200;    // 48 KiB of tiles + atoms, 1 KiB aligned
constexpr int BK8 = 128;                        // K elements per stage, e4m3

template <bool FP8> __host__ __device__ constexpr uint32_t stage_stride() { return FP8 ? STAGE_STRIDE_FP8 : STAGE_BYTES; }
constexpr uint32_t P_STAGING_1 = 4 * 8192;   // epilogue staging of the 1-CTA bf16 kernel
// epilogue staging of the 1-CTA kernels: bf16 TMA-store buffers; the MXFP8 GEMM2 dgrad's
// token-axis transposition (eight warps x 2 KB); none otherwise
template <int OP, bool FP8> __host__ __device__ constexpr uint32_t staging_bytes() {
    return FP8 ? (OP == OP_BWD2 ? 8 * 2048 : 0) : P_STAGING_1;
}
template <bool FP8> __host__ __device__ constexpr int bk_elems() { return FP8 ? BK8 : BK; }

// D[tmem] (+)= A[smem] * B[smem], e4m3 x e4m3 with E8M0 block scales read from
// tensor memory (scale_vec::1X: one scale per 32 elements of K).
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 rows x 16 bytes of shared memory -> 4 TMEM columns, replicated to the four lane quarters
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled: e4m3 A/B, E8M0 scales, both K-major.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sf_id) {
    return ((uint32_t)sf_id << 4)               // B scale byte
           | ((uint32_t)(N >> 3) << 17)         // N / 8
           | (1u << 23)                         // scale format: E8M0
           | ((uint32_t)(M >> 4) << 24)         // M / 16
           | ((uint32_t)sf_id << 29);           // A scale byte
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}

// byte offset of the scale atom that covers (row, k) of a matrix with K columns
__device__ __forceinline__ size_t atom_at(int row, int k, int K) {
    return ((size_t)(row >> 7) * (size_t)(K >> 7) + (size_t)(k >> 7)) * 512;
}

template <int OP>
struct OpTraits;
template <> struct OpTraits<OP_FWD1> { static constexpr bool grouped_k = false, a_mn = false, b_mn = true; };
template <> struct OpTraits<OP_FWD2> { static constexpr bool grouped_k = false, a_mn = false, b_mn = true; };
template <> struct OpTraits<OP_BWD2> { static constexpr bool grouped_k = false, a_mn = false, b_mn = false; };
template <> struct OpTraits<OP_BWD1> { static constexpr bool grouped_k = false, a_mn = false, b_mn = false; };
template <> struct OpTraits<OP_WG2> { static constexpr bool grouped_k = true, a_mn = true, b_mn = true; };
template <> struct OpTraits<OP_WG13> { static constexpr bool grouped_k = true, a_mn = true, b_mn = true; };

struct TileInfo {
    int e, mt, nt;
    int g0;       // grouped-M: first global padded row of the tile
    int g1;       // grouped-M CTA pairs: first row of the second CTA's 128 rows, -1 if none
    int seg_end;  // grouped-M: end of the tile's (macrobatch, expert) run (pair lists: unused)
    int nk;       // number of BK blocks
};

template <int NS>
struct CtlT {
    uint64_t full[NS], empty[NS], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int nt;                       // tiles along N
    int list_tiles;               // grouped-M over all macrobatches: M tiles in the device list
    int mt_per_group;             // grouped-K: tiles along M (fixed)
    int prefix[kMaxExperts + 1];  // grouped-M: tile prefix over experts; grouped-K: unused
    int krows[kMaxExperts];       // grouped-K: padded rows of each expert (all macrobatches)
    int seg_start[kMaxExperts];   // grouped-M: first padded row of (m, e)
    int seg_end[kMaxExperts];     // grouped-M: end of the padded run of (m, e)
};
using SmemCtl = CtlT<STAGES>;

// TM = rows of an M tile: 128 (one CTA) or 256 (a CTA pair, 128 rows each)
template <int OP, class Ctl>
__device__ __forceinline__ int num_tiles(const Ctl &c, const GemmArgs &g) {
    if constexpr (OpTraits<OP>::grouped_k) return g.E * c.mt_per_group * c.nt;
    else return (g.tiles ? c.list_tiles : c.prefix[g.E]) * c.nt;
}

template <int OP, bool FP8, int TM = BM, class Ctl>
__device__ __forceinline__ TileInfo decode_tile(const Ctl &c, const GemmArgs &g, int t) {
    TileInfo ti;
    ti.nt = t % c.nt;
    int q = t / c.nt;
    if constexpr (OpTraits<OP>::grouped_k) {
        ti.mt = q % c.mt_per_group;
        ti.e = q / c.mt_per_group;
        ti.g0 = 0;
        ti.g1 = -1;
        ti.seg_end = 0;
        ti.nk = c.krows[ti.e] / bk_elems<FP8>();
    } else {
        if (g.tiles) {
            const int4 v = g.tiles[q];
            ti.e = v.y;
            ti.mt = 0;
            ti.g0 = v.x;
            if constexpr (TM == 2 * BM) {   // (CTA 0's rows, expert, CTA 1's rows or -1, 0)
                ti.g1 = v.z;
                ti.seg_end = 0x7fffffff;
            } else {                        // (first row, expert, run end, 0)
                ti.g1 = -1;
                ti.seg_end = v.z;
            }
        } else {
            int e = 0;
            while (c.prefix[e + 1] <= q) ++e;   // E <= 64
            ti.e = e;
            ti.mt = q - c.prefix[e];
            ti.g0 = c.seg_start[e] + ti.mt * TM;
            ti.seg_end = c.seg_end[e];
            ti.g1 = (TM == 2 * BM && ti.g0 + BM < ti.seg_end) ? ti.g0 + BM : -1;
        }
        ti.nk = g.K / bk_elems<FP8>();
    }
    return ti;
}

template <int OP, int TM, class Ctl>
__device__ void init_tile_table(Ctl &c, const GemmArgs &g) {
    if constexpr (OpTraits<OP>::grouped_k) {
        c.nt = (OP == OP_WG13) ? g.N / 128 : g.N / BN;
        c.mt_per_group = g.Mw / TM;
        for (int e = 0; e < g.E; ++e) {
            int rows = 0;
            for (int mm = 0; mm < g.nM; ++mm) rows += g.offp[mm * g.E + e + 1] - g.offp[mm * g.E + e];
            c.krows[e] = rows;
        }
    } else {
        c.nt = (OP == OP_FWD1) ? g.N / 128 : g.N / BN;
        if (g.tiles) {
            c.list_tiles = *g.tile_count;
            return;
        }
        c.prefix[0] = 0;
        for (int e = 0; e < g.E; ++e) {
            const int s0 = g.offp[g.m * g.E + e], s1 = g.offp[g.m * g.E + e + 1];
            c.seg_start[e] = s0;
            c.seg_end[e] = s1;
            c.prefix[e + 1] = c.prefix[e] + (s1 - s0 + TM - 1) / TM;
        }
    }
}

// Fused dispatch (FWD1): the gather warps pull token rows of the macrobatch into
// the ring (article "O MoK do Cursor ...", section 02: pull dispatch; the ring
// token buffer is advanced by GPU-side state, minibatch by minibatch, with no
// CPU in the loop). A warp claims the next 4 rows from a global counter
// (claims go in row order, so minibatches fill in order), gathers them and adds
// 4 to ready[j] of their minibatch with release semantics. Any subset of running
// CTAs can finish the gathering, so no CTA has to wait for another to start.
// stop_bar (optional): the warp stops claiming once phase 0 of this mbarrier has
// completed — the epilogue warps gather too until their CTA's first accumulator is ready.
// A row's slot from row_slot, range-checked: one outside [-1, nslots) raises MOE_ERR_INTERNAL
// (from lane 0 of the calling warp, or from each caller when lane is always 0) and the row is
// taken as padding (-1), so no access follows it.
__device__ __forceinline__ int checked_slot(const GemmArgs &g, int slot, int lane) {
    if (slot >= -1 && slot < g.nslots) return slot;
    if (lane == 0) raise_status(g.status, kStatusInternal);
    return -1;
}

constexpr int kGatherRows = 4;
// m: the macrobatch; ready: its per-minibatch ready counters (the claim counter follows them).
template <bool FP8>
__device__ void gather_loop(const GemmArgs &g, int m, int *ready, const uint64_t *stop_bar = nullptr) {
    const int lane = threadIdx.x % 32;
    const int r0 = g.offp[m * g.E], r1 = g.offp[(m + 1) * g.E];
    const int vecs = g.H / 8;
    int *claim = ready + g.ready_slots;      // row-chunk counter, after the ready counters
    for (;;) {
        if (stop_bar) {
            int done = 0;
            if (lane == 0) done = mbar_try_wait(smem_u32(stop_bar), 0) ? 1 : 0;
            if (__shfl_sync(0xffffffffu, done, 0)) break;
        }
        int c = 0;
        if (lane == 0) c = atomicAdd(claim, 1);
        c = __shfl_sync(0xffffffffu, c, 0);
        const int rb = r0 + c * kGatherRows;
        if (rb >= r1) break;
        if constexpr (!FP8) {
            // two rows at a time, 8 vectors of each per lane in flight (8 KB per warp)
            for (int r = rb; r < rb + kGatherRows; r += 2) {
                const bf16 *src[2];
                bf16 *dst[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int slot = checked_slot(g, g.row_slot[r + i], lane);
                    src[i] = slot >= 0 ? g.xsrc + (size_t)(slot / g.k) * g.H : nullptr;
                    dst[i] = g.ringx + (size_t)(g.x_global ? r + i : r + i - r0 + g.ring_base) * g.H;
                }
                for (int v0 = 0; v0 < vecs; v0 += 256) {
                    uint4 q[2][8];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int v = v0 + lane + 32 * u;
                            q[i][u] = (src[i] && v < vecs) ? ld_nc_v4(src[i] + v * 8) : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int v = v0 + lane + 32 * u;
                            if (v < vecs) st_v4(dst[i] + v * 8, q[i][u]);
                        }
                }
            }
        } else {
            for (int r = rb; r < rb + kGatherRows; ++r) {
                const int slot = checked_slot(g, g.row_slot[r], lane);
                const bf16 *src = slot >= 0 ? g.xsrc + (size_t)(slot / g.k) * g.H : nullptr;
                const size_t drow = (size_t)(r - r0 + g.ring_base);
                uint8_t *dst = g.ringxq + drow * g.H;
                // 4 vectors per lane in flight; a quad of lanes holds one 32-element block
                // (vecs is a multiple of 16, so a quad is valid or invalid as a whole)
                for (int v0 = 0; v0 < vecs; v0 += 128) {
                    uint4 q[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int v = v0 + lane + 32 * u;
                        q[u] = (src && v < vecs) ? ld_nc_v4(src + v * 8) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int v = v0 + lane + 32 * u;
                        const uint32_t w4[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) { f[2 * i] = bf16lo(w4[i]); f[2 * i + 1] = bf16hi(w4[i]); }
                        float amax = 0.0f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                        const int sx = mx_exponent(amax);
                        const float inv = mx_inv_scale(sx);
                        uint2 cq;
                        cq.x = cvt_e4m3x4(f[0] * inv, f[1] * inv, f[2] * inv, f[3] * inv);
                        cq.y = cvt_e4m3x4(f[4] * inv, f[5] * inv, f[6] * inv, f[7] * inv);
                        if (v < vecs) {
                            *reinterpret_cast<uint2 *>(dst + v * 8) = cq;
                            if ((lane & 3) == 0) g.ringxs[mx_sf_offset(drow, (size_t)v * 8, g.H)] = (uint8_t)(sx + 127);
                        }
                    }
                }
            }
        }
        // publish: this warp's 4 rows of minibatch j are in the ring
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            fence_proxy_async_global();
            red_release_gpu_add(ready + (rb - r0) / g.mb_rows, kGatherRows);
        }
    }
}

template <int OP, bool FP8>
__device__ void producer_loop(const GemmArgs &g, const SmemCtl &c, uint8_t *tiles, uint64_t *full,
                              uint64_t *empty, const WaitCtl &ctl) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_phase = 0;   // per stage: a copy was issued / the phase of the last one
    bool ok = true;
    const int total = num_tiles<OP>(c, g);
    const int a_shift = g.a_ring ? (g.ring_base - g.offp[g.m * g.E]) : 0;
    int ready_mb = -1;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        TileInfo ti = decode_tile<OP, FP8>(c, g, t);
        if constexpr (OP == OP_FWD1) {
            if (g.fused) {
                // the tile's rows lie in one minibatch (minibatches are 128-row aligned)
                const int r0 = g.offp[g.m * g.E], nrows = g.offp[(g.m + 1) * g.E] - r0;
                const int j = (ti.g0 - r0) / g.mb_rows;
                if (j != ready_mb) {
                    const int need = min(g.mb_rows, nrows - j * g.mb_rows);
                    if (!flag_wait_geq(g.ready + j, need, ctl)) { ok = false; break; }
                    fence_proxy_async_global();
                    ready_mb = j;
                }
            }
        }
        // grouped-K ops walk expert e's runs in macrobatch order: (run, offset) advance with kb
        int run_m = 0, run_off = 0;
        for (int kb = 0; kb < ti.nk; ++kb) {
            int krow = 0;
            if constexpr (OpTraits<OP>::grouped_k) {
                for (;;) {
                    const int s0 = g.offp[run_m * g.E + ti.e], s1 = g.offp[run_m * g.E + ti.e + 1];
                    if (run_off < s1 - s0) { krow = s0 + run_off; break; }
                    run_off = 0;
                    ++run_m;
                }
                run_off += bk_elems<FP8>();
            }
            if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, ctl)) { ok = false; break; }
            uint32_t bar = smem_u32(&full[stage]);
            uint32_t sA = smem_u32(tiles + stage * stage_stride<FP8>());
            uint32_t sB = sA + A_BYTES;
            if constexpr (!FP8) {
                mbar_arrive_expect_tx(bar, STAGE_BYTES);
                if constexpr (OP == OP_FWD1) {
                    int ar = ti.g0 + a_shift, br = ti.e * g.H + kb * BK, n0 = ti.nt * 128;
                    tma_load_2d(sA, &g.a0, bar, kb * BK, ar);
                    tma_load_3d(sB, &g.b0, bar, 0, br, n0 / 64);                  // 2 chunks of W1
                    tma_load_3d(sB + 2 * CHUNK_BYTES, &g.b1, bar, 0, br, n0 / 64);   // 2 chunks of W3
                } else if constexpr (OP == OP_FWD2) {
                    int ar = ti.g0 + a_shift, br = ti.e * g.F + kb * BK, n0 = ti.nt * BN;
                    tma_load_2d(sA, &g.a0, bar, kb * BK, ar);
#pragma unroll
                    tma_load_3d(sB, &g.b0, bar, 0, br, n0 / 64);                  // 4 chunks
                } else if constexpr (OP == OP_BWD2) {
                    tma_load_2d(sA, &g.a0, bar, kb * BK, ti.g0 + a_shift);
                    tma_load_2d(sB, &g.b0, bar, kb * BK, ti.e * g.F + ti.nt * BN);
                } else if constexpr (OP == OP_BWD1) {
                    const int kf = g.F / BK;
                    const bool second = kb >= kf;
                    const int kk = second ? kb - kf : kb;
                    tma_load_2d(sA, second ? &g.a1 : &g.a0, bar, kk * BK, ti.g0 + a_shift);
                    tma_load_2d(sB, second ? &g.b1 : &g.b0, bar, kk * BK, ti.e * g.H + ti.nt * BN);
                } else if constexpr (OP == OP_WG2) {
                    const int row = krow;
                    int m0 = ti.mt * BM, n0 = ti.nt * BN;
                    tma_load_3d(sA, &g.a0, bar, 0, row, m0 / 64);                 // 2 chunks
                    tma_load_3d(sB, &g.b0, bar, 0, row, n0 / 64);                 // 4 chunks
                } else if constexpr (OP == OP_WG13) {
                    const int row = krow;
                    int m0 = ti.mt * BM, n0 = ti.nt * 128;
                    tma_load_3d(sA, &g.a0, bar, 0, row, m0 / 64);                 // 2 chunks
                    tma_load_3d(sB, &g.b0, bar, 0, row, n0 / 64);                 // 2 chunks of da
                    tma_load_3d(sB + 2 * CHUNK_BYTES, &g.b1, bar, 0, row, n0 / 64);   // 2 chunks of db
                }
            } else {
                // e4m3 tiles (all K-major, 128 B of K per row) + three scale atoms
                const uint32_t sSF = sB + B_BYTES;
                const int KS = g.kstore;
                mbar_arrive_expect_tx(bar, STAGE_BYTES + SF_BYTES);
                if constexpr (OP == OP_FWD1) {
                    const int ar = ti.g0 + a_shift, br = ti.e * g.F + ti.nt * 128, k0 = kb * BK8;
                    tma_load_2d(sA, &g.a0, bar, k0, ar);
                    tma_load_2d(sB, &g.b0, bar, k0, br);
                    tma_load_2d(sB + 16384, &g.b1, bar, k0, br);
                    bulk_load(sSF, g.sfa0 + atom_at(ar, k0, KS), 512, bar);
                    bulk_load(sSF + 512, g.sfb0 + atom_at(br, k0, KS), 512, bar);
                    bulk_load(sSF + 1024, g.sfb1 + atom_at(br, k0, KS), 512, bar);
                } else if constexpr (OP == OP_FWD2 || OP == OP_BWD2) {
                    const int ar = ti.g0 + a_shift, k0 = kb * BK8;
                    const int br = OP == OP_FWD2 ? ti.e * g.H + ti.nt * BN : ti.e * g.F + ti.nt * BN;
                    tma_load_2d(sA, &g.a0, bar, k0, ar);
                    tma_load_2d(sB, &g.b0, bar, k0, br);
                    bulk_load(sSF, g.sfa0 + atom_at(ar, k0, KS), 512, bar);
                    bulk_load(sSF + 512, g.sfb0 + atom_at(br, k0, KS), 512, bar);
                    bulk_load(sSF + 1024, g.sfb0 + atom_at(br + 128, k0, KS), 512, bar);
                } else if constexpr (OP == OP_BWD1) {
                    const int kf = g.F / BK8;
                    const bool second = kb >= kf;
                    const int k0 = (second ? kb - kf : kb) * BK8;
                    const int ar = ti.g0 + a_shift, br = ti.e * g.H + ti.nt * BN;
                    const uint8_t *sfa = second ? g.sfa1 : g.sfa0, *sfb = second ? g.sfb1 : g.sfb0;
                    tma_load_2d(sA, second ? &g.a1 : &g.a0, bar, k0, ar);
                    tma_load_2d(sB, second ? &g.b1 : &g.b0, bar, k0, br);
                    bulk_load(sSF, sfa + atom_at(ar, k0, KS), 512, bar);
                    bulk_load(sSF + 512, sfb + atom_at(br, k0, KS), 512, bar);
                    bulk_load(sSF + 1024, sfb + atom_at(br + 128, k0, KS), 512, bar);
                } else if constexpr (OP == OP_WG2) {
                    // A = (w h)^T [F][rows], B = dY^T [H][rows], both quantised along rows
                    const int row = krow;
                    const int m0 = ti.mt * BM, n0 = ti.nt * BN;
                    tma_load_2d(sA, &g.a0, bar, row, m0);
                    tma_load_2d(sB, &g.b0, bar, row, n0);
                    bulk_load(sSF, g.sfa0 + atom_at(m0, row, KS), 512, bar);
                    bulk_load(sSF + 512, g.sfb0 + atom_at(n0, row, KS), 512, bar);
                    bulk_load(sSF + 1024, g.sfb0 + atom_at(n0 + 128, row, KS), 512, bar);
                } else if constexpr (OP == OP_WG13) {
                    // A = X^T [H][rows], B = [da^T | db^T] [F][rows]
                    const int row = krow;
                    const int m0 = ti.mt * BM, n0 = ti.nt * 128;
                    tma_load_2d(sA, &g.a0, bar, row, m0);
                    tma_load_2d(sB, &g.b0, bar, row, n0);
                    tma_load_2d(sB + 16384, &g.b1, bar, row, n0);
                    bulk_load(sSF, g.sfa0 + atom_at(m0, row, KS), 512, bar);
                    bulk_load(sSF + 512, g.sfb0 + atom_at(n0, row, KS), 512, bar);
                    bulk_load(sSF + 1024, g.sfb1 + atom_at(n0, row, KS), 512, bar);
                }
            }
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok) {
        // leave no bulk copy in flight: wait (bounded, regardless of the
        // status word) for the last copy issued into every stage
        for (int s = 0; s < STAGES; ++s) {
            if (!((issued >> s) & 1u)) continue;
            uint32_t bar = smem_u32(&full[s]);
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, (last_phase >> s) & 1u) && globaltimer_ns() - t0 < ctl.budget_ns) {}
        }
    }
}

template <int OP, bool FP8>
__device__ void mma_loop(const GemmArgs &g, const SmemCtl &c, uint8_t *tiles, uint64_t *full,
                         uint64_t *empty, uint64_t *tfull, uint64_t *tempty, uint64_t *drain,
                         uint32_t tmem, const WaitCtl &ctl) {
    constexpr bool AMN = OpTraits<OP>::a_mn && !FP8, BMN = OpTraits<OP>::b_mn && !FP8;
    constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, AMN, BMN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int total = num_tiles<OP>(c, g);
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        TileInfo ti = decode_tile<OP, FP8>(c, g, t);
        if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
            if (!mbar_wait(smem_u32(&full[stage]), phase, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sA = smem_u32(tiles + stage * stage_stride<FP8>());
            const uint32_t sB = sA + A_BYTES;
            if constexpr (!FP8) {
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    uint64_t ad = AMN ? sdesc_sw128(sA + kk * 2048, 8192, 1024) : sdesc_sw128(sA + kk * 32, 16, 1024);
                    uint64_t bd = BMN ? sdesc_sw128(sB + kk * 2048, 8192, 1024) : sdesc_sw128(sB + kk * 32, 16, 1024);
                    mma_bf16_ss(d, ad, bd, idesc, (kb | kk) != 0);
                }
            } else {
                // scale atoms of this stage -> TMEM: A at column 256 + 16 * stage (4 columns),
                // B at +8 (8 columns: rows 0-127 then rows 128-255)
                const uint32_t sSF = sB + B_BYTES;
                const uint32_t t_sf = tmem + 256 + 16 * stage;
                tmem_cp_32x128b_x4(t_sf, sdesc_plain(sSF, 0, 128));
                tmem_cp_32x128b_x4(t_sf + 8, sdesc_plain(sSF + 512, 0, 128));
                tmem_cp_32x128b_x4(t_sf + 12, sdesc_plain(sSF + 1024, 0, 128));
#pragma unroll
                for (int kk = 0; kk < BK8 / 32; ++kk) {
                    const uint64_t ad = sdesc_sw128(sA + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sB + kk * 32, 16, 1024);
                    mma_mxf8_ss(d, ad, bd, idesc_mxf8(BM, BN, kk), t_sf, t_sf + 8, (kb | kk) != 0);
                }
            }
            mma_commit(smem_u32(&empty[stage]));
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[acc]));
        if constexpr (FP8) {
            acc_phase ^= 1;                 // single accumulator buffer
        } else {
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }
    // all MMAs issued by this thread must be complete before TMEM is freed
    mma_commit(smem_u32(drain));
    uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(drain), 0) && globaltimer_ns() - t0 < ctl.budget_ns) {}
}

// sigmoid with the approximate reciprocal (one MUFU op; an IEEE division here
// expands to a branchy sequence that serialises the epilogue). silu = a * sigmoid(a)
// is formed the same way in the forward and the backward epilogues, so the
// backward recomputes the forward's h bit for bit. For a < -88, exp(-a) = inf and
// the reciprocal gives 0, the limit.
__device__ __forceinline__ float sigmoid_f(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }
__device__ __forceinline__ float silu_f(float a) { return a * sigmoid_f(a); }

// 32 rows (one per lane) x 32 bf16 of this warp -> a 2 KB staging buffer (64 B per
// row, 64-byte swizzle: 16-byte chunk g of row r sits at chunk g ^ ((r >> 1) & 3), the
// order a CU_TENSOR_MAP_SWIZZLE_64B map reads) -> one TMA store at (col0, row0) of map m.
// With the swizzle the eight lanes of a quarter warp write eight different 16-byte bank
// groups (unswizzled, rows r and r + 2 share one: a 4-way conflict). NBUF buffers per
// warp rotate; a buffer is reused once the store issued NBUF stores earlier has read it.
template <int NBUF = 4>
__device__ __forceinline__ void stage_store_bf16(uint8_t *warp_stage, int &nstores, const uint32_t (&w)[16],
                                                 const CUtensorMap *m, int col0, int row0, int lane) {
    uint8_t *buf = warp_stage + (nstores % NBUF) * 2048;
    if (nstores >= NBUF) {
        if (lane == 0) bulk_wait_group_read<NBUF - 1>();
        __syncwarp();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(buf + lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16)) =
            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(m, smem_u32(buf), col0, row0);
        bulk_commit_group();
    }
    ++nstores;
}

// 32 rows (one per lane) x 32 bf16 of this warp -> a 2 KB staging buffer in the
// blocked order of blk32_offset (conflict-free: lanes write consecutive 16 B) -> one
// contiguous bulk copy to the block at dst. Shares the buffer rotation of stage_store_bf16.
template <int NBUF = 4>
__device__ __forceinline__ void stage_store_blk(uint8_t *warp_stage, int &nstores, const uint32_t (&w)[16],
                                                bf16 *dst, int lane) {
    uint8_t *buf = warp_stage + (nstores % NBUF) * 2048;
    if (nstores >= NBUF) {
        if (lane == 0) bulk_wait_group_read<NBUF - 1>();
        __syncwarp();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(buf + (q * 32 + lane) * 16) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        bulk_store(dst, smem_u32(buf), 2048);
        bulk_commit_group();
    }
    ++nstores;
}

// Epilogue of one GEMM1 tile (this thread's accumulator row r): a, b rounded to bf16 and saved
// in 32 x 32 blocks at the global padded rows, h = silu(a) * b from the rounded a, b into the ring
// (bf16, or E4M3 along F with its scale bytes).
// One warp's 32 rows x 32 columns of bf16 values (lane = row, w = its 32 columns packed)
// quantised along the rows: MXFP8 blocks of 32 padded rows (the token axis of a weight-gradient
// operand [C][R]). The tile passes through a 2 KB staging buffer (16-byte chunks XOR-swizzled as
// in stage_store_bf16, so both the row writes and the column reads are free of bank conflicts);
// lane c then holds column col0 + c whole and writes its 32 codes as one sector and its scale
// byte. The arithmetic is mx_quant32 on the bf16 values, the same bytes the standalone
// token-axis quantiser makes from those values.
__device__ __forceinline__ void token_axis_q32(uint8_t *stage, const uint32_t (&w)[16], uint8_t *codes,
                                               uint8_t *scales, int col0, int row0, int R, int lane) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(stage + lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16)) =
            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    __syncwarp();
    float v[32];
    const int cq = lane >> 3, ce = (lane & 7) * 2;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const uint32_t b = *reinterpret_cast<const uint16_t *>(stage + r * 64 + ((cq ^ ((r >> 1) & 3)) * 16) + ce);
        v[r] = __uint_as_float(b << 16);
    }
    __syncwarp();   // the buffer is free for the next tile
    uint32_t cw[8];
    const uint32_t sb = mx_quant32(v, cw);
    st_global_32B(codes + (size_t)(col0 + lane) * R + row0, cw);
    scales[mx_sf_offset((size_t)(col0 + lane), (size_t)row0, (size_t)R)] = (uint8_t)sb;
}

template <bool FP8, int NBUF>
__device__ __forceinline__ void epi_fwd1_tile(const GemmArgs &g, const TileInfo &ti, uint32_t tbase, int r,
                                              int quarter, int lane, int ring_shift, bool tma_bf16,
                                              uint8_t *warp_stage, int &store_chunks) {
    const int grow = ti.g0 + r;
    const size_t F = g.F;
    const int brow = ti.g0 + quarter * 32;   // first row of this warp's 32-row blocks of a, b
    bf16 *ph = FP8 ? nullptr : g.o2 + (size_t)(grow + ring_shift) * F + ti.nt * 128;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
        uint32_t va[32], vb[32];
        tmem_ld_32x32b_x32(tbase + cc * 32, va);
        tmem_ld_32x32b_x32(tbase + 128 + cc * 32, vb);
        tmem_ld_wait();
        uint32_t oa[16], ob[16], oh[16];
        float hf[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            oa[i] = pack_bf16x2(__uint_as_float(va[2 * i]), __uint_as_float(va[2 * i + 1]));
            ob[i] = pack_bf16x2(__uint_as_float(vb[2 * i]), __uint_as_float(vb[2 * i + 1]));
            // h from the bf16-rounded a and b, so the backward recomputes it exactly
            float a0 = bf16lo(oa[i]), a1 = bf16hi(oa[i]);
            float b0 = bf16lo(ob[i]), b1 = bf16hi(ob[i]);
            hf[2 * i] = silu_f(a0) * b0;
            hf[2 * i + 1] = silu_f(a1) * b1;
            oh[i] = pack_bf16x2(hf[2 * i], hf[2 * i + 1]);
        }
        const int col0 = ti.nt * 128 + cc * 32;
        bf16 *ba = g.o0 + blk32_offset(brow, col0, g.F), *bb = g.o1 + blk32_offset(brow, col0, g.F);
        if (tma_bf16) {
            stage_store_blk<NBUF>(warp_stage, store_chunks, oa, ba, lane);
            stage_store_blk<NBUF>(warp_stage, store_chunks, ob, bb, lane);
            stage_store_bf16<NBUF>(warp_stage, store_chunks, oh, &g.om2, col0, brow + ring_shift, lane);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                st_v4(ba + (v * 32 + lane) * 8, make_uint4(oa[4 * v], oa[4 * v + 1], oa[4 * v + 2], oa[4 * v + 3]));
                st_v4(bb + (v * 32 + lane) * 8, make_uint4(ob[4 * v], ob[4 * v + 1], ob[4 * v + 2], ob[4 * v + 3]));
                if constexpr (!FP8)
                    st_v4(ph + cc * 32 + v * 8, make_uint4(oh[4 * v], oh[4 * v + 1], oh[4 * v + 2], oh[4 * v + 3]));
            }
        }
        if constexpr (FP8) {
            // h quantised along F (blocks of 32) for GEMM2's A operand
            uint32_t q[8];
            const uint32_t sb = mx_quant32(hf, q);
            const size_t hrow = (size_t)(grow + ring_shift);
            const size_t col = (size_t)ti.nt * 128 + cc * 32;
            st_global_32B(g.q0 + hrow * F + col, q);   // one sector per row (the ring: 32-byte aligned)
            g.qs0[mx_sf_offset(hrow, col, F)] = (uint8_t)sb;
        }
    }
}

// Epilogue of one GEMM2 or GEMM1-dgrad tile: the fp32 accumulator row rounded to bf16 (GEMM2:
// Y into the ring rows; GEMM1 dgrad: dX rows).
template <int OP, int NBUF>
__device__ __forceinline__ void epi_rows_tile(const GemmArgs &g, const TileInfo &ti, uint32_t tbase, int r,
                                              int quarter, int lane, int ring_shift, bool tma_bf16,
                                              uint8_t *warp_stage, int &store_chunks) {
    const int grow = ti.g0 + r;
    const size_t orow = (OP == OP_FWD2 && g.o_ring) ? (size_t)(grow + ring_shift) : (size_t)grow;
    bf16 *py = g.o0 + orow * g.H + ti.nt * BN;
#pragma unroll 1
    for (int cc = 0; cc < BN / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tbase + cc * 32, v);
        tmem_ld_wait();
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        if (tma_bf16) {
            const int row0 = (int)(orow - r) + quarter * 32;
            stage_store_bf16<NBUF>(warp_stage, store_chunks, o, &g.om0, ti.nt * BN + cc * 32, row0, lane);
        } else if ((reinterpret_cast<uintptr_t>(py) & 31) == 0) {
            // straight from registers: two whole-sector stores per row chunk
            const uint32_t w0[8] = {o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]};
            const uint32_t w1[8] = {o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]};
            st_global_32B(py + cc * 32, w0);
            st_global_32B(py + cc * 32 + 16, w1);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st_v4(py + cc * 32 + q * 8, make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]));
        }
    }
}

// PAIR: the CTA pair computes a 256-row tile; this CTA's accumulator holds
// rows [128 * rank, +128). A half beyond its expert's run (odd number of
// 128-row tiles) is computed on whatever rows follow and not stored.
// EW = epilogue warps (warps 2 .. 2+EW): with 8, two warps read each TMEM lane
// quarter and split the tile's columns (GEMM2 dgrad: its SwiGLU backward is
// latency-bound with one warp per SM sub-partition). Each warp owns
// 32 KB / EW of staging.
template <int OP, bool FP8, bool PAIR = false, int EW = 4, class Ctl>
__device__ void epilogue_loop(const GemmArgs &g, const Ctl &c, const uint64_t *tfull, uint64_t *tempty,
                              uint32_t tmem, const WaitCtl &ctl, uint8_t *staging = nullptr) {
    static_assert(EW == 4 || EW == 8, "epilogue warps");
    constexpr int NBUF = (EW == 8 || FP8) ? 2 : 4;   // 2 KB staging buffers per warp (MXFP8 pairs: 16 KB in all)
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int half = EW == 8 ? (warp - 2) / 4 : 0;   // column half of the tile this warp takes
    const int quarter = warp & 3;             // TMEM lanes this warp may read
    const int r = quarter * 32 + lane;        // accumulator row of this thread
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int total = num_tiles<OP>(c, g);
    const int ring_shift = g.ring_base - g.offp[g.m * g.E];
    const int rank = PAIR ? (int)cluster_ctarank() : 0;
    int store_chunks = 0;   // TMA stores issued by this warp (lane 0 tracks the bulk groups)
    // bf16 row outputs leave through shared memory and TMA stores; in MXFP8 kernels only the
    // GEMM2 / GEMM1-dgrad rows (the quantised outputs are stored from registers)
    const bool tma_bf16 = staging != nullptr && g.tma_store && OP != OP_WG2 && OP != OP_WG13 &&
                          (!FP8 || OP == OP_FWD2 || OP == OP_BWD1);
    // MXFP8 GEMM2 dgrad: one 2 KB buffer per warp for the token-axis transposition
    constexpr uint32_t kWarpStage = (FP8 && OP == OP_BWD2) ? 2048 : NBUF * 2048;
    uint8_t *warp_stage = staging ? staging + (warp - 2) * kWarpStage : nullptr;
    const int t0 = PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x;
    const int tstep = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;
    for (int t = t0; t < total; t += tstep) {
        TileInfo ti = decode_tile<OP, FP8, PAIR ? 2 * BM : BM>(c, g, t);
        bool phantom = false;
        if constexpr (PAIR) {
            if constexpr (OpTraits<OP>::grouped_k) {
                ti.mt = ti.mt * 2 + rank;
            } else if (rank) {
                phantom = ti.g1 < 0;   // no second chunk: nothing to store
                ti.g0 = ti.g1;
            }
        }
        if (!mbar_wait(smem_u32(&tfull[acc]), acc_phase, ctl)) break;
        tc_fence_after();
        const uint32_t tbase = tmem + lane_base + acc * BN;
        if (phantom) {
            // nothing to store for rows past the expert's run
        } else if constexpr (OP == OP_FWD1) {
            epi_fwd1_tile<FP8, NBUF>(g, ti, tbase, r, quarter, lane, ring_shift, tma_bf16, warp_stage, store_chunks);
        } else if constexpr (OP == OP_FWD2 || OP == OP_BWD1) {
            epi_rows_tile<OP, NBUF>(g, ti, tbase, r, quarter, lane, ring_shift, tma_bf16, warp_stage, store_chunks);
        } else if constexpr (OP == OP_BWD2) {
            const int grow = ti.g0 + r;
            const size_t F = g.F;
            const int slot = checked_slot(g, g.row_slot[grow], 0);
            const float w = slot >= 0 ? g.wslot[slot] : 0.0f;
            // saved a, b in 32 x 32 blocks: this lane's 16-byte vector j of chunk cc is
            // at blk32_offset(block row, column) + (j * 32 + lane) * 8 elements
            const int brow = ti.g0 + quarter * 32;
            auto pa_at = [&](int cc) { return g.in0 + blk32_offset(brow, ti.nt * BN + cc * 32, g.F) + lane * 8; };
            auto pb_at = [&](int cc) { return g.in1 + blk32_offset(brow, ti.nt * BN + cc * 32, g.F) + lane * 8; };
            bf16 *pda = g.o0 + grow * F + ti.nt * BN;
            bf16 *pdb = g.o1 + grow * F + ti.nt * BN;
            bf16 *phw = g.o2 + grow * F + ti.nt * BN;
            // <G, h> over this warp's columns in four interleaved sums (column i % 4), added in a
            // fixed order at the end: a chain a quarter as deep, the same result every run
            float dwq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            constexpr int NCH = BN / 32 / (EW / 4);   // 32-column chunks of this warp
            const int cc0 = half * NCH, cc1 = cc0 + NCH;
            // saved a, b of the next 32 columns are loaded one chunk ahead so their
            // latency overlaps the current chunk's work
            uint4 na[4], nb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                na[q] = ld_nc_v4(pa_at(cc0) + q * 256);
                nb[q] = ld_nc_v4(pb_at(cc0) + q * 256);
            }
#pragma unroll 1
            for (int cc = cc0; cc < cc1; ++cc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tbase + cc * 32, v);
                uint32_t ra[16], rb[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ra[4 * q] = na[q].x; ra[4 * q + 1] = na[q].y; ra[4 * q + 2] = na[q].z; ra[4 * q + 3] = na[q].w;
                    rb[4 * q] = nb[q].x; rb[4 * q + 1] = nb[q].y; rb[4 * q + 2] = nb[q].z; rb[4 * q + 3] = nb[q].w;
                }
                if (cc + 1 < cc1) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        na[q] = ld_nc_v4(pa_at(cc + 1) + q * 256);
                        nb[q] = ld_nc_v4(pb_at(cc + 1) + q * 256);
                    }
                }
                tmem_ld_wait();
                uint32_t oda[16], odb[16], ohw[16];
                float daf[32], dbf[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float hw2[2];
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        float a = h2 ? bf16hi(ra[i]) : bf16lo(ra[i]);
                        float b = h2 ? bf16hi(rb[i]) : bf16lo(rb[i]);
                        float G = __uint_as_float(v[2 * i + h2]);
                        float sg = sigmoid_f(a);
                        float sl = a * sg;
                        float hval = __bfloat162float(__float2bfloat16_rn(sl * b));   // h as the forward stored it
                        dwq[(2 * i + h2) & 3] = fmaf(G, hval, dwq[(2 * i + h2) & 3]);
                        float dh = w * G;
                        daf[2 * i + h2] = dh * b * sg * (1.0f + a * (1.0f - sg));
                        dbf[2 * i + h2] = dh * sl;
                        hw2[h2] = w * hval;
                    }
                    oda[i] = pack_bf16x2(daf[2 * i], daf[2 * i + 1]);
                    odb[i] = pack_bf16x2(dbf[2 * i], dbf[2 * i + 1]);
                    ohw[i] = pack_bf16x2(hw2[0], hw2[1]);
                }
                if constexpr (FP8) {
                    // da, db quantised along F (blocks of 32) for the GEMM1 dgrad
                    const size_t col = (size_t)ti.nt * BN + cc * 32;
                    uint32_t q[8];
                    // one sector per row (workspace buffers: 32-byte aligned)
                    uint32_t sb = mx_quant32(daf, q);
                    st_global_32B(g.q0 + (size_t)grow * F + col, q);
                    g.qs0[mx_sf_offset(grow, col, F)] = (uint8_t)sb;
                    sb = mx_quant32(dbf, q);
                    st_global_32B(g.q1 + (size_t)grow * F + col, q);
                    g.qs1[mx_sf_offset(grow, col, F)] = (uint8_t)sb;
                    // the bf16 da, db and h.w quantised along the padded rows for dW1/dW3 and dW2
                    // (a warp's 32 rows are one block: runs start at multiples of 128 rows)
                    const int row0 = ti.g0 + quarter * 32, col0 = ti.nt * BN + cc * 32;
                    token_axis_q32(warp_stage, oda, g.tq[0], g.tqs[0], col0, row0, g.tR, lane);
                    token_axis_q32(warp_stage, odb, g.tq[1], g.tqs[1], col0, row0, g.tR, lane);
                    token_axis_q32(warp_stage, ohw, g.tq[2], g.tqs[2], col0, row0, g.tR, lane);
                    continue;
                }
                if (tma_bf16) {
                    const int row0 = ti.g0 + quarter * 32, col0 = ti.nt * BN + cc * 32;
                    stage_store_bf16<NBUF>(warp_stage, store_chunks, oda, &g.om0, col0, row0, lane);
                    stage_store_bf16<NBUF>(warp_stage, store_chunks, odb, &g.om1, col0, row0, lane);
                    stage_store_bf16<NBUF>(warp_stage, store_chunks, ohw, &g.om2, col0, row0, lane);
                    continue;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    st_v4(pda + cc * 32 + q * 8, make_uint4(oda[4 * q], oda[4 * q + 1], oda[4 * q + 2], oda[4 * q + 3]));
                    st_v4(pdb + cc * 32 + q * 8, make_uint4(odb[4 * q], odb[4 * q + 1], odb[4 * q + 2], odb[4 * q + 3]));
                    st_v4(phw + cc * 32 + q * 8, make_uint4(ohw[4 * q], ohw[4 * q + 1], ohw[4 * q + 2], ohw[4 * q + 3]));
                }
            }
            const float dwp = (dwq[0] + dwq[1]) + (dwq[2] + dwq[3]);
            // dw partials: one per 128 columns of F, [row][F / 128]
            float *dwo = g.of0 + (size_t)grow * (g.F / 128) + ti.nt * 2;
            if (EW == 8) {
                dwo[half] = dwp;
            } else {
                dwo[0] = dwp;
                dwo[1] = 0.0f;
            }
        } else {   // OP_WG2, OP_WG13: fp32 weight gradients
            const bool empty_k = ti.nk == 0;
            const int row = ti.mt * BM + r;
            float *dst0, *dst1 = nullptr;
            int ncol0;
            if constexpr (OP == OP_WG2) {   // dW2[e][f][h]
                dst0 = g.of0 + ((size_t)ti.e * g.F + row) * g.H + ti.nt * BN;
                ncol0 = BN;
            } else {                        // dW1/dW3[e][h][f]
                dst0 = g.of0 + ((size_t)ti.e * g.H + row) * g.F + ti.nt * 128;
                dst1 = g.of1 + ((size_t)ti.e * g.H + row) * g.F + ti.nt * 128;
                ncol0 = 128;
            }
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t v[32];
                if (!empty_k) {
                    tmem_ld_32x32b_x32(tbase + cc * 32, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                }
                if (staging != nullptr && g.tma_store && !g.accumulate) {
                    // 32 rows x 32 fp32 of this warp -> 128B-swizzled staging buffer -> one TMA store.
                    // Two buffers per warp: wait until the store issued two chunks ago has read its source.
                    uint8_t *buf = warp_stage + (store_chunks & 1) * 4096;
                    if (store_chunks >= 2) {
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<uint4 *>(buf + lane * 128 + ((q ^ (lane & 7)) * 16)) =
                            make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        const int row0 = (OP == OP_WG2 ? ti.e * g.F : ti.e * g.H) + ti.mt * BM + quarter * 32;
                        const CUtensorMap *om = (cc * 32 < ncol0) ? &g.om0 : &g.om1;
                        const int col0 = (OP == OP_WG2 ? ti.nt * BN : ti.nt * 128) + (cc * 32 < ncol0 ? cc * 32 : cc * 32 - ncol0);
                        tma_store_2d(om, smem_u32(buf), col0, row0);
                        bulk_commit_group();
                    }
                    ++store_chunks;
                    continue;
                }
                float *dst = (cc * 32 < ncol0) ? dst0 + cc * 32 : dst1 + (cc * 32 - ncol0);
                if (!g.accumulate && (reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
                    // whole 32-byte sectors: four 8-word stores of this row's 32 columns (the
                    // caller's gradient may be only 16-byte aligned: then 16-byte stores below)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t w8[8] = {v[8 * q], v[8 * q + 1], v[8 * q + 2], v[8 * q + 3],
                                                v[8 * q + 4], v[8 * q + 5], v[8 * q + 6], v[8 * q + 7]};
                        st_global_32B(dst + q * 8, w8);
                    }
                    continue;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float4 o = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                    float4 *p = reinterpret_cast<float4 *>(dst + q * 4);
                    if (g.accumulate) {
                        float4 old = *p;
                        o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
                    }
                    *p = o;
                }
            }
        }
        tc_fence_before();
        if constexpr (PAIR) {
            // the leader's MMA thread waits for both CTAs' epilogues
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
        } else {
            mbar_arrive(smem_u32(&tempty[acc]));
        }
        if constexpr (FP8) {
            acc_phase ^= 1;
        } else {
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }
    if (store_chunks > 0 && lane == 0) bulk_wait_group_all();
}

// 320 threads: ten warps over the SM's four sub-partitions, three of them on one 16K-register
// file, so at most 168 registers per thread.
template <int OP, bool FP8>
__global__ void __launch_bounds__(320, 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // bf16: 32 KB over the epilogue warps; MXFP8 GEMM2 dgrad: 2 KB per epilogue warp
    uint8_t *staging = staging_bytes<OP, FP8>() ? tiles + STAGES * stage_stride<FP8>() : nullptr;
    SmemCtl &c = *reinterpret_cast<SmemCtl *>(tiles + STAGES * stage_stride<FP8>() + staging_bytes<OP, FP8>());
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    WaitCtl ctl{g.status, g.budget_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&c.full[s]), 1);
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&c.tfull[a]), 1);
            mbar_init(smem_u32(&c.tempty[a]), OP == OP_BWD2 ? 256 : 128);   // epilogue threads
        }
        mbar_init(smem_u32(&c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&g.a0);
        tma_prefetch_map(&g.b0);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem_base), 512);
        tmem_relinquish();
    }
    pdl_wait();   // barriers and TMEM are set up while the previous kernel finishes
    if (threadIdx.x == 0) init_tile_table<OP, BM>(c, g);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = c.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer_loop<OP, FP8>(g, c, tiles, c.full, c.empty, ctl);
    } else if (warp == 1) {
        if (lane == 0) mma_loop<OP, FP8>(g, c, tiles, c.full, c.empty, c.tfull, c.tempty, &c.drain, tmem, ctl);
    } else if constexpr (OP == OP_BWD2) {
        epilogue_loop<OP, FP8, false, 8>(g, c, c.tfull, c.tempty, tmem, ctl, staging);   // warps 2-9
    } else if (warp < 6) {
        if constexpr (OP == OP_FWD1) {
            if (g.fused) gather_loop<FP8>(g, g.m, g.ready, &c.tfull[0]);   // until the first accumulator is ready
        }
        epilogue_loop<OP, FP8>(g, c, c.tfull, c.tempty, tmem, ctl, staging);
    } else {
        if constexpr (OP == OP_FWD1) gather_loop<FP8>(g, g.m, g.ready);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ======================================================================
// CTA-pair (cta_group::2) variant, bf16: 256-row tiles, each CTA holds its
// 128 rows of A and one 128-wide half of B (6 stages of 32 KB); the leader
// CTA (rank 0) issues M=256 N=256 MMAs over both CTAs' shared memory, the
// accumulator rows of each CTA land in its own TMEM. Full barriers live in
// the leader (both producers arrive with their bytes); MMA commits arrive on
// the empty / tmem-full barriers of both CTAs; both epilogues arrive on the
// leader's tmem-empty barrier.
constexpr int PSTAGES = 6;
constexpr uint32_t P_A_BYTES = BM * BK * 2;            // 16 KiB
constexpr uint32_t P_B_BYTES = 128 * BK * 2;           // 16 KiB: half of N = 256
constexpr uint32_t P_STAGE = P_A_BYTES + P_B_BYTES;    // 32 KiB
constexpr uint32_t P_STAGING = 4 * 2 * 4096;          // epilogue staging for TMA stores
using PairCtl = CtlT<PSTAGES>;

template <int OP>
__device__ void pair_producer_loop(const GemmArgs &g, const PairCtl &c, uint8_t *tiles, const WaitCtl &ctl) {
    const int rank = (int)cluster_ctarank();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_phase = 0;   // per stage: a copy was issued / the phase of the last one
    bool ok = true;
    const int total = num_tiles<OP>(c, g);
    const int a_shift = g.a_ring ? (g.ring_base - g.offp[g.m * g.E]) : 0;
    int ready_mb = -1;
    for (int t = blockIdx.x / 2; t < total && ok; t += gridDim.x / 2) {
        TileInfo ti = decode_tile<OP, false, 2 * BM>(c, g, t);
        // grouped-M: this CTA's 128 rows (a second CTA without a chunk loads rows it discards)
        const int row0 = rank ? (ti.g1 >= 0 ? ti.g1 : ti.g0 + BM) : ti.g0;
        const int m0 = (ti.mt * 2 + rank) * BM;          // grouped-K: this CTA's 128 rows of dW
        if constexpr (OP == OP_FWD1) {
            if (g.fused && (rank == 0 || ti.g1 >= 0)) {
                const int r0 = g.offp[g.m * g.E], nrows = g.offp[(g.m + 1) * g.E] - r0;
                const int j = (row0 - r0) / g.mb_rows;
                if (j != ready_mb) {
                    const int need = min(g.mb_rows, nrows - j * g.mb_rows);
                    if (!flag_wait_geq(g.ready + j, need, ctl)) { ok = false; break; }
                    fence_proxy_async_global();
                    ready_mb = j;
                }
            }
        }
        int run_m = 0, run_off = 0;
        for (int kb = 0; kb < ti.nk; ++kb) {
            int krow = 0;
            if constexpr (OpTraits<OP>::grouped_k) {
                for (;;) {
                    const int s0 = g.offp[run_m * g.E + ti.e], s1 = g.offp[run_m * g.E + ti.e + 1];
                    if (run_off < s1 - s0) { krow = s0 + run_off; break; }
                    run_off = 0;
                    ++run_m;
                }
                run_off += BK;
            }
            if (!mbar_wait(smem_u32(&c.empty[stage]), phase ^ 1, ctl)) { ok = false; break; }
            const uint32_t bar = mapa_shared(smem_u32(&c.full[stage]), 0);   // the leader's full barrier
            const uint32_t sA = smem_u32(tiles + stage * P_STAGE);
            const uint32_t sB = sA + P_A_BYTES;
            mbar_arrive_expect_tx_cluster(bar, P_STAGE);
            if constexpr (OP == OP_FWD1) {
                const int br = ti.e * g.H + kb * BK, n0 = ti.nt * 128;
                const CUtensorMap *bm = rank == 0 ? &g.b0 : &g.b1;   // W1 half, W3 half
                tma_load_2d_pair(sA, &g.a0, bar, kb * BK, row0 + a_shift);
                tma_load_3d_pair(sB, bm, bar, 0, br, n0 / 64);
            } else if constexpr (OP == OP_FWD2) {
                const int br = ti.e * g.F + kb * BK, n0 = ti.nt * BN + 128 * rank;
                tma_load_2d_pair(sA, &g.a0, bar, kb * BK, row0 + a_shift);
                tma_load_3d_pair(sB, &g.b0, bar, 0, br, n0 / 64);
            } else if constexpr (OP == OP_BWD2) {
                tma_load_2d_pair(sA, &g.a0, bar, kb * BK, row0 + a_shift);
                tma_load_2d_pair(sB, &g.b0, bar, kb * BK, ti.e * g.F + ti.nt * BN + 128 * rank);
            } else if constexpr (OP == OP_BWD1) {
                const int kf = g.F / BK;
                const bool second = kb >= kf;
                const int kk = second ? kb - kf : kb;
                tma_load_2d_pair(sA, second ? &g.a1 : &g.a0, bar, kk * BK, row0 + a_shift);
                tma_load_2d_pair(sB, second ? &g.b1 : &g.b0, bar, kk * BK, ti.e * g.H + ti.nt * BN + 128 * rank);
            } else if constexpr (OP == OP_WG2) {
                const int n0 = ti.nt * BN + 128 * rank;
                tma_load_3d_pair(sA, &g.a0, bar, 0, krow, m0 / 64);
                tma_load_3d_pair(sB, &g.b0, bar, 0, krow, n0 / 64);
            } else if constexpr (OP == OP_WG13) {
                const int n0 = ti.nt * 128;
                const CUtensorMap *bm = rank == 0 ? &g.b0 : &g.b1;   // da half, db half
                tma_load_3d_pair(sA, &g.a0, bar, 0, krow, m0 / 64);
                tma_load_3d_pair(sB, bm, bar, 0, krow, n0 / 64);
            }
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == PSTAGES) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok && rank == 0) {
        // the leader's full barriers count both CTAs' copies: wait (bounded) for the last phases
        for (int s = 0; s < PSTAGES; ++s) {
            if (!((issued >> s) & 1u)) continue;
            const uint32_t bar = smem_u32(&c.full[s]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, (last_phase >> s) & 1u) && globaltimer_ns() - t0 < ctl.budget_ns) {}
        }
    }
}

template <int OP>
__device__ void pair_mma_loop(const GemmArgs &g, PairCtl &c, uint8_t *tiles, uint32_t tmem, const WaitCtl &ctl) {
    constexpr bool AMN = OpTraits<OP>::a_mn, BMN = OpTraits<OP>::b_mn;
    constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, AMN, BMN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int total = num_tiles<OP>(c, g);
    for (int t = blockIdx.x / 2; t < total; t += gridDim.x / 2) {
        TileInfo ti = decode_tile<OP, false, 2 * BM>(c, g, t);
        if (!mbar_wait(smem_u32(&c.tempty[acc]), acc_phase ^ 1, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
            if (!mbar_wait(smem_u32(&c.full[stage]), phase, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sA = smem_u32(tiles + stage * P_STAGE);
            const uint32_t sB = sA + P_A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = AMN ? sdesc_sw128(sA + kk * 2048, 8192, 1024) : sdesc_sw128(sA + kk * 32, 16, 1024);
                const uint64_t bd = BMN ? sdesc_sw128(sB + kk * 2048, 8192, 1024) : sdesc_sw128(sB + kk * 32, 16, 1024);
                mma_bf16_pair(d, ad, bd, idesc, (kb | kk) != 0);
            }
            mma_commit_pair_mc(smem_u32(&c.empty[stage]));   // frees the stage in both CTAs
            if (++stage == PSTAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair_mc(smem_u32(&c.tfull[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
    }
    mma_commit_pair(smem_u32(&c.drain));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < ctl.budget_ns) {}
}

template <int OP>
__global__ void __launch_bounds__(320, 1) pair_gemm_kernel(const __grid_constant__ GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *staging = tiles + PSTAGES * P_STAGE;                       // 4 epilogue warps x 2 x 4 KB
    PairCtl &c = *reinterpret_cast<PairCtl *>(staging + P_STAGING);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    WaitCtl ctl{g.status, g.budget_ns};
    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(smem_u32(&c.full[s]), 2);      // one arrive.expect_tx per CTA of the pair
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&c.tfull[a]), 1);
            mbar_init(smem_u32(&c.tempty[a]), 256);  // 128 epilogue threads of each CTA
        }
        mbar_init(smem_u32(&c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&g.a0);
        tma_prefetch_map(&g.b0);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&c.tmem_base), 512);
        tmem_relinquish_pair();
    }
    pdl_wait();   // barriers and TMEM are set up while the previous kernel finishes
    if (threadIdx.x == 0) init_tile_table<OP, 2 * BM>(c, g);
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = c.tmem_base;
    if (warp == 0) {
        if (lane == 0) pair_producer_loop<OP>(g, c, tiles, ctl);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) pair_mma_loop<OP>(g, c, tiles, tmem, ctl);
    } else if (warp < 6) {
        if constexpr (OP == OP_FWD1) {
            if (g.fused) gather_loop<false>(g, g.m, g.ready, &c.tfull[0]);   // until the first accumulator is ready
        }
        epilogue_loop<OP, false, true>(g, c, c.tfull, c.tempty, tmem, ctl, staging);
    } else {
        if constexpr (OP == OP_FWD1) gather_loop<false>(g, g.m, g.ready);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // the leader's MMAs are drained before the pair frees TMEM
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// Co-resident cluster count of one kernel configuration, queried once per device and
// kept in an atomic so that first launches from several host threads do not race.
constexpr int kMaxCachedDevices = 64;
template <class Kernel>
int cached_max_clusters(std::atomic<int> (&cache)[kMaxCachedDevices][2], int slot, Kernel kernel,
                        cudaLaunchConfig_t cfg, int fallback) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    if (dev >= 0 && dev < kMaxCachedDevices) {
        const int c = cache[dev][slot].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    cfg.numAttrs = 1;   // the cluster shape alone
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) n = fallback;
    if (dev >= 0 && dev < kMaxCachedDevices) cache[dev][slot].store(n, std::memory_order_relaxed);
    return n;
}

template <int OP>
cudaError_t launch_pair(const GemmArgs &g, int grid, cudaStream_t stream) {
    constexpr size_t smem = PSTAGES * P_STAGE + P_STAGING + sizeof(PairCtl) + 1024;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t err = cudaFuncSetAttribute(pair_gemm_kernel<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const bool fused = OP == OP_FWD1 && g.fused;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(fused ? 320 : 192);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // A persistent grid must be fully co-resident: with GPCs of an odd SM count
    // not every SM can host half of a pair, so size the grid by the number of
    // clusters that fit at once (queried once per device, kernel and block size).
    static std::atomic<int> max_clusters[kMaxCachedDevices][2];
    cfg.gridDim = dim3(grid / 2 * 2);
    const int mc = cached_max_clusters(max_clusters, fused ? 1 : 0, pair_gemm_kernel<OP>, cfg, grid / 2);
    cfg.gridDim = dim3(2 * std::min(grid / 2, mc));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<OP>, g);
}

// ======================================================================
// MXFP8 CTA-pair variant: 256-row tiles, block-scaled tcgen05.mma.cta_group::2.
// Each CTA stages its 128 rows of A and one 128-row half of B (e4m3, 128 elements
// of K per stage) plus three scale atoms: A's (its rows) and B's for BOTH halves,
// because each CTA's tensor memory must hold SFB for all 256 columns. The atoms
// are TMA loads of a [bytes / 128][128] view so that, like the tiles, they count
// on the leader's full barrier. The leader's tcgen05.cp.cta_group::2 copies each
// CTA's own atoms into its own tensor memory (SFA at column 256 + 16 stage, SFB at
// +8 and +12); the accumulator is single-buffered (columns 0-255).
constexpr int P8_STAGES = 6;
constexpr uint32_t P8_TILE = 128 * 128;                        // 16 KiB: 128 rows x 128 B
constexpr uint32_t P8_TX = 2 * P8_TILE + 3 * 512;              // bytes landing per CTA per stage
constexpr uint32_t P8_STAGE = 34816;                           // 1 KiB aligned stage stride
constexpr uint32_t P8_STAGING = 4 * 2 * 2048;                  // epilogue staging: 4 warps x 2 x 2 KB
using Pair8Ctl = CtlT<P8_STAGES>;

__device__ __forceinline__ int atom_row(int row, int k, int K) { return (int)(atom_at(row, k, K) / 128); }

template <int OP>
__device__ void pair8_producer_loop(const GemmArgs &g, const Pair8Ctl &c, uint8_t *tiles, const WaitCtl &ctl) {
    const int rank = (int)cluster_ctarank();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_phase = 0;   // per stage: a copy was issued / the phase of the last one
    bool ok = true;
    const int total = num_tiles<OP>(c, g);
    const int a_shift = g.a_ring ? (g.ring_base - g.offp[g.m * g.E]) : 0;
    const int KS = g.kstore;
    int ready_mb = -1;
    for (int t = blockIdx.x / 2; t < total && ok; t += gridDim.x / 2) {
        TileInfo ti = decode_tile<OP, true, 2 * BM>(c, g, t);
        // grouped-M: this CTA's 128 rows (a second CTA without a chunk loads rows it discards)
        const int row0 = rank ? (ti.g1 >= 0 ? ti.g1 : ti.g0 + BM) : ti.g0;
        const int m0 = (ti.mt * 2 + rank) * BM;          // grouped-K: this CTA's 128 rows of dW
        if constexpr (OP == OP_FWD1) {
            if (g.fused && (rank == 0 || ti.g1 >= 0)) {
                const int r0 = g.offp[g.m * g.E], nrows = g.offp[(g.m + 1) * g.E] - r0;
                const int j = (row0 - r0) / g.mb_rows;
                if (j != ready_mb) {
                    const int need = min(g.mb_rows, nrows - j * g.mb_rows);
                    if (!flag_wait_geq(g.ready + j, need, ctl)) { ok = false; break; }
                    fence_proxy_async_global();
                    ready_mb = j;
                }
            }
        }
        int run_m = 0, run_off = 0;
        for (int kb = 0; kb < ti.nk; ++kb) {
            int krow = 0;
            if constexpr (OpTraits<OP>::grouped_k) {
                for (;;) {
                    const int s0 = g.offp[run_m * g.E + ti.e], s1 = g.offp[run_m * g.E + ti.e + 1];
                    if (run_off < s1 - s0) { krow = s0 + run_off; break; }
                    run_off = 0;
                    ++run_m;
                }
                run_off += BK8;
            }
            if (!mbar_wait(smem_u32(&c.empty[stage]), phase ^ 1, ctl)) { ok = false; break; }
            const uint32_t bar = mapa_shared(smem_u32(&c.full[stage]), 0);   // the leader's full barrier
            const uint32_t sA = smem_u32(tiles + stage * P8_STAGE);
            const uint32_t sB = sA + P8_TILE;
            const uint32_t sSF = sB + P8_TILE;
            mbar_arrive_expect_tx_cluster(bar, P8_TX);
            if constexpr (OP == OP_FWD1) {
                const int ar = row0 + a_shift, br = ti.e * g.F + ti.nt * 128, k0 = kb * BK8;
                tma_load_2d_pair(sA, &g.a0, bar, k0, ar);
                tma_load_2d_pair(sB, rank == 0 ? &g.b0 : &g.b1, bar, k0, br);   // W1^T half, W3^T half
                tma_load_2d_pair(sSF, &g.msa0, bar, 0, atom_row(ar, k0, KS));
                tma_load_2d_pair(sSF + 512, &g.msb0, bar, 0, atom_row(br, k0, KS));
                tma_load_2d_pair(sSF + 1024, &g.msb1, bar, 0, atom_row(br, k0, KS));
            } else if constexpr (OP == OP_FWD2 || OP == OP_BWD2) {
                const int ar = row0 + a_shift, k0 = kb * BK8;
                const int br = OP == OP_FWD2 ? ti.e * g.H + ti.nt * BN : ti.e * g.F + ti.nt * BN;
                tma_load_2d_pair(sA, &g.a0, bar, k0, ar);
                tma_load_2d_pair(sB, &g.b0, bar, k0, br + 128 * rank);
                tma_load_2d_pair(sSF, &g.msa0, bar, 0, atom_row(ar, k0, KS));
                tma_load_2d_pair(sSF + 512, &g.msb0, bar, 0, atom_row(br, k0, KS));
                tma_load_2d_pair(sSF + 1024, &g.msb0, bar, 0, atom_row(br + 128, k0, KS));
            } else if constexpr (OP == OP_BWD1) {
                const int kf = g.F / BK8;
                const bool second = kb >= kf;
                const int k0 = (second ? kb - kf : kb) * BK8;
                const int ar = row0 + a_shift, br = ti.e * g.H + ti.nt * BN;
                const CUtensorMap *msb = second ? &g.msb1 : &g.msb0;
                tma_load_2d_pair(sA, second ? &g.a1 : &g.a0, bar, k0, ar);
                tma_load_2d_pair(sB, second ? &g.b1 : &g.b0, bar, k0, br + 128 * rank);
                tma_load_2d_pair(sSF, second ? &g.msa1 : &g.msa0, bar, 0, atom_row(ar, k0, KS));
                tma_load_2d_pair(sSF + 512, msb, bar, 0, atom_row(br, k0, KS));
                tma_load_2d_pair(sSF + 1024, msb, bar, 0, atom_row(br + 128, k0, KS));
            } else if constexpr (OP == OP_WG2) {
                // A = (w h)^T [F][rows], B = dY^T [H][rows], both quantised along rows
                const int n0 = ti.nt * BN;
                tma_load_2d_pair(sA, &g.a0, bar, krow, m0);
                tma_load_2d_pair(sB, &g.b0, bar, krow, n0 + 128 * rank);
                tma_load_2d_pair(sSF, &g.msa0, bar, 0, atom_row(m0, krow, KS));
                tma_load_2d_pair(sSF + 512, &g.msb0, bar, 0, atom_row(n0, krow, KS));
                tma_load_2d_pair(sSF + 1024, &g.msb0, bar, 0, atom_row(n0 + 128, krow, KS));
            } else if constexpr (OP == OP_WG13) {
                // A = X^T [H][rows], B = [da^T | db^T] [F][rows]: rank 0 loads da, rank 1 db
                const int n0 = ti.nt * 128;
                tma_load_2d_pair(sA, &g.a0, bar, krow, m0);
                tma_load_2d_pair(sB, rank == 0 ? &g.b0 : &g.b1, bar, krow, n0);
                tma_load_2d_pair(sSF, &g.msa0, bar, 0, atom_row(m0, krow, KS));
                tma_load_2d_pair(sSF + 512, &g.msb0, bar, 0, atom_row(n0, krow, KS));
                tma_load_2d_pair(sSF + 1024, &g.msb1, bar, 0, atom_row(n0, krow, KS));
            }
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == P8_STAGES) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok && rank == 0) {
        for (int s = 0; s < P8_STAGES; ++s) {
            if (!((issued >> s) & 1u)) continue;
            const uint32_t bar = smem_u32(&c.full[s]);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, (last_phase >> s) & 1u) && globaltimer_ns() - t0 < ctl.budget_ns) {}
        }
    }
}

__device__ __forceinline__ void tmem_cp_pair_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

template <int OP>
__device__ void pair8_mma_loop(const GemmArgs &g, Pair8Ctl &c, uint8_t *tiles, uint32_t tmem, const WaitCtl &ctl) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    const int total = num_tiles<OP>(c, g);
    for (int t = blockIdx.x / 2; t < total; t += gridDim.x / 2) {
        TileInfo ti = decode_tile<OP, true, 2 * BM>(c, g, t);
        if (!mbar_wait(smem_u32(&c.tempty[0]), acc_phase ^ 1, ctl)) break;   // single accumulator
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < ti.nk; ++kb) {
            if (!mbar_wait(smem_u32(&c.full[stage]), phase, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sA = smem_u32(tiles + stage * P8_STAGE);
            const uint32_t sB = sA + P8_TILE;
            const uint32_t sSF = sB + P8_TILE;
            const uint32_t t_sf = tmem + 256 + 16 * stage;
            tmem_cp_pair_32x128b_x4(t_sf, sdesc_plain(sSF, 0, 128));
            tmem_cp_pair_32x128b_x4(t_sf + 8, sdesc_plain(sSF + 512, 0, 128));
            tmem_cp_pair_32x128b_x4(t_sf + 12, sdesc_plain(sSF + 1024, 0, 128));
#pragma unroll
            for (int kk = 0; kk < BK8 / 32; ++kk) {
                const uint64_t ad = sdesc_sw128(sA + kk * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(sB + kk * 32, 16, 1024);
                mma_mxf8_pair(tmem, ad, bd, idesc_mxf8(2 * BM, BN, kk), t_sf, t_sf + 8, (kb | kk) != 0);
            }
            mma_commit_pair_mc(smem_u32(&c.empty[stage]));   // frees the stage in both CTAs
            if (++stage == P8_STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair_mc(smem_u32(&c.tfull[0]));
        acc_phase ^= 1;
    }
    mma_commit_pair(smem_u32(&c.drain));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < ctl.budget_ns) {}
}

template <int OP>
__global__ void __launch_bounds__(320, 1) pair8_gemm_kernel(const __grid_constant__ GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *staging = tiles + P8_STAGES * P8_STAGE;                    // 4 epilogue warps x 2 x 2 KB
    Pair8Ctl &c = *reinterpret_cast<Pair8Ctl *>(staging + P8_STAGING);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    WaitCtl ctl{g.status, g.budget_ns};
    if (threadIdx.x == 0) {
        for (int s = 0; s < P8_STAGES; ++s) {
            mbar_init(smem_u32(&c.full[s]), 2);      // one arrive.expect_tx per CTA of the pair
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&c.tfull[a]), 1);
            mbar_init(smem_u32(&c.tempty[a]), 256);  // 128 epilogue threads of each CTA
        }
        mbar_init(smem_u32(&c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&g.a0);
        tma_prefetch_map(&g.b0);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&c.tmem_base), 512);
        tmem_relinquish_pair();
    }
    pdl_wait();
    if (threadIdx.x == 0) init_tile_table<OP, 2 * BM>(c, g);
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = c.tmem_base;
    if (warp == 0) {
        if (lane == 0) pair8_producer_loop<OP>(g, c, tiles, ctl);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) pair8_mma_loop<OP>(g, c, tiles, tmem, ctl);
    } else if (warp < 6) {
        if constexpr (OP == OP_FWD1) {
            if (g.fused) gather_loop<true>(g, g.m, g.ready, &c.tfull[0]);   // until the first accumulator is ready
        }
        epilogue_loop<OP, true, true>(g, c, c.tfull, c.tempty, tmem, ctl, staging);
    } else {
        if constexpr (OP == OP_FWD1) gather_loop<true>(g, g.m, g.ready);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // the leader's MMAs are drained before the pair frees TMEM
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

template <int OP>
cudaError_t launch_pair8(const GemmArgs &g, int grid, cudaStream_t stream) {
    constexpr size_t smem = P8_STAGES * P8_STAGE + P8_STAGING + sizeof(Pair8Ctl) + 1024;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t err = cudaFuncSetAttribute(pair8_gemm_kernel<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const bool fused = OP == OP_FWD1 && g.fused;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(fused ? 320 : 192);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    static std::atomic<int> max_clusters[kMaxCachedDevices][2];
    cfg.gridDim = dim3(grid / 2 * 2);
    const int mc = cached_max_clusters(max_clusters, fused ? 1 : 0, pair8_gemm_kernel<OP>, cfg, grid / 2);
    cfg.gridDim = dim3(2 * std::min(grid / 2, mc));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, pair8_gemm_kernel<OP>, g);
}

template <int OP, bool FP8>
cudaError_t launch_op(const GemmArgs &g, int grid, cudaStream_t stream) {
    constexpr size_t smem = STAGES * stage_stride<FP8>() + staging_bytes<OP, FP8>() + sizeof(SmemCtl) + 1024;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t err =
        cudaFuncSetAttribute(grouped_gemm_kernel<OP, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(grouped_gemm_kernel<OP, FP8>, dim3(grid), dim3(((OP == OP_FWD1 && g.fused) || OP == OP_BWD2) ? 320 : 192),
                      smem, stream, g);
}

template <bool FP8>
cudaError_t launch_any(int op, const GemmArgs &g, int grid, cudaStream_t stream) {
    switch (op) {
        case OP_FWD1: return launch_op<OP_FWD1, FP8>(g, grid, stream);
        case OP_FWD2: return launch_op<OP_FWD2, FP8>(g, grid, stream);
        case OP_BWD2: return launch_op<OP_BWD2, FP8>(g, grid, stream);
        case OP_BWD1: return launch_op<OP_BWD1, FP8>(g, grid, stream);
        case OP_WG2: return launch_op<OP_WG2, FP8>(g, grid, stream);
        case OP_WG13: return launch_op<OP_WG13, FP8>(g, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

// ======================================================================
// Persistent forward (MegaArgs): one launch of CTA pairs runs the fused dispatch, GEMM1 +
// SwiGLU, GEMM2 and the combine of every macrobatch (article "O MoK do Cursor ...", section 02:
// one persistent kernel per layer whose roles hand work on through GPU-side counters, the ring
// refilled as soon as its readers are done; noticiai.com.br, "O que e": one deterministic
// kernel). Roles per CTA: warp 0 TMA producer, warp 1 MMA issuer (leader CTA), warps 2-5
// epilogue, warps 6-9 dispatch gather and combine. The pairs walk one tile list in order
// (GEMM1 tiles of macrobatch m, then its GEMM2 tiles, then macrobatch m + 1), so GEMM2 tiles
// fill GEMM1's last wave and the next macrobatch's tiles fill GEMM2's. Hand-offs (every wait
// bounded; each waits only on list items earlier than its own, so every wait ends):
//   GEMM1 tile <- its minibatch's rows gathered (ready counters of the fused dispatch)
//   GEMM2 tile <- h of its 128-row block stored by all F/128 GEMM1 n-tiles (hready; every
//                 epilogue warp publishes its own 32 rows, so no barrier joins the warps)
//   gather of m  <- every GEMM1 tile of m - 1 has loaded its x rows (ring x reused; MXFP8)
//   h of m       <- every GEMM2 tile of m - 1 has loaded its h rows (ring h reused)
//   combine of m <- every GEMM2 tile of m has stored its Y rows (the last macrobatch's combine
//                   runs in the combine kernel after this launch, on every warp of the GPU)
//   Y of m       <- the combine of m - 1 has read every Y row (ring Y reused)
// Arithmetic and rounding are those of the one-launch-per-stage forward, so out is the same bytes.

constexpr int MEGA_OP_GEMM1 = 0, MEGA_OP_GEMM2 = 1;

struct MegaTile {
    int op, e, nt, m, g0, seg_end;
};
__device__ __forceinline__ MegaTile mega_tile(const MegaArgs &a, int t) {
    const int4 v = a.tiles[t];
    MegaTile mt;
    mt.g0 = v.x;
    mt.e = v.y & 255;
    mt.nt = (v.y >> 8) & 0xFFFF;
    mt.op = v.y >> 24;
    mt.seg_end = v.z;
    mt.m = v.w;
    return mt;
}

template <bool FP8>
__device__ void mega_producer(const MegaArgs &a, const CtlT<FP8 ? P8_STAGES : PSTAGES> &c, uint8_t *tiles,
                              int total, const WaitCtl &ctl) {
    constexpr int NS = FP8 ? P8_STAGES : PSTAGES;
    constexpr uint32_t SS = FP8 ? P8_STAGE : P_STAGE;
    const GemmArgs &g1 = a.g1, &g2 = a.g2;
    const int rank = (int)cluster_ctarank();
    int stage = 0;
    uint32_t phase = 0, issued = 0, last_phase = 0;
    bool ok = true;
    int ready_m = -1, ready_j = -1;
    for (int t = blockIdx.x / 2; t < total && ok; t += gridDim.x / 2) {
        const MegaTile mt = mega_tile(a, t);
        const int row0 = mt.g0 + BM * rank;          // this CTA's 128 rows
        const bool rows = row0 < mt.seg_end;         // not a half past the run
        const int r0m = g1.offp[mt.m * g1.E];        // first padded row of the macrobatch
        const int hrow = row0 - r0m;                 // ring row (one macrobatch in the ring)
        const int xrow = g1.a_ring ? hrow : row0;    // bf16 keeps x rows at their padded rows
        if (mt.op == MEGA_OP_GEMM1) {
            if (rows) {
                const int j = hrow / g1.mb_rows;
                if (mt.m != ready_m || j != ready_j) {
                    const int need = min(g1.mb_rows, g1.offp[(mt.m + 1) * g1.E] - r0m - j * g1.mb_rows);
                    if (!flag_wait_geq(g1.ready + (size_t)mt.m * a.ready_stride + j, need, ctl)) { ok = false; break; }
                    fence_proxy_async_global();
                    ready_m = mt.m;
                    ready_j = j;
                }
            }
        } else if (rows) {
            // four epilogue warps publish each of the F/128 GEMM1 n-tiles of the block
            if (!flag_wait_geq(a.hready + row0 / BM, 4 * (g1.F / 128), ctl)) { ok = false; break; }
            fence_proxy_async_global();
        }
        const int nk = mt.op == MEGA_OP_GEMM1 ? g1.K / bk_elems<FP8>() : g2.K / bk_elems<FP8>();
        for (int kb = 0; kb < nk; ++kb) {
            if (!mbar_wait(smem_u32(&c.empty[stage]), phase ^ 1, ctl)) { ok = false; break; }
            const uint32_t bar = mapa_shared(smem_u32(&c.full[stage]), 0);   // the leader's full barrier
            const uint32_t sA = smem_u32(tiles + stage * SS);
            if constexpr (!FP8) {
                const uint32_t sB = sA + P_A_BYTES;
                mbar_arrive_expect_tx_cluster(bar, P_STAGE);
                if (mt.op == MEGA_OP_GEMM1) {
                    tma_load_2d_pair(sA, &g1.a0, bar, kb * BK, xrow);
                    tma_load_3d_pair(sB, rank == 0 ? &g1.b0 : &g1.b1, bar, 0, mt.e * g1.H + kb * BK, mt.nt * 2);
                } else {
                    tma_load_2d_pair(sA, &g2.a0, bar, kb * BK, hrow);
                    tma_load_3d_pair(sB, &g2.b0, bar, 0, mt.e * g2.F + kb * BK, (mt.nt * BN + 128 * rank) / 64);
                }
            } else {
                const uint32_t sB = sA + P8_TILE, sSF = sB + P8_TILE;
                mbar_arrive_expect_tx_cluster(bar, P8_TX);
                const int k0 = kb * BK8;
                if (mt.op == MEGA_OP_GEMM1) {
                    const int br = mt.e * g1.F + mt.nt * 128, KS = g1.kstore;
                    tma_load_2d_pair(sA, &g1.a0, bar, k0, xrow);
                    tma_load_2d_pair(sB, rank == 0 ? &g1.b0 : &g1.b1, bar, k0, br);   // W1^T half, W3^T half
                    tma_load_2d_pair(sSF, &g1.msa0, bar, 0, atom_row(xrow, k0, KS));
                    tma_load_2d_pair(sSF + 512, &g1.msb0, bar, 0, atom_row(br, k0, KS));
                    tma_load_2d_pair(sSF + 1024, &g1.msb1, bar, 0, atom_row(br, k0, KS));
                } else {
                    const int br = mt.e * g2.H + mt.nt * BN, KS = g2.kstore;
                    tma_load_2d_pair(sA, &g2.a0, bar, k0, hrow);
                    tma_load_2d_pair(sB, &g2.b0, bar, k0, br + 128 * rank);
                    tma_load_2d_pair(sSF, &g2.msa0, bar, 0, atom_row(hrow, k0, KS));
                    tma_load_2d_pair(sSF + 512, &g2.msb0, bar, 0, atom_row(br, k0, KS));
                    tma_load_2d_pair(sSF + 1024, &g2.msb0, bar, 0, atom_row(br + 128, k0, KS));
                }
            }
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == NS) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok && rank == 0) {
        // the leader's full barriers count both CTAs' copies: wait (bounded) for the last phases
        for (int s = 0; s < NS; ++s) {
            if (!((issued >> s) & 1u)) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&c.full[s]), (last_phase >> s) & 1u) && globaltimer_ns() - t0 < ctl.budget_ns) {}
        }
    }
}

template <bool FP8>
__device__ void mega_mma(const MegaArgs &a, CtlT<FP8 ? P8_STAGES : PSTAGES> &c, uint8_t *tiles, uint32_t tmem,
                         int total, const WaitCtl &ctl) {
    constexpr int NS = FP8 ? P8_STAGES : PSTAGES;
    constexpr uint32_t SS = FP8 ? P8_STAGE : P_STAGE;
    constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, false, true);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int t = blockIdx.x / 2; t < total; t += gridDim.x / 2) {
        const MegaTile mt = mega_tile(a, t);
        const int nk = mt.op == MEGA_OP_GEMM1 ? a.g1.K / bk_elems<FP8>() : a.g2.K / bk_elems<FP8>();
        if (!mbar_wait(smem_u32(&c.tempty[acc]), acc_phase ^ 1, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            if (!mbar_wait(smem_u32(&c.full[stage]), phase, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sA = smem_u32(tiles + stage * SS);
            if constexpr (!FP8) {
                const uint32_t sB = sA + P_A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16_pair(d, sdesc_sw128(sA + kk * 32, 16, 1024), sdesc_sw128(sB + kk * 2048, 8192, 1024), idesc,
                                  (kb | kk) != 0);
            } else {
                const uint32_t sB = sA + P8_TILE, sSF = sB + P8_TILE;
                const uint32_t t_sf = tmem + 256 + 16 * stage;
                tmem_cp_pair_32x128b_x4(t_sf, sdesc_plain(sSF, 0, 128));
                tmem_cp_pair_32x128b_x4(t_sf + 8, sdesc_plain(sSF + 512, 0, 128));
                tmem_cp_pair_32x128b_x4(t_sf + 12, sdesc_plain(sSF + 1024, 0, 128));
#pragma unroll
                for (int kk = 0; kk < BK8 / 32; ++kk)
                    mma_mxf8_pair(tmem, sdesc_sw128(sA + kk * 32, 16, 1024), sdesc_sw128(sB + kk * 32, 16, 1024),
                                  idesc_mxf8(2 * BM, BN, kk), t_sf, t_sf + 8, (kb | kk) != 0);
            }
            mma_commit_pair_mc(smem_u32(&c.empty[stage]));   // frees the stage in both CTAs
            if (++stage == NS) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        // every copy of this tile has landed: its source rows in the ring may be overwritten
        fence_proxy_async_global();
        red_release_gpu_add(a.cnt + (size_t)mt.m * MEGA_NCNT + (mt.op == MEGA_OP_GEMM1 ? MEGA_G1_READ : MEGA_G2_READ), 1);
        mma_commit_pair_mc(smem_u32(&c.tfull[acc]));
        if constexpr (FP8) {
            acc_phase ^= 1;                 // single accumulator (scale atoms in TMEM columns 256+)
        } else {
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }
    mma_commit_pair(smem_u32(&c.drain));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < ctl.budget_ns) {}
}

template <bool FP8>
__device__ void mega_epilogue(const MegaArgs &a, CtlT<FP8 ? P8_STAGES : PSTAGES> &c, uint32_t tmem, int total,
                              const WaitCtl &ctl, uint8_t *staging) {
    constexpr int NBUF = FP8 ? 2 : 4;   // 2 KB staging buffers per warp
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3, r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int rank = (int)cluster_ctarank();
    const GemmArgs &g1 = a.g1, &g2 = a.g2;
    int acc = 0, store_chunks = 0;
    uint32_t acc_phase = 0;
    uint8_t *warp_stage = staging ? staging + (warp - 2) * (NBUF * 2048) : nullptr;
    int h_free = 0, y_free = 0;   // macrobatches whose ring h / Y rows may be written
    // A tile's rows are published one tile late: after the next tile's stores are issued, lane
    // 0 waits only for the older bulk groups, whose writes have had a tile's time to land. A
    // pending publication is flushed before any wait that could block, so no wait of this
    // warp ever depends on a publication it still holds.
    int *pending = nullptr;
    auto flush = [&]() {
        if (pending == nullptr) return;
        __threadfence();
        __syncwarp();
        if (lane == 0) {
            bulk_wait_group_all();
            fence_proxy_async_global();
            __threadfence();
            red_release_gpu_add(pending, 1);
        }
        __syncwarp();
        pending = nullptr;
    };
    for (int t = blockIdx.x / 2; t < total; t += gridDim.x / 2) {
        const MegaTile mt = mega_tile(a, t);
        TileInfo ti;
        ti.e = mt.e; ti.nt = mt.nt; ti.mt = 0; ti.nk = 0;
        ti.g0 = mt.g0 + BM * rank;
        ti.seg_end = mt.seg_end;
        const bool rows = ti.g0 < ti.seg_end;
        const int ring_shift = -g1.offp[mt.m * g1.E];
        // the ring rows this tile writes must be done with by the previous macrobatch's readers
        if (mt.op == MEGA_OP_GEMM1 && mt.m > h_free) {
            flush();
            const int p = mt.m - 1;
            if (!flag_wait_geq(a.cnt + (size_t)p * MEGA_NCNT + MEGA_G2_READ, a.meta[p * 4 + 1], ctl)) break;
            h_free = mt.m;
        }
        if (mt.op == MEGA_OP_GEMM2 && mt.m > y_free) {
            flush();
            const int p = mt.m - 1;
            if (!flag_wait_geq(a.cnt + (size_t)p * MEGA_NCNT + MEGA_COMBINED, a.meta[p * 4 + 3], ctl)) break;
            y_free = mt.m;
        }
        if (!mbar_try_wait(smem_u32(&c.tfull[acc]), acc_phase)) flush();   // about to wait: publish first
        if (!mbar_wait(smem_u32(&c.tfull[acc]), acc_phase, ctl)) break;
        tc_fence_after();
        const uint32_t tbase = tmem + lane_base + acc * BN;
        if (rows) {
            if (mt.op == MEGA_OP_GEMM1)
                epi_fwd1_tile<FP8, NBUF>(g1, ti, tbase, r, quarter, lane, ring_shift, !FP8 && g1.tma_store, warp_stage,
                                         store_chunks);
            else
                // MXFP8 Y rows straight from registers: the staged TMA store's chain (staging wait,
                // proxy fence, warp sync) held up the single accumulator longer
                epi_rows_tile<OP_FWD2, NBUF>(g2, ti, tbase, r, quarter, lane, ring_shift, !FP8 && g2.tma_store != 0,
                                             warp_stage, store_chunks);
        }
        tc_fence_before();
        mbar_arrive_cluster(mapa_shared(smem_u32(&c.tempty[acc]), 0));   // the leader's MMA thread waits for both CTAs
        // publish the previous tile's rows (its bulk groups are older than this tile's: wait for
        // all but this tile's), then hold this tile's. Each warp publishes its own 32 rows (it
        // writes no other), so no barrier joins the warps; the counters' targets count four per tile.
        if (pending != nullptr) {
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                if (!rows) bulk_wait_group_all();
                else if (mt.op == MEGA_OP_GEMM1 && FP8) bulk_wait_group_all();          // no bulk stores
                else if (mt.op == MEGA_OP_GEMM1) bulk_wait_group<12>();                 // a, b, h x 4 chunks
                else bulk_wait_group<BN / 32>();                                        // Y: 8 chunks
                fence_proxy_async_global();
                __threadfence();
                red_release_gpu_add(pending, 1);
            }
            __syncwarp();
            pending = nullptr;
        }
        if (rows)
            pending = mt.op == MEGA_OP_GEMM1 ? a.hready + ti.g0 / BM : a.cnt + (size_t)mt.m * MEGA_NCNT + MEGA_Y_DONE;
        if constexpr (FP8) {
            acc_phase ^= 1;
        } else {
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }
    flush();
    if (store_chunks > 0 && lane == 0) bulk_wait_group_all();
}

// warps 6-9: gather macrobatch m, then combine macrobatch m - 1 while later macrobatches run.
// The last macrobatch's combine has nothing left to overlap with: the combine kernel that
// follows this launch does it with every warp of the GPU.
template <bool FP8>
__device__ void mega_gather_combine(const MegaArgs &a, const WaitCtl &ctl) {
    const GemmArgs &g1 = a.g1;
    const int lane = threadIdx.x % 32;
    const int gw = blockIdx.x * 4 + (threadIdx.x / 32 - 6), nw = gridDim.x * 4;
    CombineArgs ca{};
    ca.Y = a.g2.o0; ca.slot_row = a.slot_row; ca.offp = g1.offp; ca.w = a.w; ca.out = a.out;
    ca.k = g1.k; ca.H = g1.H; ca.E = g1.E; ca.ring_base = 0; ca.status = g1.status;
    const int nch = (g1.H / 8 + 63) / 64;
    for (int m = 0; m < g1.nM; ++m) {
        {
            // ring x rows free: every GEMM1 tile of m - 1 has loaded its rows (bf16 keeps the
            // x rows at their own padded rows in the saved context: nothing is reused)
            if (m > 0 && g1.a_ring &&
                !flag_wait_geq(a.cnt + (size_t)(m - 1) * MEGA_NCNT + MEGA_G1_READ, a.meta[(m - 1) * 4 + 0], ctl))
                return;
            gather_loop<FP8>(g1, m, g1.ready + (size_t)m * a.ready_stride);
        }
        if (m > 0 && m < g1.nM) {
            const int p = m - 1;
            if (!flag_wait_geq(a.cnt + (size_t)p * MEGA_NCNT + MEGA_Y_DONE, a.meta[p * 4 + 2], ctl)) return;
            ca.t0 = p * a.Mb;
            ca.t1 = min(a.T, ca.t0 + a.Mb);
            ca.m = p;
            const int lo = g1.offp[p * g1.E], hi = g1.offp[(p + 1) * g1.E];
            const int shift = -lo;
            const int items = a.meta[p * 4 + 3];
            (void)gw; (void)nw;
            for (;;) {
                int it = 0;
                if (lane == 0) it = atomicAdd(a.cnt + (size_t)p * MEGA_NCNT + MEGA_COMBINE_CLAIM, 1);
                it = __shfl_sync(0xffffffffu, it, 0);
                if (it >= items) break;
                combine_item(ca, it, nch, shift, lo, hi, lane);
                __threadfence();
                __syncwarp();
                if (lane == 0) red_release_gpu_add(a.cnt + (size_t)p * MEGA_NCNT + MEGA_COMBINED, 1);
            }
        }
    }
}

template <bool FP8>
__global__ void __launch_bounds__(320, 1) fwd_mega_kernel(const __grid_constant__ MegaArgs a) {
    using Ctl = CtlT<FP8 ? P8_STAGES : PSTAGES>;
    constexpr int NS = FP8 ? P8_STAGES : PSTAGES;
    constexpr uint32_t SS = FP8 ? P8_STAGE : P_STAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *staging = tiles + NS * SS;
    Ctl &c = *reinterpret_cast<Ctl *>(tiles + NS * SS + (FP8 ? P8_STAGING : P_STAGING));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    WaitCtl ctl{a.g1.status, a.g1.budget_ns};
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&c.full[s]), 2);      // one arrive.expect_tx per CTA of the pair
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&c.tfull[i]), 1);
            mbar_init(smem_u32(&c.tempty[i]), 256);  // 128 epilogue threads of each CTA
        }
        mbar_init(smem_u32(&c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&a.g1.a0);
        tma_prefetch_map(&a.g1.b0);
        tma_prefetch_map(&a.g2.a0);
        tma_prefetch_map(&a.g2.b0);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&c.tmem_base), 512);
        tmem_relinquish_pair();
    }
    pdl_wait();   // the schedule, the tile list and the zeroed counters are in place
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = c.tmem_base;
    const int total = *a.tile_count;
    if (warp == 0) {
        if (lane == 0) mega_producer<FP8>(a, c, tiles, total, ctl);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) mega_mma<FP8>(a, c, tiles, tmem, total, ctl);
    } else if (warp < 6) {
        // the epilogue warps gather the first macrobatch too, until their first accumulator is ready
        gather_loop<FP8>(a.g1, 0, a.g1.ready, &c.tfull[0]);
        mega_epilogue<FP8>(a, c, tmem, total, ctl, staging);
    } else {
        mega_gather_combine<FP8>(a, ctl);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // the leader's MMAs are drained before the pair frees TMEM
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// One block per macrobatch m, one thread per expert: the pair m-tiles of every earlier
// macrobatch place m's entries; GEMM1 tiles (expert-major, m-tile, n-tile), then GEMM2 tiles.
__global__ void __launch_bounds__(64) mega_list_kernel(const int *offp, int E, int nM, int nt1, int nt2, int T,
                                                       int Mb, int nch, int4 *list, int *meta, int *count) {
    pdl_wait();
    __shared__ int s_n[64], s_before[64];
    const int m = blockIdx.x, e = threadIdx.x;
    int before = 0, s0 = 0, s1 = 0;
    if (e < E) {
        for (int mm = 0; mm < m; ++mm) before += (offp[mm * E + e + 1] - offp[mm * E + e] + 255) / 256;
        s0 = offp[m * E + e];
        s1 = offp[m * E + e + 1];
    }
    const int nmt = (s1 - s0 + 255) / 256;
    s_n[e] = nmt;
    s_before[e] = before;
    __syncthreads();
    int pref = 0, total_mt = 0, total_before = 0;
    for (int i = 0; i < E; ++i) {
        if (i < e) pref += s_n[i];
        total_mt += s_n[i];
        total_before += s_before[i];
    }
    const int base = total_before * (nt1 + nt2);
    const int base2 = base + total_mt * nt1;
    if (e < E) {
        for (int mt = 0; mt < nmt; ++mt) {
            for (int nt = 0; nt < nt1; ++nt)
                list[base + (pref + mt) * nt1 + nt] = make_int4(s0 + 256 * mt, e | (nt << 8) | (MEGA_OP_GEMM1 << 24), s1, m);
            for (int nt = 0; nt < nt2; ++nt)
                list[base2 + (pref + mt) * nt2 + nt] = make_int4(s0 + 256 * mt, e | (nt << 8) | (MEGA_OP_GEMM2 << 24), s1, m);
        }
    }
    if (e == 0) {
        meta[m * 4 + 0] = total_mt * nt1;
        meta[m * 4 + 1] = total_mt * nt2;
        meta[m * 4 + 2] = (offp[(m + 1) * E] - offp[m * E]) / 128 * nt2 * 4;   // one per epilogue warp
        const int t0 = m * Mb, t1 = min(T, t0 + Mb);
        meta[m * 4 + 3] = (t1 - t0) * nch;
        if (m == nM - 1) *count = base + total_mt * (nt1 + nt2);
    }
}

// One warp. The 128-row list: runs are taken 32 at a time in expert-major order (run i =
// expert i / nM, macrobatch i % nM); a warp scan of their chunk counts places each lane's
// chunks after those of the runs before it, and the first chunk of each expert is noted.
// The pair list then takes each expert's chunks two at a time, in the same order.
__global__ void __launch_bounds__(32) tile_list_kernel(const int *offp, int E, int nM, int4 *list128,
                                                        int4 *list256, int *counts) {
    __shared__ int ebase[kMaxExperts + 1];   // first list128 entry of each expert
    pdl_wait();
    const int lane = threadIdx.x;
    const int nseg = E * nM;
    int base = 0;
    for (int i0 = 0; i0 < nseg; i0 += 32) {
        const int i = i0 + lane;
        int s0 = 0, s1 = 0, e = 0, m = 0;
        if (i < nseg) {
            e = i / nM;
            m = i - e * nM;
            s0 = offp[m * E + e];
            s1 = offp[m * E + e + 1];
        }
        const int n = (s1 - s0 + BM - 1) / BM;
        int incl = n;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        const int start = base + incl - n;
        if (i < nseg && m == 0) ebase[e] = start;
        for (int j = 0; j < n; ++j) list128[start + j] = make_int4(s0 + j * BM, e, s1, 0);
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        ebase[E] = base;
        counts[0] = base;
    }
    __syncwarp();
    __threadfence_block();   // list128 and ebase of every lane, seen by every lane
    __syncwarp();
    int pbase = 0;
    for (int e = 0; e < E; ++e) {
        const int c0 = ebase[e], n = ebase[e + 1] - c0, pairs = (n + 1) / 2;
        for (int p = lane; p < pairs; p += 32) {
            const int r1 = 2 * p + 1 < n ? list128[c0 + 2 * p + 1].x : -1;
            list256[pbase + p] = make_int4(list128[c0 + 2 * p].x, e, r1, 0);
        }
        pbase += pairs;
    }
    if (lane == 0) counts[1] = pbase;
}

}  // namespace

cudaError_t launch_mega_list(const int *offp, int E, int nM, int F, int H, int T, int Mb, int4 *list, int *meta,
                             int *count, cudaStream_t stream) {
    return launch_pdl(mega_list_kernel, dim3(nM), dim3(64), 0, stream, offp, E, nM, F / 128, H / BN, T, Mb,
                      (H / 8 + 63) / 64, list, meta, count);
}

template <bool FP8>
cudaError_t launch_mega_t(const MegaArgs &a, int grid, cudaStream_t stream) {
    constexpr size_t smem = FP8 ? P8_STAGES * P8_STAGE + P8_STAGING + sizeof(Pair8Ctl) + 1024
                                : PSTAGES * P_STAGE + P_STAGING + sizeof(PairCtl) + 1024;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    static_assert(sizeof(MegaArgs) <= 32764, "kernel parameter space");
    cudaError_t err = cudaFuncSetAttribute(fwd_mega_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(320);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // every CTA waits on others' progress: the grid must be fully co-resident
    static std::atomic<int> max_clusters[kMaxCachedDevices][2];
    cfg.gridDim = dim3(grid / 2 * 2);
    const int mc = cached_max_clusters(max_clusters, 0, fwd_mega_kernel<FP8>, cfg, grid / 2);
    cfg.gridDim = dim3(2 * std::min(grid / 2, mc));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fwd_mega_kernel<FP8>, a);
}

cudaError_t launch_fwd_mega(const MegaArgs &a, int grid, cudaStream_t stream, bool fp8) {
    return fp8 ? launch_mega_t<true>(a, grid, stream) : launch_mega_t<false>(a, grid, stream);
}

cudaError_t launch_tile_lists(const int *offp, int E, int nM, int4 *list128, int4 *list256, int *counts,
                              cudaStream_t stream) {
    return launch_pdl(tile_list_kernel, dim3(1), dim3(32), 0, stream, offp, E, nM, list128, list256, counts);
}

cudaError_t launch_grouped_gemm(int op, const GemmArgs &g, int grid, cudaStream_t stream, bool fp8, bool pair) {
    if (pair && fp8) {
        switch (op) {
            case OP_FWD1: return launch_pair8<OP_FWD1>(g, grid, stream);
            case OP_FWD2: return launch_pair8<OP_FWD2>(g, grid, stream);
            case OP_BWD2: return launch_pair8<OP_BWD2>(g, grid, stream);
            case OP_BWD1: return launch_pair8<OP_BWD1>(g, grid, stream);
            case OP_WG2: return launch_pair8<OP_WG2>(g, grid, stream);
            case OP_WG13: return launch_pair8<OP_WG13>(g, grid, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    if (pair && !fp8 && op != OP_BWD2) {   // BWD2: heavy epilogue, phantom halves; 1-CTA tiles
        switch (op) {
            case OP_FWD1: return launch_pair<OP_FWD1>(g, grid, stream);
            case OP_FWD2: return launch_pair<OP_FWD2>(g, grid, stream);
            case OP_BWD2: return launch_pair<OP_BWD2>(g, grid, stream);
            case OP_BWD1: return launch_pair<OP_BWD1>(g, grid, stream);
            case OP_WG2: return launch_pair<OP_WG2>(g, grid, stream);
            case OP_WG13: return launch_pair<OP_WG13>(g, grid, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    return fp8 ? launch_any<true>(op, g, grid, stream) : launch_any<false>(op, g, grid, stream);
}

}  // namespace moe
