// Decode-shaped expert FFN on tcgen05 tensor cores: the forward of few tokens.
//
// With few tokens ("warp decode" in Cursor's earlier work, noticiai.com.br, "Por que a camada
// MoE virou o gargalo") each expert holds a handful of routed rows and the layer's time is
// the weights' trip from HBM: every byte of W1, W3 and W2 has to be read once and there is
// little arithmetic to hide it behind. The row tiles of the grouped GEMMs (128 or 256 rows)
// would be almost empty, so here the roles swap: the weights are the M operand (128 of their
// columns per tile, MN-major, straight from the row-major weights) and the expert's routed
// rows (at most 128, zero-padded) are N:
//   GEMM1 item (expert e, 128 columns f of F): D_a[f][r] = sum_h W1[e][h][f] x[r][h], D_b
//     likewise with W3; epilogue: a, b rounded to bf16 (saved for the backward, 32 x 32 blocks),
//     h = silu(a) * b rounded to bf16 into the h rows;
//   GEMM2 item (expert e, 128 columns of H): D_y[c][r] = sum_f W2[e][f][c] h[r][f]; epilogue:
//     y rows in bf16 for the combine.
// One persistent CTA per SM (192 threads): warp 0 claims work items from a device counter
// (every GEMM1 item first, then every GEMM2 item; items of experts without rows are skipped)
// and streams their operands by TMA through a ring of 36-48 KB stages (32 KB of weights and
// the expert's token rows in 32-row boxes; 4-6 stages, the more the fewer tokens); warp 1
// issues the MMAs (M = 128, N = the expert's rows rounded up to 32, K = 16) into a
// double-buffered TMEM accumulator (256 columns per item); warps 2-5 run the epilogues. A GEMM2 item waits (bounded, acquire) until all F/128
// GEMM1 items of its expert have published h (release), so GEMM2 tiles of early experts run
// while GEMM1 tiles of late ones still stream, and no SM idles at a phase boundary. Items
// are claimed in order and GEMM1 items wait on nothing, so every wait ends.
#include <cuda_fp16.h>

#include "decode_ffn.cuh"
#include "nvfp4.cuh"

namespace moe {

namespace {

constexpr int DST_MAX = 8;                           // pipeline stages (at most)
constexpr uint32_t DW_TILE = 2 * 64 * 64 * 2;        // 16 KB: 128 weight columns x 64 K rows, MN-major
constexpr uint32_t DT_BOX = 32 * 64 * 2;             // 4 KB: 32 token rows x 64 K, K-major
constexpr uint32_t DSMEM = 216 * 1024;               // shared memory for the stages
constexpr int QD = 4;                                // depth of the work-item queue in shared memory

// Stage layout for a launch: W1 (or W2) tile, W3 tile, then nb boxes of 32 token rows, where
// nb = ceil(T / 32) covers the most rows an expert can hold; fewer token rows per stage leave
// room for more stages, i.e. more weight bytes in flight per SM.
__host__ __device__ constexpr uint32_t dec_stage_bytes(int nb) { return 2 * DW_TILE + nb * DT_BOX; }
__host__ __device__ constexpr int dec_stages(int nb) {
    return (int)(DSMEM / dec_stage_bytes(nb)) < DST_MAX ? (int)(DSMEM / dec_stage_bytes(nb)) : DST_MAX;
}

struct DecCtl {
    uint64_t full[DST_MAX], empty[DST_MAX], tfull[2], tempty[2], qfull[QD], qempty[QD], drain;
    uint32_t tmem_base;
    int item[QD];
};

// element (row, col) of a [rows][C] matrix stored in 32 x 32 blocks (blk32_offset)
__device__ __forceinline__ size_t blk32_elem(int row, int col, int C) {
    return blk32_offset(row, col, C) + (size_t)((((col & 31) >> 3) * 32 + (row & 31)) * 8 + (col & 7));
}

__device__ __forceinline__ float sigmoid_d(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }

struct Item {
    bool gemm1;
    int e, col0, nk;
};

__device__ __forceinline__ Item decode_item(const DecodeArgs &a, int id) {
    const int nf = a.F / 128, n1 = a.E * nf;
    Item it;
    it.gemm1 = id < n1;
    if (it.gemm1) {
        it.e = id / nf;
        it.col0 = (id - it.e * nf) * 128;
        it.nk = a.H / 64;
    } else {
        const int nh = a.H / 128, q = id - n1;
        it.e = q / nh;
        it.col0 = (q - it.e * nh) * 128;
        it.nk = a.F / 64;
    }
    return it;
}

__device__ void dec_producer(const DecodeArgs &a, DecCtl &c, uint8_t *tiles, const WaitCtl &ctl) {
    const int total = a.E * (a.F / 128 + a.H / 128);
    const int DST = dec_stages(a.nb);
    const uint32_t DSTAGE = dec_stage_bytes(a.nb);
    int stage = 0, slot = 0;
    uint32_t phase = 0, qphase = 0;
    uint32_t issued = 0, last_phase = 0;
    bool ok = true;
    for (;;) {
        int id = -1;
        if (ok) {
            for (;;) {
                id = atomicAdd(a.claim, 1);
                if (id >= total) { id = -1; break; }
                if (a.counts[decode_item(a, id).e] > 0) break;   // experts without rows have no work
            }
        }
        if (!mbar_wait(smem_u32(&c.qempty[slot]), qphase ^ 1, ctl)) { ok = false; id = -1; }
        c.item[slot] = id;
        mbar_arrive(smem_u32(&c.qfull[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        const int s0 = a.offp[it.e];
        const int nb = (a.counts[it.e] + 31) / 32;   // 32-row boxes holding the expert's rows
        if (!it.gemm1) {
            // h of this expert: the four epilogue warps of every GEMM1 item of it have published
            if (!flag_wait_geq(a.hdone + it.e, 4 * (a.F / 128), ctl)) { ok = false; continue; }
            fence_proxy_async_global();
        }
        for (int kb = 0; kb < it.nk && ok; ++kb) {
            if (!mbar_wait(smem_u32(&c.empty[stage]), phase ^ 1, ctl)) { ok = false; break; }
            const uint32_t bar = smem_u32(&c.full[stage]);
            const uint32_t sA = smem_u32(tiles + stage * DSTAGE);
            const uint32_t sT = sA + 2 * DW_TILE;
            if (it.gemm1) {
                mbar_arrive_expect_tx(bar, 2 * DW_TILE + nb * DT_BOX);
                tma_load_3d(sA, &a.w1, bar, 0, it.e * a.H + kb * 64, it.col0 / 64);
                tma_load_3d(sA + DW_TILE, &a.w3, bar, 0, it.e * a.H + kb * 64, it.col0 / 64);
                for (int j = 0; j < nb; ++j) tma_load_2d(sT + j * DT_BOX, &a.x, bar, kb * 64, s0 + 32 * j);
            } else {
                mbar_arrive_expect_tx(bar, DW_TILE + nb * DT_BOX);
                tma_load_3d(sA, &a.w2, bar, 0, it.e * a.F + kb * 64, it.col0 / 64);
                for (int j = 0; j < nb; ++j) tma_load_2d(sT + j * DT_BOX, &a.h, bar, kb * 64, s0 + 32 * j);
            }
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == DST) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok) {
        // leave no bulk copy in flight: wait (bounded, regardless of the status word) for the
        // last copy issued into every stage
        for (int s = 0; s < DST; ++s) {
            if (!((issued >> s) & 1u)) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&c.full[s]), (last_phase >> s) & 1u) && globaltimer_ns() - t0 < ctl.budget_ns) {}
        }
    }
}

__device__ void dec_mma(const DecodeArgs &a, DecCtl &c, uint8_t *tiles, uint32_t tmem, const WaitCtl &ctl) {
    const int DST = dec_stages(a.nb);
    const uint32_t DSTAGE = dec_stage_bytes(a.nb);
    int stage = 0, slot = 0, acc = 0;
    uint32_t phase = 0, qphase = 0, acc_phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&c.qfull[slot]), qphase, ctl)) break;
        const int id = c.item[slot];
        mbar_arrive(smem_u32(&c.qempty[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        // N = the expert's rows rounded up to 32 (A MN-major weights, B K-major token rows)
        const uint32_t idesc = idesc_bf16_f32(128, 32 * ((a.counts[it.e] + 31) / 32), true, false);
        if (!mbar_wait(smem_u32(&c.tempty[acc]), acc_phase ^ 1, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256;
        bool ok = true;
        for (int kb = 0; kb < it.nk; ++kb) {
            if (!mbar_wait(smem_u32(&c.full[stage]), phase, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sA = smem_u32(tiles + stage * DSTAGE);
            const uint32_t sT = sA + 2 * DW_TILE;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc_sw128(sT + kk * 32, 16, 1024);
                mma_bf16_ss(d, sdesc_sw128(sA + kk * 2048, 8192, 1024), bd, idesc, (kb | kk) != 0);
                if (it.gemm1) mma_bf16_ss(d + 128, sdesc_sw128(sA + DW_TILE + kk * 2048, 8192, 1024), bd, idesc, (kb | kk) != 0);
            }
            mma_commit(smem_u32(&c.empty[stage]));
            if (++stage == DST) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(smem_u32(&c.tfull[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
    }
    mma_commit(smem_u32(&c.drain));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < ctl.budget_ns) {}
}

__device__ void dec_epilogue(const DecodeArgs &a, DecCtl &c, uint32_t tmem, const WaitCtl &ctl) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;                    // TMEM lanes this warp may read
    const int col = quarter * 32 + lane;             // weight column of this thread within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int slot = 0, acc = 0;
    uint32_t qphase = 0, acc_phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&c.qfull[slot]), qphase, ctl)) break;
        const int id = c.item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c.qempty[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        if (!mbar_wait(smem_u32(&c.tfull[acc]), acc_phase, ctl)) break;
        tc_fence_after();
        const uint32_t tbase = tmem + lane_base + acc * 256;
        const int s0 = a.offp[it.e];
        const int nb = (a.counts[it.e] + 31) / 32;   // 32-row column blocks the MMA computed
        if (it.gemm1) {
            // every row of the expert's 128-row padded run: padding rows have x = 0, so their
            // a, b and h are exactly 0 (the backward reads a, b of the whole run); rows past the
            // computed blocks are written as those zeros
            const int f = it.col0 + col;
#pragma unroll 1
            for (int rc = 0; rc < 4; ++rc) {
                uint32_t va[32], vb[32];
                if (rc < nb) {
                    tmem_ld_32x32b_x32(tbase + rc * 32, va);
                    tmem_ld_32x32b_x32(tbase + 128 + rc * 32, vb);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) va[i] = vb[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int row = s0 + rc * 32 + i;
                    const bf16 ab = f2bf(__uint_as_float(va[i])), bb = f2bf(__uint_as_float(vb[i]));
                    const float av = bf2f(ab), bv = bf2f(bb);
                    a.a[blk32_elem(row, f, a.F)] = ab;
                    a.b[blk32_elem(row, f, a.F)] = bb;
                    a.hrows[(size_t)row * a.F + f] = f2bf(av * sigmoid_d(av) * bv);
                }
            }
        } else {
            const int c0 = it.col0 + col, nrows = a.counts[it.e];
#pragma unroll 1
            for (int rc = 0; rc < 4 && rc * 32 < nrows; ++rc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tbase + rc * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int r = rc * 32 + i;
                    if (r < nrows) a.y[(size_t)(s0 + r) * a.H + c0] = f2bf(__uint_as_float(v[i]));
                }
            }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&c.tempty[acc]));
        if (it.gemm1) {
            // publish: this warp's 32 h columns of expert e are in memory (generic stores, read
            // by later TMA loads of other CTAs); one release per warp, so no barrier joins the
            // warps and a warp that gave up on a wait cannot hold the others
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                fence_proxy_async_global();
                red_release_gpu_add(a.hdone + it.e, 1);
            }
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
    }
}

__global__ void __launch_bounds__(192, 1) decode_ffn_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    DecCtl &c = *reinterpret_cast<DecCtl *>(tiles + DSMEM);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    WaitCtl ctl{a.status, a.budget_ns};
    if (threadIdx.x == 0) {
        for (int s = 0; s < dec_stages(a.nb); ++s) {
            mbar_init(smem_u32(&c.full[s]), 1);
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int q = 0; q < QD; ++q) {
            mbar_init(smem_u32(&c.qfull[q]), 1);
            mbar_init(smem_u32(&c.qempty[q]), 1 + 4);   // the MMA thread and the four epilogue warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&c.tfull[i]), 1);
            mbar_init(smem_u32(&c.tempty[i]), 128);
        }
        mbar_init(smem_u32(&c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&a.w1);
        tma_prefetch_map(&a.w3);
        tma_prefetch_map(&a.w2);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem_base), 512);
        tmem_relinquish();
    }
    pdl_wait();   // the dispatched rows, offsets and counters are in place
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = c.tmem_base;
    if (warp == 0) {
        if (lane == 0) dec_producer(a, c, tiles, ctl);
    } else if (warp == 1) {
        if (lane == 0) dec_mma(a, c, tiles, tmem, ctl);
    } else {
        dec_epilogue(a, c, tmem, ctl);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_decode_ffn(const DecodeArgs &a, int num_sms, cudaStream_t s) {
    constexpr size_t smem = DSMEM + sizeof(DecCtl) + 1024;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t err = cudaFuncSetAttribute(decode_ffn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(decode_ffn_kernel, dim3(num_sms), dim3(192), smem, s, a);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moe

// ======================================================================
// NVFP4 expert weights (the format of nvfp4.cu): every 128-column x 64-K weight tile is 4 KB of
// E2M1 codes and 512 B of E4M3 block scales, so the forward streams 4.5 bits per weight instead
// of 16. A stage covers 128 K: the expert's token rows (two 64-K halves of 32-row boxes, by TMA)
// and the stage's weight tiles, one contiguous bulk copy (18 KB of W1 and W3, 9 KB of W2).
// Roles (448 threads):
//   warp 0 claims items and streams their stages through a ring of up to 8;
//   warps 6-13 expand the codes to bf16 (code -> f16 by cvt, times its block scale: exact in
//     bf16, at most 7 significant bits) straight into tensor memory, the MMA's A operand, one
//     weight row per lane: two warps per lane quarter, one per 64-K half of the stage;
//   warp 1 issues the MMAs (A = the expanded weights in tensor memory, B = the token rows in
//     shared memory, K-major) into the accumulator;
//   warps 2-5 run the epilogues, multiplying the fp32 accumulator by the power-of-two matrix
//     scale (exact) before the bf16 rounding.
// Tensor memory (512 columns): the accumulators first (two buffers of 2 x 64 columns for a batch
// of at most 64 tokens, which no expert can exceed; else one of 2 x 128), then two expanded
// stages of 128 columns (64 per matrix) from column 256. Each weight element crosses into the
// tensor cores once, from tensor memory, and shared memory carries only the compressed bytes and
// the few token rows.
// Hand-offs between items are the bf16 kernel's.
namespace moe {

namespace {

constexpr int NV_CMAX = 8;                               // compressed stages (at most)
constexpr int NV_AST = 2;                                // expanded stages in tensor memory
constexpr uint32_t NV_ACOL0 = 256;                       // first tensor-memory column of the expanded stages
constexpr uint32_t NV_ACOLS = 128;                       // columns of one expanded stage (64 per matrix)
constexpr int NV_CONV_WARPS = 8;
// compressed stage: the token boxes of K half 0, those of K half 1, then the weight tiles; every
// part 1 KB aligned (32-row boxes of 4 KB; two or four tiles of 4.5 KB)
__host__ __device__ constexpr uint32_t nv_tok_half(int nb) { return nb * DT_BOX; }
__host__ __device__ constexpr uint32_t nv_cstage(int nb) { return 2 * nv_tok_half(nb) + 4 * kNvTile; }
__host__ __device__ constexpr int nv_cstages(int nb) {
    return (int)(DSMEM / nv_cstage(nb)) < NV_CMAX ? (int)(DSMEM / nv_cstage(nb)) : NV_CMAX;
}
static_assert(nv_cstage(1) % 1024 == 0 && (2 * kNvTile) % 1024 == 0, "1 KB aligned stages");
static_assert(nv_cstages(4) >= 2, "at least two compressed stages for 128 tokens");
// accumulator buffers, and the columns of one (the b accumulator of a GEMM1 item sits half
// of them after its a): N = 32 * boxes <= 64 columns while nb <= 2, <= 128 above
__host__ __device__ constexpr int nv_nacc(int nb) { return nb <= 2 ? 2 : 1; }
__host__ __device__ constexpr uint32_t nv_acc_cols(int nb) { return nb <= 2 ? 128 : 256; }
static_assert(2 * 128 <= NV_ACOL0 && 1 * 256 <= NV_ACOL0 && NV_ACOL0 + NV_AST * NV_ACOLS <= 512, "tensor memory plan");

// 32 lanes x 32 consecutive 32-bit columns of tensor memory: thread i of the warp writes lane i
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], bf16 inputs, fp32 accumulator, cta_group::1. A is K-major in
// tensor memory: row m in lane m, K elements 2c and 2c + 1 in column c (low, high half).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

struct NvDecCtl {
    uint64_t cfull[NV_CMAX], cempty[NV_CMAX], afull[NV_AST], aempty[NV_AST], tfull[2], tempty[2], qfull[QD],
        qempty[QD], drain;
    uint32_t tmem_base;
    int item[QD];
};

// Streams every stage's token rows and weight tiles; a compressed stage is freed by the MMA
// thread once the tensor cores have read its token rows (its weights were expanded before).
__device__ void nv_producer(const DecodeArgs &a, NvDecCtl &c, uint8_t *cring, const WaitCtl &ctl) {
    const int total = a.E * (a.F / 128 + a.H / 128);
    const int NC = nv_cstages(a.nb);
    const uint32_t CS = nv_cstage(a.nb), TH = nv_tok_half(a.nb);
    const int H = a.H, F = a.F;
    const uint8_t *w13 = a.nvq + a.nv_w13, *w2 = a.nvq + a.nv_w2;
    int stage = 0, slot = 0;
    uint32_t phase = 0, qphase = 0, issued = 0, last_phase = 0;
    bool ok = true;
    for (;;) {
        int id = -1;
        if (ok) {
            for (;;) {
                id = atomicAdd(a.claim, 1);
                if (id >= total) { id = -1; break; }
                if (a.counts[decode_item(a, id).e] > 0) break;   // experts without rows have no work
            }
        }
        if (!mbar_wait(smem_u32(&c.qempty[slot]), qphase ^ 1, ctl)) { ok = false; id = -1; }
        c.item[slot] = id;
        mbar_arrive(smem_u32(&c.qfull[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        const int s0 = a.offp[it.e];
        const int nb = (a.counts[it.e] + 31) / 32;
        // the item's operands in registers: the stage loop reads no kernel parameter
        const CUtensorMap *tmap = it.gemm1 ? &a.x : &a.h;
        const uint32_t wbytes = (it.gemm1 ? 4 : 2) * kNvTile;
        const uint8_t *wsrc = it.gemm1 ? w13 + ((size_t)it.e * (F / 128) + it.col0 / 128) * (H / 128) * wbytes
                                       : w2 + ((size_t)it.e * (H / 128) + it.col0 / 128) * (F / 128) * wbytes;
        const uint32_t tx = 2 * nb * DT_BOX + wbytes;
        const int ns = it.nk / 2;
        if (!it.gemm1) {
            // h of this expert: the four epilogue warps of every GEMM1 item of it have published
            if (!flag_wait_geq(a.hdone + it.e, 4 * (a.F / 128), ctl)) { ok = false; continue; }
            fence_proxy_async_global();
        }
        for (int ks = 0; ks < ns && ok; ++ks) {
            if (!mbar_wait(smem_u32(&c.cempty[stage]), phase ^ 1, ctl)) { ok = false; break; }
            const uint32_t bar = smem_u32(&c.cfull[stage]);
            const uint32_t sC = smem_u32(cring + stage * CS);
            mbar_arrive_expect_tx(bar, tx);
            for (int hh = 0; hh < 2; ++hh)
                for (int j = 0; j < nb; ++j) tma_load_2d(sC + hh * TH + j * DT_BOX, tmap, bar, (2 * ks + hh) * 64, s0 + 32 * j);
            bulk_load_1d(sC + 2 * TH, wsrc + (size_t)ks * wbytes, wbytes, bar);
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == NC) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok) {
        for (int s = 0; s < NC; ++s) {
            if (!((issued >> s) & 1u)) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(&c.cfull[s]), (last_phase >> s) & 1u) && globaltimer_ns() - t0 < ctl.budget_ns) {}
        }
    }
}

// 8 E2M1 codes (one 32-bit word; element 2i in the low nibble of byte i) times their block
// scale -> 8 bf16 packed in pairs (element 2i in the low half of word i); the matrix scale is
// applied to the accumulator
__device__ __forceinline__ uint4 nv_expand8(uint32_t codes, float scale) {
    uint32_t h[4];
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(codes));
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 v = *reinterpret_cast<const __half2 *>(&h[i]);
        o[i] = pack_bf16x2(__low2float(v) * scale, __high2float(v) * scale);   // exact products
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float nv_scale_value(uint32_t byte) {
    uint32_t h2;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(byte));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Expands one 64-K half of every stage into tensor memory: lane = weight row (a column of W),
// 32 columns of bf16 pairs per matrix.
__device__ void nv_converter(const DecodeArgs &a, NvDecCtl &c, uint8_t *cring, uint32_t tmem, const WaitCtl &ctl) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;                    // the lane quarter this warp may access
    const int half = (warp - 6) >> 2;                // warps 6-9: K half 0, warps 10-13: K half 1
    const int t = quarter * 32 + lane;               // weight row = tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int NC = nv_cstages(a.nb);
    const uint32_t CS = nv_cstage(a.nb), TH = nv_tok_half(a.nb);
    int slot = 0, cs = 0, as = 0;
    uint32_t qphase = 0, cphase = 0, aphase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&c.qfull[slot]), qphase, ctl)) break;
        const int id = c.item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c.qempty[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        const int nmat = it.gemm1 ? 2 : 1;
        bool ok = true;
        for (int ks = 0; ks < it.nk / 2; ++ks) {
            if (!mbar_wait(smem_u32(&c.cfull[cs]), cphase, ctl)) { ok = false; break; }
            if (!mbar_wait(smem_u32(&c.aempty[as]), aphase ^ 1, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint8_t *sW = cring + cs * CS + 2 * TH;
            for (int i = 0; i < nmat; ++i) {
                const uint8_t *tile = sW + (i * 2 + half) * kNvTile;
                const uint4 q0 = *reinterpret_cast<const uint4 *>(tile + t * 32);
                const uint4 q1 = *reinterpret_cast<const uint4 *>(tile + t * 32 + 16);
                const uint32_t sb = *reinterpret_cast<const uint32_t *>(tile + 4096 + t * 4);
                const float sc[4] = {nv_scale_value(sb & 0xFFu), nv_scale_value((sb >> 8) & 0xFFu),
                                     nv_scale_value((sb >> 16) & 0xFFu), nv_scale_value(sb >> 24)};
                const uint32_t w8[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                uint32_t r[32];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 v = nv_expand8(w8[ch], sc[ch / 2]);
                    r[4 * ch] = v.x;
                    r[4 * ch + 1] = v.y;
                    r[4 * ch + 2] = v.z;
                    r[4 * ch + 3] = v.w;
                }
                tmem_st_32x32b_x32(tmem + lane_base + NV_ACOL0 + as * NV_ACOLS + i * 64 + half * 32, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&c.afull[as]));
            if (++cs == NC) { cs = 0; cphase ^= 1; }
            if (++as == NV_AST) { as = 0; aphase ^= 1; }
        }
        if (!ok) break;
    }
}

__device__ void nv_mma(const DecodeArgs &a, NvDecCtl &c, uint8_t *cring, uint32_t tmem, const WaitCtl &ctl) {
    const int NC = nv_cstages(a.nb);
    const uint32_t CS = nv_cstage(a.nb), TH = nv_tok_half(a.nb);
    const int nacc = nv_nacc(a.nb);
    const uint32_t acols = nv_acc_cols(a.nb);
    int as = 0, cs = 0, slot = 0, acc = 0;
    uint32_t aphase = 0, qphase = 0, acc_phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&c.qfull[slot]), qphase, ctl)) break;
        const int id = c.item[slot];
        mbar_arrive(smem_u32(&c.qempty[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        // M = 128 weight columns (A, K-major in tensor memory), N = the expert's rows rounded up
        // to 32 (B, K-major token rows)
        const uint32_t idesc = idesc_bf16_f32(128, 32 * ((a.counts[it.e] + 31) / 32), false, false);
        if (!mbar_wait(smem_u32(&c.tempty[acc]), acc_phase ^ 1, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * acols;
        bool ok = true;
        for (int ks = 0; ks < it.nk / 2; ++ks) {
            // the converters arrive only after they saw the compressed stage (token rows included) land
            if (!mbar_wait(smem_u32(&c.afull[as]), aphase, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sT = smem_u32(cring + cs * CS);
            const uint32_t aw = tmem + NV_ACOL0 + as * NV_ACOLS;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bd = sdesc_sw128(sT + (kk >> 2) * TH + (kk & 3) * 32, 16, 1024);
                mma_bf16_ts(d, aw + kk * 8, bd, idesc, (ks | kk) != 0);
                if (it.gemm1) mma_bf16_ts(d + acols / 2, aw + 64 + kk * 8, bd, idesc, (ks | kk) != 0);
            }
            mma_commit(smem_u32(&c.aempty[as]));
            mma_commit(smem_u32(&c.cempty[cs]));   // its token rows read: the compressed stage is free
            if (++as == NV_AST) { as = 0; aphase ^= 1; }
            if (++cs == NC) cs = 0;
        }
        if (!ok) break;
        mma_commit(smem_u32(&c.tfull[acc]));
        if (++acc == nacc) { acc = 0; acc_phase ^= 1; }
    }
    mma_commit(smem_u32(&c.drain));
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < ctl.budget_ns) {}
}

// The decode epilogue with the matrix scales applied to the accumulator (16 columns at a time).
// GEMM1 writes the h rows of the boxes the MMA computed, which are the rows GEMM2 reads.
__device__ void nv_epilogue(const DecodeArgs &a, NvDecCtl &c, uint32_t tmem, const WaitCtl &ctl) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;
    const int col = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int nacc = nv_nacc(a.nb);
    const uint32_t acols = nv_acc_cols(a.nb);
    int slot = 0, acc = 0;
    uint32_t qphase = 0, acc_phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&c.qfull[slot]), qphase, ctl)) break;
        const int id = c.item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c.qempty[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        if (!mbar_wait(smem_u32(&c.tfull[acc]), acc_phase, ctl)) break;
        tc_fence_after();
        const uint32_t tbase = tmem + lane_base + acc * acols;
        const int s0 = a.offp[it.e];
        const int nb = (a.counts[it.e] + 31) / 32;
        if (it.gemm1) {
            const float g1 = a.nv_g[0 * a.E + it.e], g3 = a.nv_g[1 * a.E + it.e];
            const int f = it.col0 + col;
#pragma unroll 1
            for (int rc = 0; rc < 2 * nb; ++rc) {            // 16 rows at a time
                uint32_t va[16], vb[16];
                tmem_ld_32x32b_x16(tbase + rc * 16, va);
                tmem_ld_32x32b_x16(tbase + acols / 2 + rc * 16, vb);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int row = s0 + rc * 16 + i;
                    const float av = bf2f(f2bf(__uint_as_float(va[i]) * g1)), bv = bf2f(f2bf(__uint_as_float(vb[i]) * g3));
                    a.hrows[(size_t)row * a.F + f] = f2bf(av * sigmoid_d(av) * bv);
                }
            }
        } else {
            const float g2 = a.nv_g[2 * a.E + it.e];
            const int c0 = it.col0 + col, nrows = a.counts[it.e];
#pragma unroll 1
            for (int rc = 0; rc < 8 && rc * 16 < nrows; ++rc) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tbase + rc * 16, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = rc * 16 + i;
                    if (r < nrows) a.y[(size_t)(s0 + r) * a.H + c0] = f2bf(__uint_as_float(v[i]) * g2);
                }
            }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&c.tempty[acc]));
        if (it.gemm1) {
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                fence_proxy_async_global();
                red_release_gpu_add(a.hdone + it.e, 1);
            }
        }
        if (++acc == nacc) { acc = 0; acc_phase ^= 1; }
    }
}

__global__ void __launch_bounds__(448, 1) decode_nv_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *cring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    NvDecCtl &c = *reinterpret_cast<NvDecCtl *>(cring + DSMEM);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    WaitCtl ctl{a.status, a.budget_ns};
    if (threadIdx.x == 0) {
        for (int s = 0; s < nv_cstages(a.nb); ++s) {
            mbar_init(smem_u32(&c.cfull[s]), 1);
            mbar_init(smem_u32(&c.cempty[s]), 1);                  // the MMA thread's commit
        }
        for (int s = 0; s < NV_AST; ++s) {
            mbar_init(smem_u32(&c.afull[s]), NV_CONV_WARPS);        // one lane of every converter warp
            mbar_init(smem_u32(&c.aempty[s]), 1);
        }
        for (int q = 0; q < QD; ++q) {
            mbar_init(smem_u32(&c.qfull[q]), 1);
            mbar_init(smem_u32(&c.qempty[q]), 1 + 4 + NV_CONV_WARPS);   // MMA thread, epilogue and converter warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&c.tfull[i]), 1);
            mbar_init(smem_u32(&c.tempty[i]), 128);
        }
        mbar_init(smem_u32(&c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&a.x);
        tma_prefetch_map(&a.h);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem_base), 512);
        tmem_relinquish();
    }
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = c.tmem_base;
    if (warp == 0) {
        if (lane == 0) nv_producer(a, c, cring, ctl);
    } else if (warp == 1) {
        if (lane == 0) nv_mma(a, c, cring, tmem, ctl);
    } else if (warp < 6) {
        nv_epilogue(a, c, tmem, ctl);
    } else {
        nv_converter(a, c, cring, tmem, ctl);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_decode_nv(const DecodeArgs &a, int num_sms, cudaStream_t s) {
    constexpr size_t smem = DSMEM + sizeof(NvDecCtl) + 1024;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t err = cudaFuncSetAttribute(decode_nv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(decode_nv_kernel, dim3(num_sms), dim3(32 * (6 + NV_CONV_WARPS)), smem, s, a);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moe
