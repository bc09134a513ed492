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
// NVFP4 expert weights (the format of nvfp4.cu): each weight tile (128 columns x 64 of K) is
// 4 KB of E2M1 codes and 512 B of E4M3 block scales, so the forward streams about 4.5 bits per
// weight instead of 16. Roles (320 threads): warp 0 claims items and streams the compressed
// tiles by 1-D bulk copies through an 8-stage ring; warps 6-9 expand them to bf16 tiles in
// shared memory (code -> f16 by cvt, times its block scale: exact in bf16, at most 7
// significant bits), load the expert's token rows into the same stage and hand it to warp 1,
// which issues the MMAs (now with K-major weights) into the double-buffered accumulator; warps
// 2-5 run the epilogues, multiplying the fp32 accumulator by the power-of-two matrix scale
// (exact) before the bf16 rounding. Hand-offs between items are the bf16 kernel's.
namespace moe {

namespace {

constexpr int NV_CMAX = 8;                               // compressed stages (at most)
constexpr uint32_t NV_QTILE = 4096 + 512;                // codes + scales of one weight tile
constexpr int NV_B = 3;                                  // expanded stages
constexpr uint32_t NV_BSTAGE = 2 * DW_TILE;              // bf16 weight tiles (K-major)
constexpr int NV_CONV_THREADS = 128;
// compressed stage: the expert's token rows (nb boxes of 32 rows, 1 KB aligned for the
// 128-byte swizzle) then the compressed W1 and W3 (or W2) tiles
__host__ __device__ constexpr uint32_t nv_cstage(int nb) { return nb * DT_BOX + 2 * NV_QTILE; }
__host__ __device__ constexpr int nv_cstages(int nb) {
    return (int)((DSMEM - NV_B * NV_BSTAGE) / nv_cstage(nb)) < NV_CMAX ? (int)((DSMEM - NV_B * NV_BSTAGE) / nv_cstage(nb))
                                                                       : NV_CMAX;
}
static_assert(nv_cstage(4) % 1024 == 0 && nv_cstage(1) % 1024 == 0, "1 KB aligned stages");

struct NvDecCtl {
    uint64_t cfull[NV_CMAX], cempty[NV_CMAX], bfull[NV_B], bempty[NV_B], tfull[2], tempty[2], qfull[QD], qempty[QD],
        drain;
    uint32_t tmem_base;
    int item[QD];
};

// byte offset of the tile holding (column block, K block) of matrix mat of expert e
__device__ __forceinline__ size_t nv_tile(const DecodeArgs &a, int mat, int e, int col0, int kb) {
    const int K = mat == 2 ? a.F : a.H, N = mat == 2 ? a.H : a.F;
    return ((size_t)e * (N / 128) + col0 / 128) * (K / 64) + kb;
}

// Streams every stage's token rows and compressed weight tiles; a compressed stage is freed by
// the MMA thread once the tensor cores have read its token rows (its weights were expanded
// before that), so the token copies run as far ahead as the compressed ring is deep.
__device__ void nv_producer(const DecodeArgs &a, NvDecCtl &c, uint8_t *cring, const WaitCtl &ctl) {
    const int total = a.E * (a.F / 128 + a.H / 128);
    const int NC = nv_cstages(a.nb);
    const uint32_t CS = nv_cstage(a.nb);
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
        if (!it.gemm1) {
            // h of this expert: the four epilogue warps of every GEMM1 item of it have published
            if (!flag_wait_geq(a.hdone + it.e, 4 * (a.F / 128), ctl)) { ok = false; continue; }
            fence_proxy_async_global();
        }
        for (int kb = 0; kb < it.nk && ok; ++kb) {
            if (!mbar_wait(smem_u32(&c.cempty[stage]), phase ^ 1, ctl)) { ok = false; break; }
            const uint32_t bar = smem_u32(&c.cfull[stage]);
            const uint32_t sC = smem_u32(cring + stage * CS);
            const int nmat = it.gemm1 ? 2 : 1;
            mbar_arrive_expect_tx(bar, nb * DT_BOX + nmat * NV_QTILE);
            for (int j = 0; j < nb; ++j) tma_load_2d(sC + j * DT_BOX, it.gemm1 ? &a.x : &a.h, bar, kb * 64, s0 + 32 * j);
            const uint32_t sQ = sC + a.nb * DT_BOX;
            for (int i = 0; i < nmat; ++i) {
                const int mat = it.gemm1 ? i : 2;
                const size_t t = nv_tile(a, mat, it.e, it.col0, kb);
                bulk_load_1d(sQ + i * NV_QTILE, a.nvq + a.nv_codes[mat] + t * 4096, 4096, bar);
                bulk_load_1d(sQ + i * NV_QTILE + 4096, a.nvq + a.nv_scales[mat] + t * 512, 512, bar);
            }
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
// scale -> 8 bf16 (one 16-byte chunk); the matrix scale is applied to the accumulator
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

__device__ void nv_converter(const DecodeArgs &a, NvDecCtl &c, uint8_t *bring, uint8_t *cring, const WaitCtl &ctl) {
    const int t = threadIdx.x - 192;             // 0..127: the weight row (column of W) this thread expands
    const int lane = threadIdx.x % 32;
    const int NC = nv_cstages(a.nb);
    const uint32_t CS = nv_cstage(a.nb);
    int slot = 0, cs = 0, bs = 0;
    uint32_t qphase = 0, cphase = 0, bphase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&c.qfull[slot]), qphase, ctl)) break;
        const int id = c.item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&c.qempty[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        bool ok = true;
        for (int kb = 0; kb < it.nk; ++kb) {
            if (!mbar_wait(smem_u32(&c.cfull[cs]), cphase, ctl)) { ok = false; break; }
            if (!mbar_wait(smem_u32(&c.bempty[bs]), bphase ^ 1, ctl)) { ok = false; break; }
            uint8_t *sB = bring + bs * NV_BSTAGE;
            const uint8_t *sQ = cring + cs * CS + a.nb * DT_BOX;
            const int nmat = it.gemm1 ? 2 : 1;
            for (int i = 0; i < nmat; ++i) {
                const uint4 q0 = *reinterpret_cast<const uint4 *>(sQ + i * NV_QTILE + t * 32);
                const uint4 q1 = *reinterpret_cast<const uint4 *>(sQ + i * NV_QTILE + t * 32 + 16);
                const uint32_t sb = *reinterpret_cast<const uint32_t *>(sQ + i * NV_QTILE + 4096 + t * 4);
                const float sc[4] = {nv_scale_value(sb & 0xFFu), nv_scale_value((sb >> 8) & 0xFFu),
                                     nv_scale_value((sb >> 16) & 0xFFu), nv_scale_value(sb >> 24)};
                const uint32_t w8[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                uint8_t *row = sB + i * DW_TILE + t * 128;   // K-major, 128-byte swizzle
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(row + ((ch ^ (t & 7)) * 16)) = nv_expand8(w8[ch], sc[ch / 2]);
            }
            fence_proxy_async_shared();   // generic shared-memory writes, read by the tensor cores
            mbar_arrive(smem_u32(&c.bfull[bs]));
            if (++cs == NC) { cs = 0; cphase ^= 1; }
            if (++bs == NV_B) { bs = 0; bphase ^= 1; }
        }
        if (!ok) break;
    }
}

__device__ void nv_mma(const DecodeArgs &a, NvDecCtl &c, uint8_t *bring, uint8_t *cring, uint32_t tmem,
                       const WaitCtl &ctl) {
    const int NC = nv_cstages(a.nb);
    const uint32_t CS = nv_cstage(a.nb);
    int bs = 0, cs = 0, slot = 0, acc = 0;
    uint32_t bphase = 0, qphase = 0, acc_phase = 0;
    for (;;) {
        if (!mbar_wait(smem_u32(&c.qfull[slot]), qphase, ctl)) break;
        const int id = c.item[slot];
        mbar_arrive(smem_u32(&c.qempty[slot]));
        if (++slot == QD) { slot = 0; qphase ^= 1; }
        if (id < 0) break;
        const Item it = decode_item(a, id);
        const uint32_t idesc = idesc_bf16_f32(128, 32 * ((a.counts[it.e] + 31) / 32), false, false);   // both K-major
        if (!mbar_wait(smem_u32(&c.tempty[acc]), acc_phase ^ 1, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256;
        bool ok = true;
        for (int kb = 0; kb < it.nk; ++kb) {
            // the converters arrive only after they saw the compressed stage (token rows included) land
            if (!mbar_wait(smem_u32(&c.bfull[bs]), bphase, ctl)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sB = smem_u32(bring + bs * NV_BSTAGE);
            const uint32_t sT = smem_u32(cring + cs * CS);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc_sw128(sT + kk * 32, 16, 1024);
                mma_bf16_ss(d, sdesc_sw128(sB + kk * 32, 16, 1024), bd, idesc, (kb | kk) != 0);
                if (it.gemm1) mma_bf16_ss(d + 128, sdesc_sw128(sB + DW_TILE + kk * 32, 16, 1024), bd, idesc, (kb | kk) != 0);
            }
            mma_commit(smem_u32(&c.bempty[bs]));
            mma_commit(smem_u32(&c.cempty[cs]));   // its token rows read: the compressed stage is free
            if (++bs == NV_B) { bs = 0; bphase ^= 1; }
            if (++cs == NC) { cs = 0; } 
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

// The bf16 decode epilogue with the matrix scales applied to the accumulator (16 columns at
// a time: this kernel has 320 threads, so at most 168 registers each).
__device__ void nv_epilogue(const DecodeArgs &a, NvDecCtl &c, uint32_t tmem, const WaitCtl &ctl) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;
    const int col = quarter * 32 + lane;
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
        const int nb = (a.counts[it.e] + 31) / 32;
        if (it.gemm1) {
            const float g1 = a.nv_g[0 * a.E + it.e], g3 = a.nv_g[1 * a.E + it.e];
            const int f = it.col0 + col;
#pragma unroll 1
            for (int rc = 0; rc < 8; ++rc) {            // 16 rows at a time; rows past the blocks: zeros
                uint32_t va[16], vb[16];
                if (rc < 2 * nb) {
                    tmem_ld_32x32b_x16(tbase + rc * 16, va);
                    tmem_ld_32x32b_x16(tbase + 128 + rc * 16, vb);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) va[i] = vb[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int row = s0 + rc * 16 + i;
                    const bf16 ab = f2bf(__uint_as_float(va[i]) * g1), bb = f2bf(__uint_as_float(vb[i]) * g3);
                    const float av = bf2f(ab), bv = bf2f(bb);
                    a.a[blk32_elem(row, f, a.F)] = ab;
                    a.b[blk32_elem(row, f, a.F)] = bb;
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
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
    }
}

__global__ void __launch_bounds__(320, 1) decode_nv_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *bring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *cring = bring + NV_B * NV_BSTAGE;   // 1 KB aligned: the token boxes come first in a stage
    NvDecCtl &c = *reinterpret_cast<NvDecCtl *>(bring + DSMEM);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    WaitCtl ctl{a.status, a.budget_ns};
    if (threadIdx.x == 0) {
        for (int s = 0; s < nv_cstages(a.nb); ++s) {
            mbar_init(smem_u32(&c.cfull[s]), 1);
            mbar_init(smem_u32(&c.cempty[s]), 1);                  // the MMA thread's commit
        }
        for (int s = 0; s < NV_B; ++s) {
            mbar_init(smem_u32(&c.bfull[s]), NV_CONV_THREADS);       // every converter thread
            mbar_init(smem_u32(&c.bempty[s]), 1);
        }
        for (int q = 0; q < QD; ++q) {
            mbar_init(smem_u32(&c.qfull[q]), 1);
            mbar_init(smem_u32(&c.qempty[q]), 1 + 4 + 4);   // MMA thread, epilogue and converter warps
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
        if (lane == 0) nv_mma(a, c, bring, cring, tmem, ctl);
    } else if (warp < 6) {
        nv_epilogue(a, c, tmem, ctl);
    } else {
        nv_converter(a, c, bring, cring, ctl);
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
    err = launch_pdl(decode_nv_kernel, dim3(num_sms), dim3(320), smem, s, a);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moe
