// Router, schedule, dispatch, combine and the token-side backward kernels.
//
//   router_topk      logits = x W_r (+bias) in fp32 on tensor cores (mma.sync,
//                    fixed-order reduction), softmax, top-k (descending, ties to
//                    the lower expert index), renormalised weights
//   schedule_*       per-(macrobatch, expert) counts with warp match/ballot
//                    histograms, exclusive scans, stable scatter (article
//                    "O MoK do Cursor ...", section 01: count, place, group)
//   dispatch_rows    pull-style gather of token rows into expert-sorted rows
//                    (section 02: the destination reads the rows it needs)
//   combine          top-k weighted sum in fixed slot order (section 03:
//                    combine and final weighted fusion; deterministic)
//   router_bwd       dw -> dp -> dlogits through renormalisation and softmax
//   reverse_dispatch dx = sum_j dX rows (fixed order) + dlogits W_r^T
//   router_wgrad     dW_r = x^T dlogits with fixed-order split reduction
#include "route_kernels.cuh"
#include "combine_item.cuh"

namespace moe {

// ------------------------------------------------------------------ router

// W_r [H,E] -> WrT [EP,H] (EP = E rounded up to 8, extra rows zero), so the
// tensor-core B fragments are contiguous along H.
// One thread per output element (coalesced stores; the reads of W_r stride by E).
__global__ void transpose_wr_kernel(const bf16 *__restrict__ Wr, bf16 *__restrict__ WrT, int H, int E, int EP) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= H * EP) return;
    const int e = i / H, h = i % H;
    WrT[i] = e < E ? Wr[(size_t)h * E + e] : f2bf(0.0f);
}

__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

constexpr int kRouterTokens = 16;   // tokens per block (one m16 tile)
constexpr int kRouterMT = kRouterTokens / 16;
constexpr int kRouterWarps = 8;     // warps split H

// Block: 16 tokens x all experts. Warp w covers H range [w*H/8, (w+1)*H/8).
// The contraction order inside a warp is permuted (thread c of a quad loads 8
// consecutive h with one 16-byte load and feeds them as its k-slots of two
// m16n8k16 steps); A and B use the same permutation, so the sum is exact in
// structure and fixed in order. PF = 32-h steps loaded ahead of the MMAs: 1 when
// the grid fills the GPU, deeper for the few blocks of a small batch, whose warps
// would otherwise wait out one memory round trip per step. The MMAs run in the
// same order either way, so the logits do not depend on PF.
template <int NT, int PF>
__global__ void __launch_bounds__(256) router_topk_kernel(RouterArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    extern __shared__ float part[];   // [warps][kRouterTokens][EP]
    const int EP = NT * 8;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int g = lane >> 2, c = lane & 3;
    const int t0 = blockIdx.x * kRouterTokens;
    const int hspan = a.H / kRouterWarps;
    const int hbeg = warp * hspan;
    float acc[kRouterMT][NT][4];
#pragma unroll
    for (int mt = 0; mt < kRouterMT; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][n][i] = 0.0f;
    // the token rows this thread feeds: mt*16 + g and mt*16 + g + 8
    const bf16 *xrow[kRouterMT][2];
    bool valid[kRouterMT][2];
#pragma unroll
    for (int mt = 0; mt < kRouterMT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            int t = t0 + mt * 16 + g + hh * 8;
            valid[mt][hh] = t < a.T;
            xrow[mt][hh] = a.x + (size_t)(valid[mt][hh] ? t : 0) * a.H;
        }
    // 32 h per step; the loads of step i+PF are issued right after the MMAs of step i
    auto load = [&](int h0, uint4 (&xv)[kRouterMT][2], uint4 (&wv)[NT]) {
        const int hc = h0 + 8 * c;
#pragma unroll
        for (int mt = 0; mt < kRouterMT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                xv[mt][hh] = valid[mt][hh] ? ld_nc_v4(xrow[mt][hh] + hc) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int n = 0; n < NT; ++n) wv[n] = ld_nc_v4(a.WrT + (size_t)(n * 8 + g) * a.H + hc);
    };
    auto step = [&](const uint4 (&xv)[kRouterMT][2], const uint4 (&wv)[NT]) {
#pragma unroll
        for (int mt = 0; mt < kRouterMT; ++mt) {
            // step 0 uses h = hc+0..3, step 1 uses hc+4..7
            uint32_t A0[4] = {xv[mt][0].x, xv[mt][1].x, xv[mt][0].y, xv[mt][1].y};
            uint32_t A1[4] = {xv[mt][0].z, xv[mt][1].z, xv[mt][0].w, xv[mt][1].w};
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                mma_16816_bf16(acc[mt][n], A0, wv[n].x, wv[n].y);
                mma_16816_bf16(acc[mt][n], A1, wv[n].z, wv[n].w);
            }
        }
    };
    const int nsteps = hspan / 32;   // hspan is a multiple of 32
    uint4 xv[PF + 1][kRouterMT][2], wv[PF + 1][NT];
#pragma unroll
    for (int j = 0; j < PF; ++j)
        if (j < nsteps) load(hbeg + 32 * j, xv[j], wv[j]);
    // PF + 1 slots, so the load for step i + PF never overwrites the operands of step i
    for (int i0 = 0; i0 < nsteps; i0 += PF + 1) {
#pragma unroll
        for (int j = 0; j <= PF; ++j) {
            const int i = i0 + j;
            if (i < nsteps) {
                if (i + PF < nsteps) load(hbeg + 32 * (i + PF), xv[(j + PF) % (PF + 1)], wv[(j + PF) % (PF + 1)]);
                step(xv[j], wv[j]);
            }
        }
    }
    // partial logits of this warp -> shared memory
    float *my = part + (size_t)warp * kRouterTokens * EP;
#pragma unroll
    for (int mt = 0; mt < kRouterMT; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            int row = mt * 16 + g, col = n * 8 + 2 * c;
            my[row * EP + col] = acc[mt][n][0];
            my[row * EP + col + 1] = acc[mt][n][1];
            my[(row + 8) * EP + col] = acc[mt][n][2];
            my[(row + 8) * EP + col + 1] = acc[mt][n][3];
        }
    __syncthreads();
    // each warp finishes kRouterTokens / kRouterWarps tokens; lane owns experts lane and lane+32
    constexpr int kPerWarp = kRouterTokens / kRouterWarps;
    for (int tt = warp * kPerWarp; tt < warp * kPerWarp + kPerWarp; ++tt) {
        const int t = t0 + tt;
        if (t >= a.T) break;
        float l[2];
        bool ok[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            int e = lane + 32 * s;
            ok[s] = e < a.E;
            float v = 0.0f;
            if (ok[s]) {
                for (int w = 0; w < kRouterWarps; ++w) v += part[((size_t)w * kRouterTokens + tt) * EP + e];
                if (a.bias) v += a.bias[e];
            }
            l[s] = ok[s] ? v : -INFINITY;
        }
        float mx = fmaxf(l[0], l[1]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float ex[2], sum = 0.0f;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            ex[s] = ok[s] ? __expf(l[s] - mx) : 0.0f;
            sum += ex[s];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.0f / sum;
#pragma unroll
        for (int s = 0; s < 2; ++s)
            if (ok[s]) a.probs[(size_t)t * a.E + lane + 32 * s] = ex[s] * inv;
        // top-k: k rounds of a warp argmax over logits (ties -> lower index)
        bool taken[2] = {!ok[0], !ok[1]};
        float psel_sum = 0.0f;
        float my_p = 0.0f;
        int my_e = -1;
        for (int j = 0; j < a.k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                int e = lane + 32 * s;
                if (!taken[s] && (l[s] > bv || (l[s] == bv && e < bi))) { bv = l[s]; bi = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
#pragma unroll
            for (int s = 0; s < 2; ++s)
                if (lane + 32 * s == bi) taken[s] = true;
            float p = __expf(bv - mx) * inv;
            psel_sum += p;
            if (lane == j) { my_p = p; my_e = bi; }
        }
        if (lane < a.k) {
            const size_t o = (size_t)t * a.k + lane;
            const float w = my_p / psel_sum;
            a.ids[o] = my_e;
            a.w[o] = w;
            if (a.ids2) { a.ids2[o] = my_e; a.w2[o] = w; }
        }
    }
}

cudaError_t launch_router(const RouterArgs &a, cudaStream_t s) {
    const int EP = (a.E + 7) / 8 * 8;
    const int blocks = ceil_div(a.T, kRouterTokens);
    const size_t smem = (size_t)kRouterWarps * kRouterTokens * EP * sizeof(float);
    cudaError_t le = launch_pdl(transpose_wr_kernel, dim3(ceil_div(a.H * EP, 256)), dim3(256), 0, s, a.Wr, a.WrT, a.H, a.E, EP);
    if (le != cudaSuccess) return le;
    if (blocks == 0) return cudaGetLastError();
    // a batch of up to 64 blocks (1024 tokens) leaves most SMs idle: load four steps ahead
    const bool deep = blocks <= 64;
#define MOE_ROUTER_CASE(NT)                                                                           \
    case NT: {                                                                                       \
        auto *kern = deep ? router_topk_kernel<NT, 4> : router_topk_kernel<NT, 1>;                   \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        if (e != cudaSuccess) return e;                                                              \
        e = launch_pdl(kern, dim3(blocks), dim3(256), smem, s, a);                                   \
        if (e != cudaSuccess) return e;                                                              \
        break;                                                                                       \
    }
    switch (EP / 8) {
        MOE_ROUTER_CASE(1)
        MOE_ROUTER_CASE(2)
        MOE_ROUTER_CASE(3)
        MOE_ROUTER_CASE(4)
        MOE_ROUTER_CASE(5)
        MOE_ROUTER_CASE(6)
        MOE_ROUTER_CASE(7)
        MOE_ROUTER_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef MOE_ROUTER_CASE
    return cudaGetLastError();
}

// ------------------------------------------------------------------ schedule
//
// Slots s = t*k + j of macrobatch m occupy [m*Mb*k, min(T,(m+1)*Mb)*k). Chunk
// c = m*chunks_per_mb + i covers slots [m*Mb*k + i*kSchedChunk, ...) of that
// macrobatch only. Inside a chunk, warp w walks its own contiguous sub-range of
// 256 slots in order; the rank of a slot among equal experts is its warp's
// running count plus its rank inside the 32-slot group (match_any + popc).

__device__ __forceinline__ void chunk_range(const SchedArgs &a, int c, int &m, int &s0, int &s1) {
    m = c / a.chunks_per_mb;
    const int i = c % a.chunks_per_mb;
    const int mb_s0 = m * a.Mb * a.k;
    const int mb_s1 = min(a.T, (m + 1) * a.Mb) * a.k;
    s0 = mb_s0 + i * kSchedChunk;
    s1 = min(mb_s1, s0 + kSchedChunk);
}

// Pass over one chunk; calls f(slot, expert, rank_within_chunk) per valid slot
// after the per-warp bases are known. With FINAL=false it only counts.
template <bool FINAL>
__device__ void chunk_pass(const SchedArgs &a, int c, int *s_warp_cnt /* [warps][E] */, int *s_base /* [E] */) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int m, s0, s1;
    chunk_range(a, c, m, s0, s1);
    const int per_warp = kSchedChunk / kSchedWarps;
    const int w0 = s0 + warp * per_warp, w1 = min(s1, w0 + per_warp);
    int *cnt = s_warp_cnt + warp * a.E;
    for (int e = lane; e < a.E; e += 32) cnt[e] = 0;
    __syncwarp();
    // counting walk
    for (int base = w0; base < w1; base += 32) {
        const int s = base + lane;
        int e = s < w1 ? a.ids[s] : -1;
        if (e >= a.E || (e < 0 && s < w1)) { raise_status(a.status, kStatusInternal); e = -1; }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int leader = __ffs(peers) - 1;
        if (e >= 0 && lane == leader) cnt[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    if (!FINAL) return;
    // exclusive scan over warps per expert (in place: cnt becomes the warp base)
    if (threadIdx.x < a.E) {
        const int e = threadIdx.x;
        int run = s_base[e];
        for (int w = 0; w < kSchedWarps; ++w) {
            int v = s_warp_cnt[w * a.E + e];
            s_warp_cnt[w * a.E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    // scatter walk
    for (int base = w0; base < w1; base += 32) {
        const int s = base + lane;
        int e = s < w1 ? a.ids[s] : -1;
        if (e >= a.E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int leader = __ffs(peers) - 1;
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0) {
            const int pos = cnt[e] + rank;                 // unpadded sorted position
            const int me = m * a.E + e;
            const int prow = pos - a.offsets[m * (a.E + 1) + e] + a.offp[me];
            a.sorted_to_slot[pos] = s;
            a.slot_to_sorted[s] = pos;
            if (a.slot_row) {
                a.slot_row[s] = prow;
                a.row_slot[prow] = s;
            }
        }
        __syncwarp();
        if (e >= 0 && lane == leader) cnt[e] += __popc(peers);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kSchedWarps * 32) schedule_count_kernel(SchedArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ int s_cnt[kSchedWarps * kMaxExperts];
    chunk_pass<false>(a, blockIdx.x, s_cnt, nullptr);
    if (threadIdx.x < a.E) {
        int v = 0;
        for (int w = 0; w < kSchedWarps; ++w) v += s_cnt[w * a.E + threadIdx.x];
        a.chunk_counts[blockIdx.x * a.E + threadIdx.x] = v;
    }
}

// One block: per-(m,e) counts, unpadded and padded exclusive scans, chunk bases,
// and -1 marks on padding rows.
// Exclusive scan of two values per thread across a 1024-thread block.
__device__ void block_exclusive_scan2(int &a, int &b, int *s_w /* [64] */) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32, nw = blockDim.x / 32;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ta = __shfl_up_sync(0xffffffffu, ia, o), tb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) { ia += ta; ib += tb; }
    }
    if (lane == 31) { s_w[warp] = ia; s_w[32 + warp] = ib; }
    __syncthreads();
    if (warp == 0) {
        const int va = lane < nw ? s_w[lane] : 0, vb = lane < nw ? s_w[32 + lane] : 0;
        int xa = va, xb = vb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, xa, o), tb = __shfl_up_sync(0xffffffffu, xb, o);
            if (lane >= o) { xa += ta; xb += tb; }
        }
        __syncwarp();
        s_w[lane] = xa - va;
        s_w[32 + lane] = xb - vb;
    }
    __syncthreads();
    a = ia - a + s_w[warp];
    b = ib - b + s_w[32 + warp];
}

// Scan with every intermediate in shared memory (used when nchunks*E + 3*nM*E + 2
// ints fit the dynamic allocation): one coalesced read of the chunk counts, no
// global round trips between the phases.
__global__ void __launch_bounds__(1024) schedule_scan_smem_kernel(SchedArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    extern __shared__ int sm[];
    __shared__ int s_tot[64];
    const int n = a.nM * a.E, ncc = a.nchunks * a.E;
    int *s_cc = sm;                  // [nchunks*E]: counts, then bases relative to the (m, e) start
    int *s_cnt = s_cc + ncc;         // [n]
    int *s_off = s_cnt + n;          // [n + 1] exclusive scan of the counts
    int *s_offp = s_off + n + 1;     // [n + 1] exclusive scan of the 128-padded counts
    for (int i = threadIdx.x; i < ncc; i += blockDim.x) s_cc[i] = a.chunk_counts[i];
    if (a.ready)
        for (int i = threadIdx.x; i < a.ready_n; i += blockDim.x) a.ready[i] = 0;
    for (int z = 0; z < 2; ++z)
        if (a.zero[z])
            for (int i = threadIdx.x; i < a.zero_n[z]; i += blockDim.x) a.zero[z][i] = 0;
    __syncthreads();
    for (int me = threadIdx.x; me < n; me += blockDim.x) {
        const int m = me / a.E, e = me % a.E;
        int run = 0;
        for (int i = 0; i < a.chunks_per_mb; ++i) {
            const int c = m * a.chunks_per_mb + i;
            if (c >= a.nchunks) break;   // no slots (T = 0)
            const int v = s_cc[c * a.E + e];
            s_cc[c * a.E + e] = run;
            run += v;
        }
        s_cnt[me] = run;
    }
    __syncthreads();
    const int per = ceil_div(max(n, 1), (int)blockDim.x);
    const int b0 = threadIdx.x * per, b1 = min(n, b0 + per);
    int tot = 0, totp = 0;
    for (int i = b0; i < b1; ++i) {
        tot += s_cnt[i];
        totp += (s_cnt[i] + kRowPad - 1) / kRowPad * kRowPad;
    }
    int run = tot, runp = totp;
    block_exclusive_scan2(run, runp, s_tot);
    for (int i = b0; i < b1; ++i) {
        s_off[i] = run;
        s_offp[i] = runp;
        run += s_cnt[i];
        runp += (s_cnt[i] + kRowPad - 1) / kRowPad * kRowPad;
    }
    if (threadIdx.x == blockDim.x - 1) { s_off[n] = run; s_offp[n] = runp; }
    if (n == 0 && threadIdx.x == 0) { s_off[0] = 0; s_offp[0] = 0; }
    __syncthreads();
    for (int me = threadIdx.x; me < n; me += blockDim.x) {
        const int m = me / a.E, e = me % a.E;
        a.counts[me] = s_cnt[me];
        a.offsets[m * (a.E + 1) + e] = s_off[me];
        if (e == a.E - 1) a.offsets[m * (a.E + 1) + a.E] = s_off[me] + s_cnt[me];
        a.offp[me] = s_offp[me];
    }
    if (threadIdx.x == 0) a.offp[n] = s_offp[n];
    for (int i = threadIdx.x; i < ncc; i += blockDim.x) {   // chunk bases -> absolute sorted positions
        const int c = i / a.E, e = i % a.E;
        a.chunk_base[i] = s_cc[i] + s_off[(c / a.chunks_per_mb) * a.E + e];
    }
    if (a.row_slot) {   // padding rows of every (m, e) run hold no slot: 128 candidates per run
        for (int i = threadIdx.x; i < n * kRowPad; i += blockDim.x) {
            const int me = i / kRowPad, r = s_offp[me] + s_cnt[me] + i % kRowPad;
            if (r < s_offp[me + 1]) a.row_slot[r] = -1;
        }
    }
}

size_t schedule_scan_smem_bytes(const SchedArgs &a) {
    return 4 * ((size_t)a.nchunks * a.E + 3 * (size_t)a.nM * a.E + 2);
}

__global__ void __launch_bounds__(1024) schedule_scan_kernel(SchedArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ int s_tot[64];
    if (a.ready)
        for (int i = threadIdx.x; i < a.ready_n; i += blockDim.x) a.ready[i] = 0;
    for (int z = 0; z < 2; ++z)
        if (a.zero[z])
            for (int i = threadIdx.x; i < a.zero_n[z]; i += blockDim.x) a.zero[z][i] = 0;
    const int n = a.nM * a.E;
    // counts and chunk bases (relative to the (m,e) start); the chunk counts are
    // read eight at a time so their loads overlap
    for (int me = threadIdx.x; me < n; me += blockDim.x) {
        const int m = me / a.E, e = me % a.E;
        int run = 0;
        for (int i0 = 0; i0 < a.chunks_per_mb; i0 += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = m * a.chunks_per_mb + i0 + u;
                // no slots (T = 0): no count block wrote chunks past nchunks
                v[u] = (i0 + u < a.chunks_per_mb && c < a.nchunks) ? __ldg(a.chunk_counts + c * a.E + e) : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = m * a.chunks_per_mb + i0 + u;
                if (i0 + u < a.chunks_per_mb && c < a.nchunks) a.chunk_base[c * a.E + e] = run;
                run += v[u];
            }
        }
        a.counts[me] = run;
    }
    __syncthreads();
    // exclusive scans over (m, e) of the counts and of the 128-padded counts:
    // each thread owns a contiguous range, the range totals go through a
    // warp-shuffle block scan
    const int per = ceil_div(max(n, 1), (int)blockDim.x);
    const int b0 = threadIdx.x * per, b1 = min(n, b0 + per);
    int tot = 0, totp = 0;
    for (int i = b0; i < b1; ++i) {
        tot += a.counts[i];
        totp += (a.counts[i] + kRowPad - 1) / kRowPad * kRowPad;
    }
    int run = tot, runp = totp;
    block_exclusive_scan2(run, runp, s_tot);
    for (int i = b0; i < b1; ++i) {
        const int m = i / a.E, e = i % a.E;
        a.offsets[m * (a.E + 1) + e] = run;
        a.offp[i] = runp;
        run += a.counts[i];
        runp += (a.counts[i] + kRowPad - 1) / kRowPad * kRowPad;
        if (e == a.E - 1) a.offsets[m * (a.E + 1) + a.E] = run;
    }
    if (threadIdx.x == blockDim.x - 1) a.offp[n] = runp;
    if (n == 0 && threadIdx.x == 0) a.offp[0] = 0;
    __syncthreads();
    // chunk bases become absolute sorted positions
    for (int me = threadIdx.x; me < n; me += blockDim.x) {
        const int m = me / a.E, e = me % a.E;
        const int start = a.offsets[m * (a.E + 1) + e];
        for (int i = 0; i < a.chunks_per_mb && m * a.chunks_per_mb + i < a.nchunks; ++i)
            a.chunk_base[(m * a.chunks_per_mb + i) * a.E + e] += start;
    }
    // padding rows of every (m, e) run hold no slot
    if (a.row_slot) {
        for (int me = threadIdx.x; me < n; me += blockDim.x) {
            const int r1 = a.offp[me + 1];
            for (int r = a.offp[me] + a.counts[me]; r < r1; ++r) a.row_slot[r] = -1;
        }
    }
}

__global__ void __launch_bounds__(kSchedWarps * 32) schedule_scatter_kernel(SchedArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ int s_cnt[kSchedWarps * kMaxExperts];
    __shared__ int s_base[kMaxExperts];
    if (threadIdx.x < a.E) s_base[threadIdx.x] = a.chunk_base[blockIdx.x * a.E + threadIdx.x];
    __syncthreads();
    chunk_pass<true>(a, blockIdx.x, s_cnt, s_base);
}

// The whole schedule in one block when every slot sits in one macrobatch of at most
// kSchedSingleChunks chunks (a small batch, where three launches would cost more than the
// work): the count pass of every chunk, the scans over the experts by one warp, then the
// scatter pass of every chunk. The passes and the layout are those of the three kernels.
constexpr int kSchedSingleChunks = 8;
__global__ void __launch_bounds__(kSchedWarps * 32) schedule_single_kernel(SchedArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ int s_cnt[kSchedWarps * kMaxExperts];
    __shared__ int s_cc[kSchedSingleChunks * kMaxExperts];   // chunk counts, then bases inside the expert's run
    __shared__ int s_start[kMaxExperts], s_num[kMaxExperts], s_offp[kMaxExperts + 1], s_base[kMaxExperts];
    const int E = a.E, warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (a.ready)
        for (int i = threadIdx.x; i < a.ready_n; i += blockDim.x) a.ready[i] = 0;
    for (int z = 0; z < 2; ++z)
        if (a.zero[z])
            for (int i = threadIdx.x; i < a.zero_n[z]; i += blockDim.x) a.zero[z][i] = 0;
    for (int c = 0; c < a.nchunks; ++c) {
        chunk_pass<false>(a, c, s_cnt, nullptr);   // ends at a block barrier
        if (threadIdx.x < E) {
            int v = 0;
            for (int w = 0; w < kSchedWarps; ++w) v += s_cnt[w * E + threadIdx.x];
            s_cc[c * E + threadIdx.x] = v;
        }
        __syncthreads();   // the next pass clears s_cnt
    }
    if (warp == 0) {
        // expert e = lane + 32 s: its count, the chunk bases inside its run, and exclusive scans
        // over the experts in index order (lanes for s = 0, then lanes for s = 1)
        int cnt[2], pad[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int e = lane + 32 * q;
            cnt[q] = 0;
            if (e < E)
                for (int c = 0; c < a.nchunks; ++c) {
                    const int v = s_cc[c * E + e];
                    s_cc[c * E + e] = cnt[q];
                    cnt[q] += v;
                }
            pad[q] = (cnt[q] + kRowPad - 1) / kRowPad * kRowPad;
        }
        int off = 0, offp = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            int x = cnt[q], y = pad[q];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tx = __shfl_up_sync(0xffffffffu, x, o), ty = __shfl_up_sync(0xffffffffu, y, o);
                if (lane >= o) { x += tx; y += ty; }
            }
            const int e = lane + 32 * q;
            if (e < E) {
                s_num[e] = cnt[q];
                s_start[e] = off + x - cnt[q];
                s_offp[e] = offp + y - pad[q];
                a.counts[e] = cnt[q];
                a.offsets[e] = s_start[e];
                a.offp[e] = s_offp[e];
            }
            off += __shfl_sync(0xffffffffu, x, 31);
            offp += __shfl_sync(0xffffffffu, y, 31);
        }
        if (lane == 0) {
            a.offsets[E] = off;
            a.offp[E] = offp;
            s_offp[E] = offp;
        }
    }
    __syncthreads();
    if (a.row_slot) {   // padding rows of every expert's run hold no slot: 128 candidates per run
        for (int i = threadIdx.x; i < E * kRowPad; i += blockDim.x) {
            const int e = i / kRowPad, r = s_offp[e] + s_num[e] + i % kRowPad;
            if (r < s_offp[e + 1]) a.row_slot[r] = -1;
        }
    }
    for (int c = 0; c < a.nchunks; ++c) {
        if (threadIdx.x < E) s_base[threadIdx.x] = s_start[threadIdx.x] + s_cc[c * E + threadIdx.x];
        __syncthreads();
        chunk_pass<true>(a, c, s_cnt, s_base);
        __syncthreads();   // the next chunk rewrites s_base and s_cnt
    }
}

cudaError_t launch_schedule(const SchedArgs &a, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (a.nM == 1 && a.nchunks >= 1 && a.nchunks <= kSchedSingleChunks) {
        if ((e = launch_pdl(schedule_single_kernel, dim3(1), dim3(kSchedWarps * 32), 0, s, a)) != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (a.nchunks > 0 && (e = launch_pdl(schedule_count_kernel, dim3(a.nchunks), dim3(kSchedWarps * 32), 0, s, a)) != cudaSuccess)
        return e;
    const size_t scan_smem = schedule_scan_smem_bytes(a);
    if (scan_smem <= 48 * 1024)
        e = launch_pdl(schedule_scan_smem_kernel, dim3(1), dim3(1024), scan_smem, s, a);
    else
        e = launch_pdl(schedule_scan_kernel, dim3(1), dim3(1024), 0, s, a);
    if (e != cudaSuccess) return e;
    if (a.nchunks > 0 && (e = launch_pdl(schedule_scatter_kernel, dim3(a.nchunks), dim3(kSchedWarps * 32), 0, s, a)) != cudaSuccess)
        return e;
    return cudaGetLastError();
}

// ------------------------------------------------------------------ dispatch

// Warp per padded row r in [offp[beg], offp[end]): dst[dst_row0 + r - offp[beg]]
// = src[row_slot[r] / k], zeros for padding rows. 16-byte loads and stores. A slot outside
// [-1, nslots) raises MOE_ERR_INTERNAL and its row is written as zeros.
__global__ void __launch_bounds__(256) dispatch_rows_kernel(DispatchArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    const int lane = threadIdx.x % 32;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int nw = gridDim.x * blockDim.x / 32;
    const int r0 = a.offp[a.beg], r1 = a.offp[a.end];
    const int vecs = a.H / 8;
    for (int r = r0 + gw; r < r1; r += nw) {
        int slot = a.row_slot[r];
        if (slot < -1 || slot >= a.nslots) {
            if (lane == 0) raise_status(a.status, kStatusInternal);
            slot = -1;
        }
        bf16 *dst = a.dst + (size_t)(a.dst_row0 + r - r0) * a.H;
        if (slot < 0) {
            for (int v = lane; v < vecs; v += 32) st_v4(dst + v * 8, make_uint4(0, 0, 0, 0));
        } else {
            const bf16 *src = a.src + (size_t)(slot / a.k) * a.H;
            // 8 vectors per lane in flight (4 KB per warp)
            for (int v0 = 0; v0 < vecs; v0 += 256) {
                uint4 xv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + lane + 32 * u;
                    xv[u] = v < vecs ? ld_nc_v4(src + v * 8) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + lane + 32 * u;
                    if (v < vecs) st_v4(dst + v * 8, xv[u]);
                }
            }
        }
    }
}

cudaError_t launch_dispatch(const DispatchArgs &a, int max_rows, int num_sms, cudaStream_t s) {
    if (max_rows <= 0) return cudaSuccess;
    int blocks = min(ceil_div(max_rows, 8), num_sms * 8);
    cudaError_t e = launch_pdl(dispatch_rows_kernel, dim3(blocks), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ------------------------------------------------------------------ combine

// Warp per token t in [t0, t1): out[t] = bf16( sum_{j=0}^{k-1} w[t,j] * Y[row(t,j)] ),
// fp32 accumulation in fixed j order.
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    const int lane = threadIdx.x % 32;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int nw = gridDim.x * blockDim.x / 32;
    const int lo = a.offp[a.m * a.E], hi = a.offp[(a.m + 1) * a.E];
    const int shift = a.ring_base - lo;
    const int vecs = a.H / 8;   // a multiple of 32
    // work item = (token, 512 columns): a macrobatch with few tokens still spreads
    // over every warp, and each item is one or two rounds of loads
    const int nch = (vecs + 63) / 64;
    const int items = (a.t1 - a.t0) * nch;
    for (int it = gw; it < items; it += nw) {
        combine_item(a, it, nch, shift, lo, hi, lane);
    }
}

cudaError_t launch_combine(const CombineArgs &a, int num_sms, cudaStream_t s) {
    const int n = a.t1 - a.t0;
    if (n <= 0) return cudaSuccess;
    const int items = n * ((a.H / 8 + 63) / 64);
    int blocks = min(ceil_div(items, 8), num_sms * 8);
    cudaError_t e = launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ------------------------------------------------------------------ backward

// Warp per token: dw[t,j] = sum of the per-N-tile partials of row(t,j) (fixed
// order); dp_j = (dw_j - sum_i w_i dw_i) / S on the chosen experts, 0 elsewhere;
// dlogits = p * (dp - sum_l p_l dp_l).
__global__ void __launch_bounds__(256) router_bwd_kernel(RouterBwdArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    const int lane = threadIdx.x % 32;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (t >= a.T) return;
    // lane j < k: dw and w of slot j
    float dwj = 0.0f, wj = 0.0f, pj = 0.0f;
    int ej = -1;
    if (lane < a.k) {
        const int s = t * a.k + lane;
        const int row = a.slot_row[s];
        if (row >= 0 && row < a.rows) {
            for (int n = 0; n < a.nparts; ++n) dwj += a.dw_part[(size_t)row * a.nparts + n];
        } else {
            raise_status(a.status, kStatusInternal);   // the slot's dw is left at 0
        }
        wj = a.w[s];
        ej = a.ids[s];
        pj = a.probs[(size_t)t * a.E + ej];
    }
    float swd = wj * dwj, S = pj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        swd += __shfl_xor_sync(0xffffffffu, swd, o);
        S += __shfl_xor_sync(0xffffffffu, S, o);
    }
    const float dpj = lane < a.k ? (dwj - swd) / S : 0.0f;
    // scatter dp to experts: lane owns experts lane, lane+32
    float dp[2] = {0.0f, 0.0f}, p[2] = {0.0f, 0.0f};
    for (int j = 0; j < a.k; ++j) {
        const int e = __shfl_sync(0xffffffffu, ej, j);
        const float v = __shfl_sync(0xffffffffu, dpj, j);
        if (e == lane) dp[0] = v;
        if (e == lane + 32) dp[1] = v;
    }
    float spdp = 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
        const int e = lane + 32 * s2;
        if (e < a.E) p[s2] = a.probs[(size_t)t * a.E + e];
        spdp += p[s2] * dp[s2];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) spdp += __shfl_xor_sync(0xffffffffu, spdp, o);
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
        const int e = lane + 32 * s2;
        if (e < a.E) a.dlogits[(size_t)t * a.E + e] = p[s2] * (dp[s2] - spdp);
    }
}

// Reverse dispatch (article section 02: push reverse-dispatch, here a local
// gather-sum):
//   dx[t] = bf16( sum_j dXs[row(t,j)]  (fixed j order)  +  sum_e dlogits[t,e] W_r[h,e] ).
// Block: 64 tokens (4 warps x 16) x 256 h (four 64-wide chunks). Per chunk the
// block stages W_r[h0..h0+63][0..E) once in shared memory; each warp computes
// its 16 x 64 router term on mma.sync with dlogits split into bf16 hi + lo
// parts (about 16 significant bits), parks it in a shared tile, and then each
// lane owns 32 contiguous h of one token for the 16-byte gathers of the k rows.
constexpr int kRdTokens = 64;
__global__ void __launch_bounds__(128, 4) reverse_dispatch_kernel(RevDispatchArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ float s_acc[4][16][64 + 4];
    __shared__ __align__(16) bf16 s_wr[64][64 + 8];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int g = lane >> 2, c = lane & 3;
    const int t0 = blockIdx.x * kRdTokens + warp * 16;
    const int hb0 = blockIdx.y * 256;
    const int KS = (a.E + 15) / 16;   // k16 steps over experts (<= 4)
    // A fragments of dlogits (rows g, g+8; k-slots 2c, 2c+1, 2c+8, 2c+9)
    uint32_t Ahi[4][4], Alo[4][4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            Ahi[ks][r] = 0u;
            Alo[ks][r] = 0u;
            if (ks < KS) {
                const int t = t0 + g + ((r & 1) ? 8 : 0);
                const int e = ks * 16 + 2 * c + ((r & 2) ? 8 : 0);
                float v0 = 0.0f, v1 = 0.0f;
                if (t < a.T) {
                    if (e < a.E) v0 = a.dlogits[(size_t)t * a.E + e];
                    if (e + 1 < a.E) v1 = a.dlogits[(size_t)t * a.E + e + 1];
                }
                const uint32_t hi = pack_bf16x2(v0, v1);
                Ahi[ks][r] = hi;
                Alo[ks][r] = pack_bf16x2(v0 - bf16lo(hi), v1 - bf16hi(hi));
            }
        }
    const int my_t = t0 + (lane >> 1);
    const int half = lane & 1;
    int rows[32];
    const int kk = a.k < 32 ? a.k : 32;
    // a row outside [0, rows) raises MOE_ERR_INTERNAL and is skipped (-1)
    auto checked_row = [&](int j) {
        const int r = a.slot_row[(size_t)my_t * a.k + j];
        if (r >= 0 && r < a.rows) return r;
        raise_status(a.status, kStatusInternal);
        return -1;
    };
    for (int j = 0; j < kk; ++j) rows[j] = my_t < a.T ? checked_row(j) : -1;
    for (int h0 = hb0; h0 < hb0 + 256; h0 += 64) {
        // W_r rows h0..h0+63, E values each, zero padded to 64 experts
        __syncthreads();
        if ((a.E & 7) == 0) {
            const int vrow = a.E / 8;   // 16-byte vectors per W_r row
            for (int i = threadIdx.x; i < 64 * 8; i += blockDim.x) {
                const int hh = i / 8, v = i % 8;
                uint4 q = make_uint4(0, 0, 0, 0);
                if (v < vrow) q = ld_nc_v4(a.Wr + (size_t)(h0 + hh) * a.E + v * 8);
                *reinterpret_cast<uint4 *>(&s_wr[hh][v * 8]) = q;
            }
        } else {
            for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
                const int hh = i / 64, e = i % 64;
                s_wr[hh][e] = e < a.E ? a.Wr[(size_t)(h0 + hh) * a.E + e] : f2bf(0.0f);
            }
        }
        __syncthreads();
        float acc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            if (ks < KS) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const bf16 *wr = &s_wr[nt * 8 + g][ks * 16 + 2 * c];
                    const uint32_t b0 = *reinterpret_cast<const uint32_t *>(wr);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t *>(wr + 8);
                    mma_16816_bf16(acc[nt], Ahi[ks], b0, b1);
                    mma_16816_bf16(acc[nt], Alo[ks], b0, b1);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            s_acc[warp][g][nt * 8 + 2 * c] = acc[nt][0];
            s_acc[warp][g][nt * 8 + 2 * c + 1] = acc[nt][1];
            s_acc[warp][g + 8][nt * 8 + 2 * c] = acc[nt][2];
            s_acc[warp][g + 8][nt * 8 + 2 * c + 1] = acc[nt][3];
        }
        __syncwarp();
        if (my_t < a.T) {
            const int hb = h0 + half * 32;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            for (int j0 = 0; j0 < a.k; j0 += 2) {
                const int nj = min(2, a.k - j0);
                uint4 q[2][4];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                    if (jj < nj) {
                        const int j = j0 + jj;
                        const int row = j < 32 ? rows[j] : checked_row(j);
                        const bf16 *src = a.dXs + (size_t)(row < 0 ? 0 : row) * a.H + hb;
#pragma unroll
                        for (int u = 0; u < 4; ++u) q[jj][u] = row < 0 ? make_uint4(0, 0, 0, 0) : ld_v4(src + u * 8);
                    }
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                    if (jj < nj) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t qq[4] = {q[jj][u].x, q[jj][u].y, q[jj][u].z, q[jj][u].w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                v[u * 8 + 2 * i] += bf16lo(qq[i]);
                                v[u * 8 + 2 * i + 1] += bf16hi(qq[i]);
                            }
                        }
                    }
            }
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                o[i] = pack_bf16x2(v[2 * i] + s_acc[warp][lane >> 1][half * 32 + 2 * i],
                                   v[2 * i + 1] + s_acc[warp][lane >> 1][half * 32 + 2 * i + 1]);
            bf16 *dst = a.dx + (size_t)my_t * a.H + hb;
#pragma unroll
            for (int u = 0; u < 4; ++u) st_v4(dst + u * 8, make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]));
        }
        __syncwarp();
    }
}

// dW_r partials on tensor cores: D[h][e] = sum_t x[t][h] dl[t][e] as m16n8k16
// MMAs with M = h, N = e, K = tokens. x is bf16 (exact); dlogits (fp32) enter as
// a bf16 high part plus a bf16 low part (about 16 significant bits), both
// products accumulate in fp32. Block = 64 h (warp w owns h 16w..16w+15) x all
// experts, tokens of split sp in chunks of 64 staged in shared memory: x as
// [t][h] (A fragments by ldmatrix.trans), dlogits transposed as [e][t] hi and lo
// (B fragments). The partial tile leaves through shared memory as [split][e][h].
constexpr int kWgTok = 64;
constexpr int kWgPad = 8;   // bf16 row padding: conflict-free fragment loads
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}
__global__ void __launch_bounds__(128) router_wgrad_part_kernel(RouterWgradArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    __shared__ __align__(16) bf16 s_x[kWgTok][64 + kWgPad];
    __shared__ __align__(16) bf16 s_hi[kMaxExperts][kWgTok + kWgPad];
    __shared__ __align__(16) bf16 s_lo[kMaxExperts][kWgTok + kWgPad];
    __shared__ __align__(16) float s_out[kMaxExperts][64 + 4];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int g = lane >> 2, c = lane & 3;
    const int hb = blockIdx.x * 64;
    const int sp = blockIdx.y;
    const int ts = ceil_div(a.T, a.splits);
    const int tb = sp * ts, te = min(a.T, tb + ts);
    const int EP = (a.E + 7) / 8 * 8;
    const int NT = EP / 8;
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
    // this lane's ldmatrix row: matrix q = lane / 8 covers h +8*(q&1), t +8*(q>>1)
    const int lq = lane >> 3, li = lane & 7;
    // the next chunk's x and dlogits are loaded into registers while this chunk
    // computes: x as 4 vectors per thread, dlogits as rows of token pairs with
    // lanes over experts (up to 64 -> 2 per lane, 8 pairs per warp)
    uint4 xr[4];
    float dr[8][2][2];   // [token pair][expert half][token of the pair]
    auto fetch = [&](int c0) {
        const int cn = min(kWgTok, te - c0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = threadIdx.x + 128 * u, tt = i >> 3, v = i & 7;
            xr[u] = tt < cn ? ld_nc_v4(a.x + (size_t)(c0 + tt) * a.H + hb + v * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int tt = 2 * (warp + 4 * u);
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const int e = lane + 32 * s2;
#pragma unroll
                for (int p = 0; p < 2; ++p)
                    dr[u][s2][p] = (tt + p < cn && e < a.E) ? __ldg(a.dlogits + (size_t)(c0 + tt + p) * a.E + e) : 0.0f;
            }
        }
    };
    if (tb < te) fetch(tb);
    for (int c0 = tb; c0 < te; c0 += kWgTok) {
        __syncthreads();   // the previous chunk's fragments have been read
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = threadIdx.x + 128 * u;
            *reinterpret_cast<uint4 *>(&s_x[i >> 3][(i & 7) * 8]) = xr[u];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int tt = 2 * (warp + 4 * u);
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const int e = lane + 32 * s2;
                if (e < EP) {
                    const uint32_t hi = pack_bf16x2(dr[u][s2][0], dr[u][s2][1]);
                    *reinterpret_cast<uint32_t *>(&s_hi[e][tt]) = hi;
                    *reinterpret_cast<uint32_t *>(&s_lo[e][tt]) =
                        pack_bf16x2(dr[u][s2][0] - bf16lo(hi), dr[u][s2][1] - bf16hi(hi));
                }
            }
        }
        __syncthreads();
        if (c0 + kWgTok < te) fetch(c0 + kWgTok);
#pragma unroll
        for (int ks = 0; ks < kWgTok / 16; ++ks) {
            uint32_t A[4];
            ldmatrix_x4_trans(A, &s_x[ks * 16 + li + 8 * (lq >> 1)][warp * 16 + 8 * (lq & 1)]);
            // ldmatrix.trans hands out matrices in the order (h0-7,t0-7) (h8-15,t0-7) (h0-7,t8-15) (h8-15,t8-15):
            // exactly the a0..a3 registers of the m16n8k16 A fragment
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                if (n < NT) {
                    const bf16 *ph = &s_hi[n * 8 + g][ks * 16 + 2 * c];
                    const bf16 *pl = &s_lo[n * 8 + g][ks * 16 + 2 * c];
                    mma_16816_bf16(acc[n], A, *reinterpret_cast<const uint32_t *>(ph),
                                   *reinterpret_cast<const uint32_t *>(ph + 8));
                    mma_16816_bf16(acc[n], A, *reinterpret_cast<const uint32_t *>(pl),
                                   *reinterpret_cast<const uint32_t *>(pl + 8));
                }
            }
        }
    }
    // D fragment: rows h = 16 warp + g (+8), columns e = 8n + 2c (+1)
#pragma unroll
    for (int n = 0; n < 8; ++n) {
        if (n < NT) {
            const int h = warp * 16 + g, e = n * 8 + 2 * c;
            s_out[e][h] = acc[n][0];
            s_out[e + 1][h] = acc[n][1];
            s_out[e][h + 8] = acc[n][2];
            s_out[e + 1][h + 8] = acc[n][3];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.E * 16; i += blockDim.x) {   // 16 float4 per expert row of 64 h
        const int e = i / 16, v = i % 16;
        const float4 q = *reinterpret_cast<const float4 *>(&s_out[e][v * 4]);
        *reinterpret_cast<float4 *>(a.part + ((size_t)sp * a.E + e) * a.H + hb + v * 4) = q;
    }
}

// dW_r[h][e] (+)= sum over splits in increasing order; thread per (e, h), h fastest,
// eight split loads in flight at a time.
__global__ void router_wgrad_reduce_kernel(RouterWgradArgs a) {
    pdl_wait();      // predecessor's outputs visible
    pdl_trigger();   // let the next kernel launch
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.H * a.E) return;
    const int e = i / a.H, h = i % a.H;
    const size_t stride = (size_t)a.E * a.H;
    float v = 0.0f;
    for (int sp0 = 0; sp0 < a.splits; sp0 += 8) {
        float p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) p[u] = sp0 + u < a.splits ? __ldg(a.part + (size_t)(sp0 + u) * stride + i) : 0.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u) v += p[u];
    }
    const size_t o = (size_t)h * a.E + e;
    a.dWr[o] = a.accumulate ? a.dWr[o] + v : v;
}

cudaError_t launch_router_bwd_dlogits(const RouterBwdArgs &rb, cudaStream_t s) {
    if (rb.T > 0) {
        cudaError_t e = launch_pdl(router_bwd_kernel, dim3(ceil_div(rb.T, 8)), dim3(256), 0, s, rb);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_reverse_dispatch(const RevDispatchArgs &rd, cudaStream_t s) {
    if (rd.T > 0) {
        // 128 registers: four blocks per SM, so the usual grid fits in one wave
        cudaError_t e = launch_pdl(reverse_dispatch_kernel, dim3(ceil_div(rd.T, kRdTokens), rd.H / 256), dim3(128), 0, s, rd);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const RouterWgradArgs &rw, cudaStream_t s) {
    dim3 grid(rw.H / 64, rw.splits);
    cudaError_t e = launch_pdl(router_wgrad_part_kernel, grid, dim3(128), 0, s, rw);
    if (e != cudaSuccess) return e;
    e = launch_pdl(router_wgrad_reduce_kernel, dim3(ceil_div(rw.H * rw.E, 256)), dim3(256), 0, s, rw);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
