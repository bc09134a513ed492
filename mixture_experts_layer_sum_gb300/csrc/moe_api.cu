// Host side of the C ABI declared in include/moe.h: argument checks, the
// execution plan (minibatch, macrobatches, ring), carving of the caller's
// workspace and saved buffers, TMA tensor maps, and the launch sequence of the
// forward and backward passes. Nothing here allocates device memory.
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "decode_ffn.cuh"
#include "grouped_gemm.cuh"
#include "mx_quant.cuh"
#include "nvfp4.cuh"
#include "route_kernels.cuh"

using namespace moe;

namespace {

thread_local std::string g_last_error;

moe_status_t fail(moe_status_t s, const std::string &msg) {
    g_last_error = msg;
    return s;
}

// ---------------------------------------------------------------- profiling
// Thread-local record of (kernel name, start event, end event) around every
// launch while moe_profile_begin is active.
struct ProfRec {
    const char *name;
    cudaEvent_t start, end;
};
struct Profiler {
    bool on = false;
    std::vector<ProfRec> recs;
};
thread_local Profiler g_prof;

struct ProfScope {
    ProfRec rec{};
    cudaStream_t stream;
    bool active;
    ProfScope(const char *name, cudaStream_t s) : stream(s), active(g_prof.on) {
        if (!active) return;
        rec.name = name;
        cudaEventCreate(&rec.start);
        cudaEventCreate(&rec.end);
        cudaEventRecord(rec.start, stream);
    }
    ~ProfScope() {
        if (!active) return;
        cudaEventRecord(rec.end, stream);
        g_prof.recs.push_back(rec);
    }
};

// bf16 grouped GEMMs run as CTA pairs (cta_group::2, 256-row tiles)
constexpr bool kPairGemm = true;
// MXFP8 CTA pairs (block-scaled cta_group::2); the GEMM2 dgrad keeps 1-CTA tiles with eight
// epilogue warps (its quantising SwiGLU backward: CTA pairs with four or eight epilogue warps
// measured slower)
constexpr bool kPairGemmFp8 = true;
inline bool pair_fp8(int op) { return kPairGemmFp8 && op != OP_BWD2; }
constexpr int kGemmBN1 = 256;   // GEMM1 tile: 128 rows x (128 a-columns + 128 b-columns)
// bf16 forward of at most kDecodeMaxTokens tokens through the decode kernel
constexpr bool kDecodePath = true;
constexpr int kGemmBM = 128;

// ---------------------------------------------------------------- planning

int query_num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

moe_status_t check_shape(const moe_config_t *c) {
    if (!c) return fail(MOE_ERR_INVALID_ARG, "config is NULL");
    if (c->T < 0 || c->H <= 0 || c->F <= 0 || c->E <= 0 || c->k <= 0)
        return fail(MOE_ERR_INVALID_ARG, "T must be >= 0 and H, F, E, k > 0");
    if (c->E > kMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "E > 64 experts is not supported");
    if (c->k > c->E) return fail(MOE_ERR_INVALID_ARG, "k > E");
    if (c->k > 32) return fail(MOE_ERR_UNSUPPORTED, "k > 32 is not supported");
    if (c->H % 256 || c->F % 256) return fail(MOE_ERR_UNSUPPORTED, "H and F must be multiples of 256");
    if (c->precision != MOE_PRECISION_BF16 && c->precision != MOE_PRECISION_MXFP8 &&
        c->precision != MOE_PRECISION_NVFP4)
        return fail(MOE_ERR_INVALID_ARG, "unknown precision");
    if (c->minibatch_rows < 0 || c->macrobatch_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "negative minibatch/macrobatch");
    if (c->forward_mode != MOE_FORWARD_PERSISTENT && c->forward_mode != MOE_FORWARD_PER_STAGE)
        return fail(MOE_ERR_INVALID_ARG, "unknown forward mode");
    const long long R = (long long)c->T * c->k;
    if (R > (1LL << 30) / 2) return fail(MOE_ERR_UNSUPPORTED, "T*k too large");
    return MOE_OK;
}

size_t a1024(size_t v) { return align_up(v, 1024); }

// Minimum minibatch: GEMM1 covers the 2F columns of [W1|W3] with tiles of
// 128 rows x 256 columns, so r rows give (r/128)(2F/256) tiles; two full waves
// on S SMs need r >= 2 S 128 256 / (2F).
int minibatch_floor(int num_sms, int F) {
    const long long num = 2LL * num_sms * kGemmBM * kGemmBN1;
    const long long den = 2LL * F;
    return (int)((num + den - 1) / den);
}

moe_status_t make_layout(const moe_config_t *c, Layout &L) {
    moe_status_t st = check_shape(c);
    if (st != MOE_OK) return st;
    std::memset(&L, 0, sizeof(L));
    L.T = c->T; L.H = c->H; L.F = c->F; L.E = c->E; L.k = c->k;
    L.R = c->T * c->k;
    L.precision = c->precision;
    L.num_sms = c->num_sms > 0 ? c->num_sms : query_num_sms();
    if (L.num_sms <= 0) return fail(MOE_ERR_CUDA, "could not query the SM count (no device?)");
    const int floor_rows = minibatch_floor(L.num_sms, c->F);
    L.minibatch_rows = c->minibatch_rows > 0 ? c->minibatch_rows : floor_rows;
    const bool mx = c->precision == MOE_PRECISION_MXFP8;
    const size_t xrow = mx ? (size_t)c->H + c->H / kMxBlock : 2 * (size_t)c->H;
    const size_t hrow = mx ? (size_t)c->F + c->F / kMxBlock : 2 * (size_t)c->F;
    const size_t yrow = 2 * (size_t)c->H;
    // The ring holds the dispatched token rows of the macrobatch in flight, in the layer's
    // compute format (article "O MoK do Cursor ...", section 02: a fixed-size token ring whose
    // slots the dispatch fills and which are reused once the experts and the combine are done
    // with them). MXFP8: E4M3 along H plus scales, in the workspace; bf16: the fused dispatch
    // writes the rows straight into the saved context (the backward's dW1/dW3 reads them
    // there), so the ring is a window of it. The macrobatch's FFN hidden rows and expert
    // outputs live in buffers of the same row count.
    const size_t ring_row_bytes = xrow;
    const int pad = (kRowPad - 1) * c->E;
    int Mb;
    if (c->macrobatch_tokens > 0) {
        Mb = c->macrobatch_tokens;
    } else if (c->ring_bytes == 0) {
        Mb = c->T > 0 ? c->T : 1;
    } else {
        // largest Mb whose padded rows fit the ring: (Mb*k + pad) * row_bytes <= ring_bytes.
        // One macrobatch at a time: every kernel waits for its predecessor on the stream to
        // complete (programmatic launches included), so macrobatch m+1's dispatch never runs
        // while macrobatch m's rows are still read, and a second ring half would buy no overlap.
        // whole 128-row tiles of padded rows, with room for the 1 KiB alignment of each ring buffer
        const size_t usable = c->ring_bytes > 8 * 1024 ? c->ring_bytes - 8 * 1024 : 0;
        const long long rows = (long long)(usable / ring_row_bytes) / kRowPad * kRowPad - pad;
        if (rows < c->k) return fail(MOE_ERR_UNSUPPORTED, "ring_bytes too small for one token per macrobatch");
        Mb = (int)(rows / c->k);
    }
    if (c->T > 0 && Mb > c->T) Mb = c->T;
    if (Mb <= 0) Mb = 1;
    L.Mb = Mb;
    L.nM = c->T > 0 ? ceil_div(c->T, Mb) : 1;
    L.ring_halves = 1;
    const long long rows_pad_max = (long long)L.R + (long long)L.nM * pad;
    const long long half_rows = (long long)std::min<long long>((long long)Mb * c->k, L.R) + pad;
    L.rows_pad_max = (int)align_up((size_t)std::max<long long>(rows_pad_max, kRowPad), kRowPad);
    L.half_rows = L.nM > 1 ? (int)align_up((size_t)half_rows, kRowPad) : L.rows_pad_max;
    L.chunks_per_mb = std::max(1, ceil_div(std::min(Mb, std::max(c->T, 1)) * c->k, kSchedChunk));
    L.nchunks = c->T > 0 ? L.nM * L.chunks_per_mb : 0;
    // router-weight gradient: about eight blocks per SM over (H/64) x splits
    L.dwr_splits = std::max(1, std::min(ceil_div(4 * L.num_sms, c->H / 64), ceil_div(std::max(c->T, 1), 64)));

    const size_t R = L.R, T = L.T, E = L.E, H = L.H, F = L.F, nM = L.nM, rp = L.rows_pad_max;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = a1024(o + std::max<size_t>(bytes, 1)); return at; };
    L.s_ids = take(4 * R);
    L.s_w = take(4 * R);
    L.s_probs = take(4 * T * E);
    L.s_counts = take(4 * nM * E);
    L.s_offsets = take(4 * nM * (E + 1));
    L.s_offp = take(4 * (nM * E + 1));
    L.s_s2sorted = take(4 * R);
    L.s_sorted2s = take(4 * R);
    L.s_slot_row = take(4 * R);
    L.s_row_slot = take(4 * rp);
    L.s_a = take(2 * rp * F);
    L.s_b = take(2 * rp * F);
    // bf16: the dispatched x rows stay in the saved context at their global padded rows (the
    // order the dW1/dW3 GEMM reads X in), so the backward never gathers them again
    L.keep_x = !mx;
    L.s_xs = L.keep_x ? take(2 * rp * H) : 0;
    L.saved_bytes = o;

    o = 0;
    L.w_status = take(256);
    L.w_chunk_counts = take(4 * std::max(L.nchunks, 1) * E);
    L.w_chunk_base = take(4 * std::max(L.nchunks, 1) * E);
    const size_t EP = (E + 7) / 8 * 8;
    L.w_wrt = take(2 * EP * H);
    L.w_offp = take(4 * (nM * E + 1));
    L.mb_rows = (int)align_up((size_t)std::max(L.minibatch_rows, kRowPad), kRowPad);
    // per macrobatch: per-minibatch ready rows + the claim counter (zeroed by the schedule scan)
    L.w_ready = take(4 * (size_t)L.nM * ((size_t)L.half_rows / kRowPad + 2));
    L.tile_list_max = L.rows_pad_max / kRowPad + L.nM * L.E;
    L.w_tiles128 = take(16 * (size_t)L.tile_list_max);
    L.w_tiles256 = take(16 * (size_t)L.tile_list_max);
    L.w_tile_counts = take(2 * 4);
    L.w_decode = take(4 * (1 + (size_t)L.E));
    // persistent forward: tile list, per-macrobatch counts, counters zeroed per call (the
    // per-macrobatch counters and the per-128-row-block h counters, one contiguous range)
    L.mega_list_max = ((size_t)L.rows_pad_max / 256 + (size_t)L.nM * L.E) * ((size_t)L.F / 128 + (size_t)L.H / 256);
    L.w_mega_list = take(16 * L.mega_list_max);
    L.w_mega_meta = take(16 * (size_t)L.nM);
    L.w_mega_count = take(4);
    L.w_mega_cnt = o;
    L.mega_zero_bytes = 4 * ((size_t)L.nM * MEGA_NCNT + (size_t)L.rows_pad_max / kRowPad);
    L.w_mega_hready = L.w_mega_cnt + 4 * (size_t)L.nM * MEGA_NCNT;
    take(L.mega_zero_bytes);
    // few bf16 tokens in one macrobatch: every expert holds at most T <= 128 rows, and the
    // forward streams each expert's weights once through the decode kernel
    L.decode = kDecodePath && !mx && c->T > 0 && c->T <= kDecodeMaxTokens && L.nM == 1;
    if (c->precision == MOE_PRECISION_NVFP4 && c->T > 0 && !L.decode)
        return fail(MOE_ERR_UNSUPPORTED, "NVFP4 weights run the forward of at most 128 tokens in one macrobatch");
    const size_t region = o;
    const size_t ring_rows = (size_t)L.half_rows * L.ring_halves;
    // forward region: the token ring (MXFP8), then the macrobatch's h and Y rows
    o = region;
    L.w_ringX = take(L.keep_x ? 0 : ring_rows * (mx ? H : 2 * H));   // kept X rows: in saved
    L.w_ringXs = mx ? take(ring_rows * (H / kMxBlock)) : 0;
    L.ring_bytes = L.keep_x ? ring_rows * xrow : o - region;
    L.w_ringH = take(ring_rows * (mx ? F : 2 * F));
    L.w_ringHs = mx ? take(ring_rows * (F / kMxBlock)) : 0;
    L.w_ringY = take(ring_rows * 2 * H);
    const size_t fwd_end = o;
    // backward region (X rows: bf16 in saved, MXFP8 only along the tokens; dout rows: bf16 only,
    // MXFP8 gathers them straight into its two quantised copies)
    o = region;
    L.w_Gin = take(mx ? 0 : rp * 2 * H);
    // bf16 da, db, h.w rows: the bf16 weight gradients' operands (MXFP8 writes them quantised
    // along the rows straight from the GEMM2 dgrad epilogue instead)
    L.w_da = take(mx ? 0 : rp * 2 * F);
    L.w_db = take(mx ? 0 : rp * 2 * F);
    L.w_hw = take(mx ? 0 : rp * 2 * F);
    L.w_dXs = take(rp * 2 * H);
    L.w_dwpart = take(4 * rp * (F / 128));
    L.w_dlogits = take(4 * T * E);
    L.w_dwr_part = take(4 * (size_t)L.dwr_splits * H * E);
    if (mx) {
        const size_t qh = rp * H, qf = rp * F;
        L.w_Ginq = take(qh); L.w_Ginq_s = take(qh / kMxBlock);
        L.w_daq = take(qf); L.w_daq_s = take(qf / kMxBlock);
        L.w_dbq = take(qf); L.w_dbq_s = take(qf / kMxBlock);
        L.w_GinT = take(qh); L.w_GinT_s = take(qh / kMxBlock);
        L.w_XsT = take(qh); L.w_XsT_s = take(qh / kMxBlock);
        L.w_hwT = take(qf); L.w_hwT_s = take(qf / kMxBlock);
        L.w_daT = take(qf); L.w_daT_s = take(qf / kMxBlock);
        L.w_dbT = take(qf); L.w_dbT_s = take(qf / kMxBlock);
    }
    const size_t bwd_end = o;
    L.workspace_bytes = std::max(fwd_end, bwd_end);
    return MOE_OK;
}

// ---------------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 map over a row-major [rows, cols] array; box = 64 columns (128 B,
// the 128-byte swizzle span) x box_rows rows.
bool make_map(CUtensorMap *m, const void *base, size_t rows, size_t cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over a row-major [rows, cols] array of bytes (E4M3 codes); box = 128
// columns (the 128-byte swizzle span) x box_rows rows.
bool make_map_u8(CUtensorMap *m, const void *base, size_t rows, size_t cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MXFP8 scale atoms of a [rows, K] operand stored as 512-byte atoms: the array viewed as
// [bytes / 128][128] bytes, no swizzle; box 128 x 4 = one atom (row = byte offset / 128)
bool make_map_atoms(CUtensorMap *m, const void *base, size_t bytes) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || bytes < 512) return false;
    cuuint64_t dims[2] = {128, bytes / 128};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 4};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map of an MN-major bf16 operand stored row-major [rows (K), cols (M or N)]:
// dims (64 columns, rows, cols / 64 chunks) with the chunk stride 128 B, box
// (64, box_rows, chunks): one load lands `chunks` 64-column slabs of box_rows
// rows one after another, the layout the MN-major UMMA descriptor expects.
bool make_map_mn(CUtensorMap *m, const void *base, size_t rows, size_t cols, int box_rows, int chunks) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows == 0) return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// fp32 [rows, cols] output map for TMA stores of 32 x 32 boxes (128-byte swizzle)
bool make_map_f32_out(CUtensorMap *m, void *base, size_t rows, size_t cols) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 [rows, cols] output map for TMA stores of 32 x 32 boxes (64 B rows, 64-byte swizzle:
// the staging layout of the epilogues)
bool make_map_bf16_out(CUtensorMap *m, void *base, size_t rows, size_t cols) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MXFP8 weight copies made by moe_quantize_weights, each K-major for one GEMM:
//   w1t, w3t: W1^T, W3^T [E][F][H] along H (GEMM1)     w2t: W2^T [E][H][F] along F (GEMM2)
//   w2q:      W2 [E][F][H] along H (GEMM2 dgrad)       w1q, w3q: W1, W3 [E][H][F] along F (GEMM1 dgrad)
// Each is E*H*F bytes of E4M3 codes followed by E*H*F/32 bytes of scale atoms.
struct QwLayout {
    size_t codes[6], scales[6], bytes;
};
enum { QW_W1T = 0, QW_W3T, QW_W2T, QW_W2Q, QW_W1Q, QW_W3Q };
QwLayout qw_layout(const moe_config_t *c) {
    QwLayout q{};
    const size_t n = (size_t)c->E * c->H * c->F;
    size_t o = 0;
    for (int i = 0; i < 6; ++i) {
        q.codes[i] = o;
        o = align_up(o + n, 1024);
        q.scales[i] = o;
        o = align_up(o + n / kMxBlock, 1024);
    }
    q.bytes = o;
    return q;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspace and saved buffers may start anywhere: the library uses them from
// the next 1024-byte boundary on (TMA tiles and the layout want that), and the
// size queries include that slack.
constexpr size_t kBaseSlack = 1024;
void *align_base(void *p) {
    return reinterpret_cast<void *>((reinterpret_cast<uintptr_t>(p) + kBaseSlack - 1) & ~uintptr_t(kBaseSlack - 1));
}
const void *align_base(const void *p) { return align_base(const_cast<void *>(p)); }
bool fits(const void *base, size_t bytes, size_t need) {
    const size_t lost = reinterpret_cast<uintptr_t>(align_base(base)) - reinterpret_cast<uintptr_t>(base);
    return bytes >= lost && bytes - lost >= need;
}

template <class T>
T *at(void *base, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(base) + off); }
template <class T>
const T *at(const void *base, size_t off) { return reinterpret_cast<const T *>(static_cast<const char *>(base) + off); }

moe_status_t cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MOE_OK;
    return fail(MOE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

unsigned long long budget_ns(const moe_config_t *c) {
    return (unsigned long long)(c->timeout_ms ? c->timeout_ms : 2000u) * 1000000ull;
}

SchedArgs sched_args(const Layout &L, const int32_t *ids, void *ws, int32_t *counts, int32_t *offsets, int32_t *offp,
                     int32_t *s2s, int32_t *s2sorted, int32_t *slot_row, int32_t *row_slot) {
    SchedArgs a{};
    a.ids = ids;
    a.T = L.T; a.k = L.k; a.E = L.E; a.Mb = L.Mb; a.nM = L.nM;
    a.chunks_per_mb = L.chunks_per_mb; a.nchunks = L.nchunks;
    a.chunk_counts = at<int>(ws, L.w_chunk_counts);
    a.chunk_base = at<int>(ws, L.w_chunk_base);
    a.counts = counts; a.offsets = offsets; a.offp = offp;
    a.sorted_to_slot = s2s; a.slot_to_sorted = s2sorted;
    a.slot_row = slot_row; a.row_slot = row_slot;
    a.status = at<int>(ws, L.w_status);
    return a;
}

GemmArgs gemm_base(const Layout &L, void *ws, const int32_t *offp, const moe_config_t *c) {
    GemmArgs g;
    std::memset(&g, 0, sizeof(g));
    g.offp = offp;
    g.E = L.E; g.nM = L.nM; g.H = L.H; g.F = L.F;
    g.status = at<int>(ws, L.w_status);
    g.budget_ns = budget_ns(c);
    g.nslots = L.R;
    return g;
}

}  // namespace

namespace moe {
void set_last_error(const char *msg) { g_last_error = msg; }
}  // namespace moe

// ======================================================================== ABI

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_last_error_string(void) { return g_last_error.c_str(); }

moe_status_t moe_profile_begin(void) {
    for (auto &r : g_prof.recs) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.end);
    }
    g_prof.recs.clear();
    g_prof.on = true;
    return MOE_OK;
}

int moe_profile_end(moe_kernel_time_t *out, int max_entries) {
    g_prof.on = false;
    std::vector<moe_kernel_time_t> rows;
    int rc = 0;
    for (auto &r : g_prof.recs) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.end) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.end) != cudaSuccess)
            rc = -(int)MOE_ERR_CUDA;
        size_t i = 0;
        for (; i < rows.size(); ++i)
            if (std::strncmp(rows[i].name, r.name, sizeof(rows[i].name)) == 0) break;
        if (i == rows.size()) {
            moe_kernel_time_t t{};
            std::strncpy(t.name, r.name, sizeof(t.name) - 1);
            rows.push_back(t);
        }
        rows[i].launches += 1;
        rows[i].total_ms += ms;
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.end);
    }
    g_prof.recs.clear();
    if (rc < 0) return fail(MOE_ERR_CUDA, "profiling events failed"), rc;
    for (size_t i = 0; i < rows.size() && (int)i < max_entries; ++i) out[i] = rows[i];
    return (int)rows.size();
}

moe_status_t moe_plan(const moe_config_t *cfg, moe_plan_t *plan) {
    if (!plan) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    Layout L;
    moe_status_t st = make_layout(cfg, L);
    if (st != MOE_OK) return st;
    plan->num_sms = L.num_sms;
    plan->minibatch_rows = L.minibatch_rows;
    plan->macrobatch_tokens = L.Mb;
    plan->num_macrobatches = L.nM;
    plan->rows_padded_max = L.rows_pad_max;
    plan->ring_rows = L.half_rows * L.ring_halves;
    plan->ring_bytes = L.ring_bytes;
    plan->workspace_bytes = L.workspace_bytes + kBaseSlack;
    plan->saved_bytes = L.saved_bytes + kBaseSlack;
    plan->qweights_bytes = 0;
    return MOE_OK;
}

moe_status_t moe_buffer_location(const moe_config_t *cfg, int which, int *in_saved, size_t *offset,
                                 size_t *bytes) {
    if (!in_saved || !offset || !bytes) return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
    Layout L;
    moe_status_t st = make_layout(cfg, L);
    if (st != MOE_OK) return st;
    const bool mx = L.precision == MOE_PRECISION_MXFP8;
    const size_t rp = L.rows_pad_max, H = L.H, F = L.F;
    const size_t ring_rows = (size_t)L.half_rows * L.ring_halves;
    struct Loc { int saved; size_t off, bytes; int only; };   // only: 1 MXFP8, 2 bf16 configurations
    Loc loc{};
    switch (which) {
        case MOE_BUF_PADDED_OFFSETS: loc = {1, L.s_offp, 4 * ((size_t)L.nM * L.E + 1), false}; break;
        case MOE_BUF_ROW_SLOT: loc = {1, L.s_row_slot, 4 * rp, false}; break;
        case MOE_BUF_SLOT_ROW: loc = {1, L.s_slot_row, 4 * (size_t)L.R, false}; break;
        case MOE_BUF_A: loc = {1, L.s_a, 2 * rp * F, false}; break;
        case MOE_BUF_B: loc = {1, L.s_b, 2 * rp * F, false}; break;
        case MOE_BUF_RING_X:
            loc = L.keep_x ? Loc{1, L.s_xs, 2 * rp * H, false} : Loc{0, L.w_ringX, ring_rows * (mx ? H : 2 * H), false};
            break;
        case MOE_BUF_RING_X_SCALES: loc = {0, L.w_ringXs, ring_rows * H / kMxBlock, true}; break;
        case MOE_BUF_RING_H: loc = {0, L.w_ringH, ring_rows * (mx ? F : 2 * F), false}; break;
        case MOE_BUF_RING_H_SCALES: loc = {0, L.w_ringHs, ring_rows * F / kMxBlock, true}; break;
        case MOE_BUF_DA: loc = {0, L.w_da, 2 * rp * F, 2}; break;
        case MOE_BUF_DB: loc = {0, L.w_db, 2 * rp * F, 2}; break;
        case MOE_BUF_HW: loc = {0, L.w_hw, 2 * rp * F, 2}; break;
        case MOE_BUF_DY_ROWS: loc = {0, L.w_Ginq, rp * H, true}; break;
        case MOE_BUF_DY_ROWS_SCALES: loc = {0, L.w_Ginq_s, rp * H / kMxBlock, true}; break;
        case MOE_BUF_DA_ROWS: loc = {0, L.w_daq, rp * F, true}; break;
        case MOE_BUF_DA_ROWS_SCALES: loc = {0, L.w_daq_s, rp * F / kMxBlock, true}; break;
        case MOE_BUF_DB_ROWS: loc = {0, L.w_dbq, rp * F, true}; break;
        case MOE_BUF_DB_ROWS_SCALES: loc = {0, L.w_dbq_s, rp * F / kMxBlock, true}; break;
        case MOE_BUF_X_TOKENS: loc = {0, L.w_XsT, rp * H, true}; break;
        case MOE_BUF_X_TOKENS_SCALES: loc = {0, L.w_XsT_s, rp * H / kMxBlock, true}; break;
        case MOE_BUF_DY_TOKENS: loc = {0, L.w_GinT, rp * H, true}; break;
        case MOE_BUF_DY_TOKENS_SCALES: loc = {0, L.w_GinT_s, rp * H / kMxBlock, true}; break;
        case MOE_BUF_HW_TOKENS: loc = {0, L.w_hwT, rp * F, true}; break;
        case MOE_BUF_HW_TOKENS_SCALES: loc = {0, L.w_hwT_s, rp * F / kMxBlock, true}; break;
        case MOE_BUF_DA_TOKENS: loc = {0, L.w_daT, rp * F, true}; break;
        case MOE_BUF_DA_TOKENS_SCALES: loc = {0, L.w_daT_s, rp * F / kMxBlock, true}; break;
        case MOE_BUF_DB_TOKENS: loc = {0, L.w_dbT, rp * F, true}; break;
        case MOE_BUF_DB_TOKENS_SCALES: loc = {0, L.w_dbT_s, rp * F / kMxBlock, true}; break;
        default: return fail(MOE_ERR_INVALID_ARG, "unknown buffer");
    }
    if (loc.only == 1 && !mx) return fail(MOE_ERR_UNSUPPORTED, "buffer exists in MXFP8 configurations only");
    if (loc.only == 2 && mx) return fail(MOE_ERR_UNSUPPORTED, "buffer exists in bf16 configurations only");
    *in_saved = loc.saved;
    *offset = loc.off;
    *bytes = loc.bytes;
    return MOE_OK;
}

size_t moe_workspace_size(const moe_config_t *cfg) {
    Layout L;
    return make_layout(cfg, L) == MOE_OK ? L.workspace_bytes + kBaseSlack : 0;
}

size_t moe_saved_size(const moe_config_t *cfg) {
    Layout L;
    return make_layout(cfg, L) == MOE_OK ? L.saved_bytes + kBaseSlack : 0;
}

size_t moe_qweights_size(const moe_config_t *cfg) {
    if (check_shape(cfg) != MOE_OK) return 0;
    if (cfg->precision == MOE_PRECISION_NVFP4) return nv_layout(cfg->E, cfg->H, cfg->F).bytes + kBaseSlack;
    if (cfg->precision != MOE_PRECISION_MXFP8) return 0;
    return qw_layout(cfg).bytes + kBaseSlack;
}

moe_status_t moe_quantize_weights(const moe_config_t *cfg, const void *W1, const void *W3, const void *W2,
                                  void *qweights, size_t qweights_bytes, moe_stream_t stream) {
    moe_status_t st = check_shape(cfg);
    if (st != MOE_OK) return st;
    if (cfg->precision == MOE_PRECISION_BF16) return fail(MOE_ERR_UNSUPPORTED, "weight quantisation is for MXFP8 and NVFP4 configs");
    if (!W1 || !W3 || !W2 || !qweights) return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
    if (cfg->precision == MOE_PRECISION_NVFP4) {
        const NvLayout nl = nv_layout(cfg->E, cfg->H, cfg->F);
        if (!fits(qweights, qweights_bytes, nl.bytes)) return fail(MOE_ERR_WORKSPACE, "qweights buffer too small");
        const void *ptrs[] = {W1, W3, W2};
        for (const void *p : ptrs)
            if (!aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
        const int sms = cfg->num_sms > 0 ? cfg->num_sms : query_num_sms();
        if (sms <= 0) return fail(MOE_ERR_CUDA, "could not query the SM count");
        ProfScope ps("quantize_weights", (cudaStream_t)stream);
        return cuda_check(launch_nv_quantize((const bf16 *)W1, (const bf16 *)W3, (const bf16 *)W2,
                                             static_cast<uint8_t *>(align_base(qweights)), nl, cfg->E, cfg->H,
                                             cfg->F, sms, (cudaStream_t)stream),
                          "NVFP4 weight quantise launch");
    }
    const QwLayout q = qw_layout(cfg);
    if (!fits(qweights, qweights_bytes, q.bytes)) return fail(MOE_ERR_WORKSPACE, "qweights buffer too small");
    const void *ptrs16[] = {W1, W3, W2};
    for (const void *p : ptrs16)
        if (!aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    uint8_t *qw = static_cast<uint8_t *>(align_base(qweights));
    cudaStream_t s = (cudaStream_t)stream;
    const int E = cfg->E, H = cfg->H, F = cfg->F;
    int sms = cfg->num_sms > 0 ? cfg->num_sms : query_num_sms();
    if (sms <= 0) return fail(MOE_ERR_CUDA, "could not query the SM count");
    ProfScope ps("quantize_weights", s);
    // transposed copies (contraction axis = rows of the stored weight)
    const struct { const void *src; int idx, R, C; } tr[3] = {{W1, QW_W1T, H, F}, {W3, QW_W3T, H, F}, {W2, QW_W2T, F, H}};
    for (const auto &t : tr) {
        MxTransposeArgs a{};
        a.src = (const bf16 *)t.src; a.codes = qw + q.codes[t.idx]; a.scales = qw + q.scales[t.idx];
        a.R = t.R; a.C = t.C; a.r_limit_ptr = nullptr;
        st = cuda_check(launch_mx_transpose(a, E, s), "weight transpose-quantise launch");
        if (st != MOE_OK) return st;
    }
    // row-wise copies (contraction axis = columns of the stored weight)
    const struct { const void *src; int idx, rows, C; } rw[3] = {{W2, QW_W2Q, E * F, H}, {W1, QW_W1Q, E * H, F}, {W3, QW_W3Q, E * H, F}};
    for (const auto &t : rw) {
        MxRowsArgs a{};
        a.src = (const bf16 *)t.src; a.codes = qw + q.codes[t.idx]; a.scales = qw + q.scales[t.idx];
        a.nrows = t.rows; a.C = t.C;
        st = cuda_check(launch_mx_rows(a, t.rows, sms, s), "weight quantise launch");
        if (st != MOE_OK) return st;
    }
    return MOE_OK;
}

moe_status_t moe_reset_status(void *workspace, moe_stream_t stream) {
    if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    return cuda_check(cudaMemsetAsync(align_base(workspace), 0, 256, (cudaStream_t)stream), "cudaMemsetAsync(status)");
}

moe_status_t moe_query_status(void *workspace, moe_stream_t stream) {
    if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    moe_status_t st = cuda_check(cudaStreamSynchronize((cudaStream_t)stream), "cudaStreamSynchronize");
    if (st != MOE_OK) return st;
    int v = 0;
    void *status = align_base(workspace);
    st = cuda_check(cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost), "cudaMemcpy(status)");
    if (st != MOE_OK) return st;
    st = cuda_check(cudaMemset(status, 0, sizeof(int)), "cudaMemset(status)");
    if (st != MOE_OK) return st;
    if (v == MOE_ERR_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a device-side wait ran out of time");
    if (v != 0) return fail(MOE_ERR_INTERNAL, "a device-side check failed (status " + std::to_string(v) + ")");
    return MOE_OK;
}

moe_status_t moe_schedule(const moe_config_t *cfg, const int32_t *topk_ids, int32_t *counts, int32_t *offsets,
                          int32_t *sorted_to_slot, int32_t *slot_to_sorted, void *workspace, size_t workspace_bytes,
                          moe_stream_t stream) {
    Layout L;
    moe_status_t st = make_layout(cfg, L);
    if (st != MOE_OK) return st;
    if (!counts || !offsets || !workspace || (L.R > 0 && (!topk_ids || !sorted_to_slot || !slot_to_sorted)))
        return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
    if (!fits(workspace, workspace_bytes, L.workspace_bytes)) return fail(MOE_ERR_WORKSPACE, "workspace too small");
    workspace = align_base(workspace);
    cudaStream_t s = (cudaStream_t)stream;
    st = cuda_check(cudaMemsetAsync(at<int>(workspace, L.w_status), 0, 256, s), "status clear");
    if (st != MOE_OK) return st;
    int32_t *offp = at<int32_t>(workspace, L.w_offp);   // padded run starts (scratch)
    SchedArgs a = sched_args(L, topk_ids, workspace, counts, offsets, offp, sorted_to_slot, slot_to_sorted, nullptr,
                             nullptr);
    {
        ProfScope ps("schedule", s);
        st = cuda_check(launch_schedule(a, s), "schedule launch");
    }
    return st;
}

moe_status_t moe_forward(const moe_config_t *cfg, const void *x, const void *W_r, const float *bias, const void *W1,
                         const void *W3, const void *W2, const void *qweights, void *out, int32_t *topk_ids,
                         float *topk_w, void *saved, size_t saved_bytes, void *workspace, size_t workspace_bytes,
                         moe_stream_t stream) {
    Layout L;
    moe_status_t st = make_layout(cfg, L);
    if (st != MOE_OK) return st;
    if (cfg->precision != MOE_PRECISION_BF16 && !qweights)
        return fail(MOE_ERR_INVALID_ARG, "MXFP8 and NVFP4 forwards need qweights");
    if (!W_r || !W1 || !W3 || !W2 || !saved || !workspace || (L.T > 0 && (!x || !out || !topk_ids || !topk_w)))
        return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
    if (!fits(saved, saved_bytes, L.saved_bytes)) return fail(MOE_ERR_WORKSPACE, "saved buffer too small");
    if (!fits(workspace, workspace_bytes, L.workspace_bytes)) return fail(MOE_ERR_WORKSPACE, "workspace too small");
    saved = align_base(saved);
    workspace = align_base(workspace);
    const void *ptrs16[] = {x, W_r, W1, W3, W2, out};
    for (const void *p : ptrs16)
        if (p && !aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    void *ws = workspace;
    st = cuda_check(cudaMemsetAsync(at<int>(ws, L.w_status), 0, 256, s), "status clear");
    if (st != MOE_OK) return st;

    int32_t *s_ids = at<int32_t>(saved, L.s_ids);
    float *s_w = at<float>(saved, L.s_w);
    float *s_probs = at<float>(saved, L.s_probs);
    int32_t *s_offp = at<int32_t>(saved, L.s_offp);
    int32_t *s_slot_row = at<int32_t>(saved, L.s_slot_row);
    int32_t *s_row_slot = at<int32_t>(saved, L.s_row_slot);
    bf16 *s_a = at<bf16>(saved, L.s_a);
    bf16 *s_b = at<bf16>(saved, L.s_b);

    // 1. router
    RouterArgs ra{};
    ra.x = (const bf16 *)x; ra.Wr = (const bf16 *)W_r; ra.bias = bias;
    ra.WrT = at<bf16>(ws, L.w_wrt);
    ra.T = L.T; ra.H = L.H; ra.E = L.E; ra.k = L.k;
    ra.probs = s_probs; ra.ids = topk_ids; ra.w = topk_w; ra.ids2 = s_ids; ra.w2 = s_w;
    {
        ProfScope ps("router_topk", s);
        st = cuda_check(launch_router(ra, s), "router launch");
    }
    if (st != MOE_OK) return st;

    // 2. schedule
    SchedArgs sa = sched_args(L, s_ids, ws, at<int32_t>(saved, L.s_counts), at<int32_t>(saved, L.s_offsets), s_offp,
                              at<int32_t>(saved, L.s_sorted2s), at<int32_t>(saved, L.s_s2sorted), s_slot_row,
                              s_row_slot);
    sa.ready = at<int>(ws, L.w_ready);   // GEMM1's per-minibatch counters of every macrobatch
    sa.ready_n = L.nM * (L.half_rows / kRowPad + 2);
    // the counters of the kernel that follows: the decode kernel's claim and h counts, or the
    // persistent forward's hand-off counters (zeroed by the scan: no memset in the chain)
    if (L.decode) {
        sa.zero[0] = at<int>(ws, L.w_decode);
        sa.zero_n[0] = 1 + L.E;
    } else if (cfg->forward_mode == MOE_FORWARD_PERSISTENT && L.T > 0) {
        sa.zero[0] = at<int>(ws, L.w_mega_cnt);
        sa.zero_n[0] = (int)(L.mega_zero_bytes / 4);
    }
    {
        ProfScope ps("schedule", s);
        st = cuda_check(launch_schedule(sa, s), "schedule launch");
    }
    if (st != MOE_OK) return st;
    if ((cfg->fault_mask & MOE_FAULT_GEMM1_READY) && L.T > 0) {
        // failure-detection tests: the first minibatch's ready count (zeroed by the schedule)
        // becomes a large negative number that the gather's additions cannot lift to its
        // target; the claim counter next to it is untouched, so every gather stays in bounds
        st = cuda_check(cudaMemsetAsync(at<int>(ws, L.w_ready), 0x80, sizeof(int), s), "fault injection");
        if (st != MOE_OK) return st;
    }

    const bool mx = cfg->precision == MOE_PRECISION_MXFP8;
    if (L.decode) {
        // 3'. few tokens: dispatch into the saved x rows -> decode FFN (both GEMMs, weights
        // streamed once) -> combine
        bf16 *xs = at<bf16>(saved, L.s_xs);
        bf16 *ringH = at<bf16>(ws, L.w_ringH), *ringY = at<bf16>(ws, L.w_ringY);
        const size_t rp = L.rows_pad_max;
        DecodeArgs da;
        std::memset(&da, 0, sizeof(da));
        if (!make_map_mn(&da.w1, W1, (size_t)L.E * L.H, L.F, 64, 2) || !make_map_mn(&da.w3, W3, (size_t)L.E * L.H, L.F, 64, 2) ||
            !make_map_mn(&da.w2, W2, (size_t)L.E * L.F, L.H, 64, 2) || !make_map(&da.x, xs, rp, L.H, 32) ||
            !make_map(&da.h, ringH, rp, L.F, 32))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        da.offp = s_offp; da.counts = at<int32_t>(saved, L.s_counts);
        da.a = s_a; da.b = s_b; da.hrows = ringH; da.y = ringY;
        int *dc = at<int>(ws, L.w_decode);
        da.claim = dc; da.hdone = dc + 1;
        da.E = L.E; da.H = L.H; da.F = L.F; da.nb = ceil_div(L.T, 32);
        da.status = at<int>(ws, L.w_status); da.budget_ns = budget_ns(cfg);
        const bool nv = cfg->precision == MOE_PRECISION_NVFP4;
        if (nv) {
            const NvLayout nl = nv_layout(L.E, L.H, L.F);
            da.nvq = static_cast<const uint8_t *>(align_base(qweights));
            da.nv_w13 = nl.w13;
            da.nv_w2 = nl.w2;
            da.nv_g = reinterpret_cast<const float *>(da.nvq + nl.gscale);
        }
        DispatchArgs d{};
        d.src = (const bf16 *)x; d.dst = xs; d.row_slot = s_row_slot; d.offp = s_offp;
        d.beg = 0; d.end = L.E; d.dst_row0 = 0; d.H = L.H; d.k = L.k;
        d.nslots = L.R; d.status = at<int>(ws, L.w_status);
        {
            ProfScope ps("dispatch", s);
            st = cuda_check(launch_dispatch(d, L.rows_pad_max, L.num_sms, s), "dispatch launch");
        }
        if (st != MOE_OK) return st;
        {
            ProfScope ps(nv ? "decode_ffn_nvfp4" : "decode_ffn", s);
            st = cuda_check(nv ? launch_decode_nv(da, L.num_sms, s) : launch_decode_ffn(da, L.num_sms, s),
                            "decode FFN launch");
        }
        if (st != MOE_OK) return st;
        CombineArgs ca{};
        ca.Y = ringY; ca.slot_row = s_slot_row; ca.offp = s_offp; ca.w = s_w; ca.out = (bf16 *)out;
        ca.t0 = 0; ca.t1 = L.T; ca.k = L.k; ca.H = L.H; ca.E = L.E; ca.m = 0; ca.ring_base = 0;
        ca.status = at<int>(ws, L.w_status);
        ProfScope ps("combine", s);
        return cuda_check(launch_combine(ca, L.num_sms, s), "combine launch");
    }

    // 3. dispatch -> GEMM1+SwiGLU -> GEMM2 -> combine: one persistent launch, or per macrobatch
    bf16 *ringX = L.keep_x ? at<bf16>(saved, L.s_xs) : at<bf16>(ws, L.w_ringX);
    bf16 *ringH = at<bf16>(ws, L.w_ringH), *ringY = at<bf16>(ws, L.w_ringY);
    uint8_t *ringXq = at<uint8_t>(ws, L.w_ringX), *ringHq = at<uint8_t>(ws, L.w_ringH);
    uint8_t *ringXs = mx ? at<uint8_t>(ws, L.w_ringXs) : nullptr, *ringHs = mx ? at<uint8_t>(ws, L.w_ringHs) : nullptr;
    const size_t ring_rows = (size_t)L.half_rows * L.ring_halves;
    GemmArgs g1 = gemm_base(L, ws, s_offp, cfg), g2 = gemm_base(L, ws, s_offp, cfg);
    if (!mx) {
        const int nb2 = kPairGemm ? 2 : 4;   // 64-column chunks of GEMM2's B per CTA
        // kept x rows: GEMM1's A rows are global padded rows of the saved context
        if (!make_map(&g1.a0, ringX, L.keep_x ? (size_t)L.rows_pad_max : ring_rows, L.H, 128) ||
            !make_map_mn(&g1.b0, W1, (size_t)L.E * L.H, L.F, 64, 2) ||
            !make_map_mn(&g1.b1, W3, (size_t)L.E * L.H, L.F, 64, 2) || !make_map(&g2.a0, ringH, ring_rows, L.F, 128) ||
            !make_map_mn(&g2.b0, W2, (size_t)L.E * L.F, L.H, 64, nb2))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        g1.o2 = ringH;
        // epilogue tiles leave through shared memory and TMA stores
        // a, b leave in 2 KB blocks by contiguous bulk copies (blk32_offset); h and Y by tensor stores
        if (!make_map_bf16_out(&g1.om2, ringH, ring_rows, L.F) || !make_map_bf16_out(&g2.om0, ringY, ring_rows, L.H))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        g1.tma_store = 1;
        g2.tma_store = 1;
    } else {
        const QwLayout q = qw_layout(cfg);
        const uint8_t *qw = static_cast<const uint8_t *>(align_base(qweights));
        const size_t EF = (size_t)L.E * L.F, EH = (size_t)L.E * L.H;
        const int kb2 = pair_fp8(OP_FWD2) ? 128 : 256;   // K-major B box: half of N per CTA of a pair
        const size_t nw = (size_t)L.E * L.H * L.F / kMxBlock;   // scale bytes of one weight copy
        if (!make_map_u8(&g1.a0, ringXq, ring_rows, L.H, 128) || !make_map_u8(&g1.b0, qw + q.codes[QW_W1T], EF, L.H, 128) ||
            !make_map_u8(&g1.b1, qw + q.codes[QW_W3T], EF, L.H, 128) ||
            !make_map_u8(&g2.a0, ringHq, ring_rows, L.F, 128) || !make_map_u8(&g2.b0, qw + q.codes[QW_W2T], EH, L.F, kb2) ||
            !make_map_atoms(&g1.msa0, ringXs, ring_rows * (L.H / kMxBlock)) ||
            !make_map_atoms(&g1.msb0, qw + q.scales[QW_W1T], nw) || !make_map_atoms(&g1.msb1, qw + q.scales[QW_W3T], nw) ||
            !make_map_atoms(&g2.msa0, ringHs, ring_rows * (L.F / kMxBlock)) ||
            !make_map_atoms(&g2.msb0, qw + q.scales[QW_W2T], nw))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        // Y rows leave through shared memory and TMA stores (64-byte swizzled 32 x 32 boxes)
        if (!make_map_bf16_out(&g2.om0, ringY, ring_rows, L.H)) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        g2.tma_store = 1;
        g1.sfa0 = ringXs; g1.sfb0 = qw + q.scales[QW_W1T]; g1.sfb1 = qw + q.scales[QW_W3T]; g1.kstore = L.H;
        g1.q0 = ringHq; g1.qs0 = ringHs;
        g2.sfa0 = ringHs; g2.sfb0 = qw + q.scales[QW_W2T]; g2.kstore = L.F;
    }
    g1.N = L.F; g1.K = L.H; g1.a_ring = L.keep_x ? 0 : 1;
    g1.x_global = L.keep_x ? 1 : 0;
    g1.o0 = s_a; g1.o1 = s_b;
    g2.N = L.H; g2.K = L.F; g2.a_ring = 1; g2.o_ring = 1;
    g2.o0 = ringY;
    // the dispatch runs inside GEMM1: its gather warps fill the ring minibatch by
    // minibatch and GEMM1 tiles start as soon as their minibatch is complete
    int *ready = at<int>(ws, L.w_ready);
    g1.fused = 1; g1.xsrc = (const bf16 *)x; g1.row_slot = s_row_slot; g1.k = L.k; g1.mb_rows = L.mb_rows;
    const int ready_stride = L.half_rows / kRowPad + 2;
    g1.ready_slots = L.half_rows / kRowPad + 1;
    if (!mx) g1.ringx = ringX;
    else { g1.ringxq = ringXq; g1.ringxs = ringXs; }
    if (cfg->forward_mode == MOE_FORWARD_PERSISTENT && L.T > 0) {
        MegaArgs ma;
        std::memset(&ma, 0, sizeof(ma));
        g1.ready = ready; g1.m = 0; g1.ring_base = 0;
        g2.m = 0; g2.ring_base = 0;
        ma.g1 = g1; ma.g2 = g2;
        int4 *list = at<int4>(ws, L.w_mega_list);
        int *meta = at<int>(ws, L.w_mega_meta), *count = at<int>(ws, L.w_mega_count);
        ma.tiles = list; ma.tile_count = count; ma.meta = meta;
        ma.cnt = at<int>(ws, L.w_mega_cnt); ma.hready = at<int>(ws, L.w_mega_hready);
        ma.slot_row = s_slot_row; ma.w = s_w; ma.out = (bf16 *)out;
        ma.T = L.T; ma.Mb = L.Mb; ma.ready_stride = ready_stride;
        {
            ProfScope ps("forward_tile_list", s);
            st = cuda_check(launch_mega_list(s_offp, L.E, L.nM, L.F, L.H, L.T, L.Mb, list, meta, count, s),
                            "tile list launch");
        }
        if (st != MOE_OK) return st;
        {
            ProfScope ps("forward_persistent", s);
            st = cuda_check(launch_fwd_mega(ma, L.num_sms, s, mx), "persistent forward launch");
        }
        if (st != MOE_OK) return st;
        // the last macrobatch's combine: nothing left to overlap with, so it gets the whole GPU
        CombineArgs ca{};
        ca.Y = ringY; ca.slot_row = s_slot_row; ca.offp = s_offp; ca.w = s_w; ca.out = (bf16 *)out;
        ca.t0 = (L.nM - 1) * L.Mb; ca.t1 = L.T; ca.k = L.k; ca.H = L.H; ca.E = L.E; ca.m = L.nM - 1; ca.ring_base = 0;
        ca.status = at<int>(ws, L.w_status);
        ProfScope ps("combine", s);
        return cuda_check(launch_combine(ca, L.num_sms, s), "combine launch");
    }
    for (int m = 0; m < L.nM; ++m) {
        const int ring_base = (m % L.ring_halves) * L.half_rows;
        g1.ready = ready + (size_t)m * ready_stride;   // zeroed by the schedule scan
        g1.m = m; g1.ring_base = ring_base;
        {
            ProfScope ps("grouped_gemm_fwd1_swiglu", s);
            st = cuda_check(launch_grouped_gemm(OP_FWD1, g1, L.num_sms, s, mx, mx ? pair_fp8(OP_FWD1) : kPairGemm), "GEMM1 launch");
        }
        if (st != MOE_OK) return st;
        g2.m = m; g2.ring_base = ring_base;
        {
            ProfScope ps("grouped_gemm_fwd2", s);
            st = cuda_check(launch_grouped_gemm(OP_FWD2, g2, L.num_sms, s, mx, mx ? pair_fp8(OP_FWD2) : kPairGemm), "GEMM2 launch");
        }
        if (st != MOE_OK) return st;
        CombineArgs ca{};
        ca.Y = ringY; ca.slot_row = s_slot_row; ca.offp = s_offp; ca.w = s_w; ca.out = (bf16 *)out;
        ca.t0 = m * L.Mb; ca.t1 = std::min(L.T, (m + 1) * L.Mb); ca.k = L.k; ca.H = L.H; ca.E = L.E; ca.m = m;
        ca.ring_base = ring_base;
        ca.status = at<int>(ws, L.w_status);
        {
            ProfScope ps("combine", s);
            st = cuda_check(launch_combine(ca, L.num_sms, s), "combine launch");
        }
        if (st != MOE_OK) return st;
    }
    return MOE_OK;
}

moe_status_t moe_backward(const moe_config_t *cfg, const void *dout, const void *x, const void *W_r, const void *W1,
                          const void *W3, const void *W2, const void *qweights, const void *saved, void *dx,
                          float *dW_r, float *dW1, float *dW3, float *dW2, int accumulate, void *workspace,
                          size_t workspace_bytes, moe_stream_t stream) {
    Layout L;
    moe_status_t st = make_layout(cfg, L);
    if (st != MOE_OK) return st;
    const bool mx = cfg->precision == MOE_PRECISION_MXFP8;
    if (cfg->precision == MOE_PRECISION_NVFP4) return fail(MOE_ERR_UNSUPPORTED, "the NVFP4 layer runs the forward only");
    if (mx && !qweights) return fail(MOE_ERR_INVALID_ARG, "MXFP8 backward needs qweights");
    if (!W_r || !W1 || !W3 || !W2 || !saved || !workspace || !dW_r || !dW1 || !dW3 || !dW2 ||
        (L.T > 0 && (!x || !dout || !dx)))
        return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
    if (!fits(workspace, workspace_bytes, L.workspace_bytes)) return fail(MOE_ERR_WORKSPACE, "workspace too small");
    saved = align_base(saved);
    workspace = align_base(workspace);
    const void *ptrs16[] = {x, dout, W_r, W1, W3, W2, dx, dW_r, dW1, dW3, dW2};
    for (const void *p : ptrs16)
        if (p && !aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    void *ws = workspace;

    const int32_t *s_ids = at<int32_t>(saved, L.s_ids);
    const float *s_w = at<float>(saved, L.s_w);
    const float *s_probs = at<float>(saved, L.s_probs);
    const int32_t *s_offp = at<int32_t>(saved, L.s_offp);
    const int32_t *s_slot_row = at<int32_t>(saved, L.s_slot_row);
    const int32_t *s_row_slot = at<int32_t>(saved, L.s_row_slot);
    const bf16 *s_a = at<bf16>(saved, L.s_a);
    const bf16 *s_b = at<bf16>(saved, L.s_b);
    // bf16: the X rows the forward's dispatch kept in saved (no replay); MXFP8 gathers X along
    // the tokens from x instead (the dW1/dW3 operand is quantised along the other axis)
    const bf16 *Xs = L.keep_x ? at<bf16>(saved, L.s_xs) : nullptr;
    bf16 *Gin = at<bf16>(ws, L.w_Gin), *dA = at<bf16>(ws, L.w_da),
         *dB = at<bf16>(ws, L.w_db), *HW = at<bf16>(ws, L.w_hw), *dXs = at<bf16>(ws, L.w_dXs);
    float *dwpart = at<float>(ws, L.w_dwpart), *dlogits = at<float>(ws, L.w_dlogits);
    const size_t rp = L.rows_pad_max;

    // 1. reverse combine (dout rows), all macrobatches (bf16 path; the MXFP8 path gathers
    //    straight into its quantised operands)
    if (L.T > 0 && !mx) {
        DispatchArgs d2{};
        d2.src = (const bf16 *)dout; d2.dst = Gin; d2.row_slot = s_row_slot; d2.offp = s_offp;
        d2.beg = 0; d2.end = L.nM * L.E; d2.dst_row0 = 0; d2.H = L.H; d2.k = L.k;
        d2.nslots = L.R; d2.status = at<int>(ws, L.w_status);
        {
            ProfScope ps("reverse_combine", s);
            st = cuda_check(launch_dispatch(d2, L.rows_pad_max, L.num_sms, s), "reverse combine launch");
        }
        if (st != MOE_OK) return st;
    }
    GemmArgs gb2 = gemm_base(L, ws, s_offp, cfg), gb1 = gemm_base(L, ws, s_offp, cfg);
    GemmArgs gw2 = gemm_base(L, ws, s_offp, cfg), gw13 = gemm_base(L, ws, s_offp, cfg);
    const size_t EF = (size_t)L.E * L.F, EH = (size_t)L.E * L.H;
    if (!mx) {
        const int kb_rows = kPairGemm ? 128 : 256;   // K-major B box: half of N per CTA of a pair
        const int nbw = kPairGemm ? 2 : 4;           // 64-column chunks of dW2's B per CTA
        if (!make_map(&gb2.a0, Gin, rp, L.H, 128) || !make_map(&gb2.b0, W2, EF, L.H, 256) ||
            !make_map(&gb1.a0, dA, rp, L.F, 128) || !make_map(&gb1.a1, dB, rp, L.F, 128) ||
            !make_map(&gb1.b0, W1, EH, L.F, kb_rows) || !make_map(&gb1.b1, W3, EH, L.F, kb_rows) ||
            !make_map_mn(&gw2.a0, HW, rp, L.F, 64, 2) || !make_map_mn(&gw2.b0, Gin, rp, L.H, 64, nbw) ||
            !make_map_mn(&gw13.a0, Xs, rp, L.H, 64, 2) || !make_map_mn(&gw13.b0, dA, rp, L.F, 64, 2) ||
            !make_map_mn(&gw13.b1, dB, rp, L.F, 64, 2))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        if (!make_map_bf16_out(&gb2.om0, dA, rp, L.F) || !make_map_bf16_out(&gb2.om1, dB, rp, L.F) ||
            !make_map_bf16_out(&gb2.om2, HW, rp, L.F) || !make_map_bf16_out(&gb1.om0, dXs, rp, L.H))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        gb2.tma_store = 1;
        gb1.tma_store = 1;
    } else {
        const QwLayout q = qw_layout(cfg);
        const uint8_t *qw = static_cast<const uint8_t *>(align_base(qweights));
        auto u8 = [&](size_t off) { return at<uint8_t>(ws, off); };
        // K-major B boxes: half of N per CTA of a pair (pair_fp8), the whole 256 otherwise
        const int kbb2 = pair_fp8(OP_BWD2) ? 128 : 256, kbb1 = pair_fp8(OP_BWD1) ? 128 : 256;
        const int kbw2 = pair_fp8(OP_WG2) ? 128 : 256;
        const size_t nw = (size_t)L.E * L.H * L.F / kMxBlock;   // scale bytes of one weight copy
        const size_t sh = rp * (L.H / kMxBlock), sf = rp * (L.F / kMxBlock);   // token-side scale bytes
        if (!make_map_u8(&gb2.a0, u8(L.w_Ginq), rp, L.H, 128) || !make_map_u8(&gb2.b0, qw + q.codes[QW_W2Q], EF, L.H, kbb2) ||
            !make_map_u8(&gb1.a0, u8(L.w_daq), rp, L.F, 128) || !make_map_u8(&gb1.a1, u8(L.w_dbq), rp, L.F, 128) ||
            !make_map_u8(&gb1.b0, qw + q.codes[QW_W1Q], EH, L.F, kbb1) ||
            !make_map_u8(&gb1.b1, qw + q.codes[QW_W3Q], EH, L.F, kbb1) ||
            !make_map_u8(&gw2.a0, u8(L.w_hwT), L.F, rp, 128) || !make_map_u8(&gw2.b0, u8(L.w_GinT), L.H, rp, kbw2) ||
            !make_map_u8(&gw13.a0, u8(L.w_XsT), L.H, rp, 128) || !make_map_u8(&gw13.b0, u8(L.w_daT), L.F, rp, 128) ||
            !make_map_u8(&gw13.b1, u8(L.w_dbT), L.F, rp, 128) ||
            !make_map_atoms(&gb2.msa0, u8(L.w_Ginq_s), sh) || !make_map_atoms(&gb2.msb0, qw + q.scales[QW_W2Q], nw) ||
            !make_map_atoms(&gb1.msa0, u8(L.w_daq_s), sf) || !make_map_atoms(&gb1.msa1, u8(L.w_dbq_s), sf) ||
            !make_map_atoms(&gb1.msb0, qw + q.scales[QW_W1Q], nw) || !make_map_atoms(&gb1.msb1, qw + q.scales[QW_W3Q], nw) ||
            !make_map_atoms(&gw2.msa0, u8(L.w_hwT_s), sf) || !make_map_atoms(&gw2.msb0, u8(L.w_GinT_s), sh) ||
            !make_map_atoms(&gw13.msa0, u8(L.w_XsT_s), sh) || !make_map_atoms(&gw13.msb0, u8(L.w_daT_s), sf) ||
            !make_map_atoms(&gw13.msb1, u8(L.w_dbT_s), sf))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        gb2.sfa0 = u8(L.w_Ginq_s); gb2.sfb0 = qw + q.scales[QW_W2Q]; gb2.kstore = L.H;
        gb2.q0 = u8(L.w_daq); gb2.qs0 = u8(L.w_daq_s); gb2.q1 = u8(L.w_dbq); gb2.qs1 = u8(L.w_dbq_s);
        gb2.tq[0] = u8(L.w_daT); gb2.tqs[0] = u8(L.w_daT_s); gb2.tq[1] = u8(L.w_dbT); gb2.tqs[1] = u8(L.w_dbT_s);
        gb2.tq[2] = u8(L.w_hwT); gb2.tqs[2] = u8(L.w_hwT_s); gb2.tR = (int)rp;
        if (!make_map_bf16_out(&gb1.om0, dXs, rp, L.H)) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        gb1.tma_store = 1;   // dX rows through shared memory and TMA stores
        gb1.sfa0 = u8(L.w_daq_s); gb1.sfa1 = u8(L.w_dbq_s);
        gb1.sfb0 = qw + q.scales[QW_W1Q]; gb1.sfb1 = qw + q.scales[QW_W3Q]; gb1.kstore = L.F;
        gw2.sfa0 = u8(L.w_hwT_s); gw2.sfb0 = u8(L.w_GinT_s); gw2.kstore = (int)rp;
        gw13.sfa0 = u8(L.w_XsT_s); gw13.sfb0 = u8(L.w_daT_s); gw13.sfb1 = u8(L.w_dbT_s); gw13.kstore = (int)rp;
    }
    // a (macrobatch, expert) run holds each token of the macrobatch at most once, padded to kRowPad
    const int seg_rows_max = (int)align_up((size_t)std::min(L.Mb, std::max(L.T, 1)), kRowPad);
    // token-axis MXFP8 copies: bf16 [rows][C] -> [C][rows] quantised along rows
    auto transpose_q = [&](const bf16 *src, size_t codes, size_t scales, int C, const char *name,
                           bool gather = false, size_t rcodes = 0, size_t rscales = 0) {
        MxTransposeArgs a{};
        a.src = src; a.codes = at<uint8_t>(ws, codes); a.scales = at<uint8_t>(ws, scales);
        if (rcodes) { a.rcodes = at<uint8_t>(ws, rcodes); a.rscales = at<uint8_t>(ws, rscales); }
        a.R = (int)rp; a.C = C; a.r_limit_ptr = s_offp + L.nM * L.E;
        a.nslots = L.R; a.status = at<int>(ws, L.w_status);
        if (gather) {
            // experts visited in step (see MxTransposeArgs) so each token row is read once from HBM
            a.row_slot = s_row_slot; a.k = L.k;
            a.offp = s_offp; a.ilv_E = L.E; a.ilv_nseg = L.nM * L.E; a.ilv_jb = seg_rows_max / kRowPad;
        }
        ProfScope ps(name, s);
        return cuda_check(launch_mx_transpose(a, 1, s), "token-axis quantise launch");
    };
    if (mx && L.T > 0) {
        // dY rows gathered from dout (reverse combine) quantised along H for the GEMM2 dgrad and,
        // from the same staged tiles, along the token axis for dW2; X along the token axis for
        // dW1/dW3 (activation replay)
        if ((st = transpose_q((const bf16 *)dout, L.w_GinT, L.w_GinT_s, L.H, "quantize_dy", true, L.w_Ginq,
                              L.w_Ginq_s)) != MOE_OK)
            return st;
        if ((st = transpose_q((const bf16 *)x, L.w_XsT, L.w_XsT_s, L.H, "quantize_x_tokens", true)) != MOE_OK)
            return st;
    }
    // 2. GEMM2 dgrad + SwiGLU backward, per macrobatch (global rows)
    gb2.N = L.F; gb2.K = L.H;
    gb2.in0 = s_a; gb2.in1 = s_b; gb2.o0 = dA; gb2.o1 = dB; gb2.o2 = HW; gb2.of0 = dwpart;
    gb2.row_slot = s_row_slot; gb2.wslot = s_w;
    gb1.N = L.H; gb1.K = 2 * L.F; gb1.o0 = dXs;
    // With several macrobatches the dgrads still run as one launch each: their operands and
    // outputs are full size, so the M tiles of every (macrobatch, expert) run come from a
    // device-built list in expert-major order, and the CTAs running at one time share one
    // expert's weights (read from HBM about once per dgrad instead of once per macrobatch).
    const int dgrad_launches = L.nM > 1 ? 1 : L.nM;
    if (L.nM > 1 && L.T > 0) {
        int4 *l128 = at<int4>(ws, L.w_tiles128), *l256 = at<int4>(ws, L.w_tiles256);
        int *cnt = at<int>(ws, L.w_tile_counts);
        {
            ProfScope ps("tile_lists", s);
            st = cuda_check(launch_tile_lists(s_offp, L.E, L.nM, l128, l256, cnt, s), "tile list launch");
        }
        if (st != MOE_OK) return st;
        // CTA pairs take 256-row tiles, 1-CTA kernels 128-row ones (the GEMM2 dgrad runs 1-CTA
        // tiles in bf16 whatever kPairGemm says)
        const bool pair2 = mx && pair_fp8(OP_BWD2), pair1 = mx ? pair_fp8(OP_BWD1) : kPairGemm;
        gb2.tiles = pair2 ? l256 : l128;
        gb2.tile_count = pair2 ? cnt + 1 : cnt;
        gb1.tiles = pair1 ? l256 : l128;
        gb1.tile_count = pair1 ? cnt + 1 : cnt;
    }
    if (L.T > 0) {
        for (int m = 0; m < dgrad_launches; ++m) {
            gb2.m = m;
            {
                ProfScope ps("grouped_gemm_bwd2_swiglu", s);
                st = cuda_check(launch_grouped_gemm(OP_BWD2, gb2, L.num_sms, s, mx, mx ? pair_fp8(OP_BWD2) : kPairGemm), "GEMM2 dgrad launch");
            }
            if (st != MOE_OK) return st;
        }
        for (int m = 0; m < dgrad_launches; ++m) {
            gb1.m = m;
            {
                ProfScope ps("grouped_gemm_bwd1", s);
                st = cuda_check(launch_grouped_gemm(OP_BWD1, gb1, L.num_sms, s, mx, mx ? pair_fp8(OP_BWD1) : kPairGemm), "GEMM1 dgrad launch");
            }
            if (st != MOE_OK) return st;
        }
    }
    // 3. router backward, reverse dispatch, router weight gradient
    RouterBwdArgs rb{};
    rb.dw_part = dwpart; rb.nparts = L.F / 128; rb.slot_row = s_slot_row; rb.ids = s_ids; rb.w = s_w;
    rb.probs = s_probs; rb.dlogits = dlogits; rb.T = L.T; rb.k = L.k; rb.E = L.E;
    rb.rows = L.rows_pad_max; rb.status = at<int>(ws, L.w_status);
    RevDispatchArgs rd{};
    rd.dXs = dXs; rd.slot_row = s_slot_row; rd.dlogits = dlogits; rd.Wr = (const bf16 *)W_r; rd.dx = (bf16 *)dx;
    rd.T = L.T; rd.k = L.k; rd.E = L.E; rd.H = L.H;
    rd.rows = L.rows_pad_max; rd.status = at<int>(ws, L.w_status);
    RouterWgradArgs rw{};
    rw.x = (const bf16 *)x; rw.dlogits = dlogits; rw.part = at<float>(ws, L.w_dwr_part); rw.dWr = dW_r;
    rw.T = L.T; rw.H = L.H; rw.E = L.E; rw.splits = L.dwr_splits; rw.accumulate = accumulate;
    {
        ProfScope ps("router_bwd_dlogits", s);
        st = cuda_check(launch_router_bwd_dlogits(rb, s), "router backward launch");
    }
    if (st != MOE_OK) return st;
    {
        ProfScope ps("reverse_dispatch", s);
        st = cuda_check(launch_reverse_dispatch(rd, s), "reverse dispatch launch");
    }
    if (st != MOE_OK) return st;
    {
        ProfScope ps("router_wgrad", s);
        st = cuda_check(launch_router_wgrad(rw, s), "router weight gradient launch");
    }
    if (st != MOE_OK) return st;
    // 4. weight gradients (contraction over each expert's rows, all macrobatches)
    gw2.Mw = L.F; gw2.N = L.H; gw2.of0 = dW2; gw2.accumulate = accumulate;
    if (kPairGemm && !mx && !accumulate) {
        // weight-gradient tiles leave through shared memory and TMA stores
        if (!make_map_f32_out(&gw2.om0, dW2, EF, L.H) || !make_map_f32_out(&gw13.om0, dW1, EH, L.F) ||
            !make_map_f32_out(&gw13.om1, dW3, EH, L.F))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        gw2.tma_store = 1;
        gw13.tma_store = 1;
    }
    {
        ProfScope ps("grouped_gemm_wgrad2", s);
        st = cuda_check(launch_grouped_gemm(OP_WG2, gw2, L.num_sms, s, mx, mx ? pair_fp8(OP_WG2) : kPairGemm), "dW2 launch");
    }
    if (st != MOE_OK) return st;
    gw13.Mw = L.H; gw13.N = L.F; gw13.of0 = dW1; gw13.of1 = dW3; gw13.accumulate = accumulate;
    {
        ProfScope ps("grouped_gemm_wgrad13", s);
        st = cuda_check(launch_grouped_gemm(OP_WG13, gw13, L.num_sms, s, mx, mx ? pair_fp8(OP_WG13) : kPairGemm), "dW1/dW3 launch");
    }
    return st;
}

}  // extern "C"
