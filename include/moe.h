/*
 * moe.h - C ABI of a single-GPU Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * One MoE layer, forward and backward, over one GPU's tokens:
 *   router (softmax over E experts, top-k, ties to the lower expert index,
 *   weights renormalised over the k chosen) -> schedule (per-expert counts,
 *   exclusive offsets, stable expert-sorted permutation) -> pull dispatch
 *   (gather of token rows into expert-grouped rows, optionally quantised to
 *   MXFP8 inside the gather) -> expert FFN y = W2 (silu(x W1) * (x W3)) as
 *   grouped GEMMs -> combine (top-k weighted sum in fixed slot order), and the
 *   mirrored backward.
 *
 * The stages are the ones the Mixture-of-Kittens articles name:
 *   "O MoK do Cursor alcanca aumento de desempenho de 2,37x no NVIDIA GB300
 *   NVL72" (kucoin.com), section 01 (count tokens per expert, decide where they
 *   go, group each expert's rows for the grouped GEMM), section 02 (pull
 *   dispatch and push combine, reverse-combine and reverse-dispatch in the
 *   backward, minibatches of at least two SM waves, a fixed-size ring token
 *   buffer advanced by GPU-side state, MXFP8 quantisation fused into dispatch,
 *   grouped GEMM and SwiGLU) and section 03 (Schedule, Dispatch, Expert FFN,
 *   Combine, final weighted fusion); "Cursor abre codigo do Mixture-of-Kittens"
 *   (noticiai.com.br), "O que e" (one deterministic kernel) and "As tres
 *   decisoes de design" (no token dropping; macrobatch interleave).
 * The pages give no formulas; the router and SwiGLU forms above are the plain
 * reading of a softmax top-k SwiGLU MoE.
 *
 * Conventions for every call below
 *   - All tensor arguments are DEVICE pointers owned by the caller. The library
 *     never allocates or frees device memory; scratch comes from the caller's
 *     workspace, and the forward->backward context from the caller's `saved`
 *     buffer, both sized by the query functions.
 *   - Layouts are dense row-major: x, out, dout, dx [T,H] bf16; W_r [H,E] bf16;
 *     bias [E] fp32; W1, W3 [E,H,F] bf16; W2 [E,F,H] bf16; topk ids [T,k]
 *     int32; topk weights [T,k] fp32; weight gradients fp32 in the shape of
 *     their weight. bf16 is IEEE bfloat16 stored as 16-bit words.
 *   - Every call is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without synchronising the host. Inputs are never
 *     written.
 *   - Host-detected errors (null pointer, unsupported size, workspace too
 *     small, misalignment) return a non-zero status and launch nothing.
 *     A failed kernel launch returns MOE_ERR_CUDA. Errors detected on the
 *     device (a bounded wait that ran out, an index check that failed) are
 *     written to a status word inside the workspace; moe_query_status reads it.
 *   - Tensor pointers must be 16-byte aligned. The workspace and saved
 *     buffers may start anywhere: the library uses them from the next
 *     1024-byte boundary on, and the size queries include that slack.
 *   - Calls sharing one workspace must not overlap in time (same stream, or
 *     ordered by events).
 *   - Thread safety: calls from several host threads are safe when they use
 *     distinct workspaces. State shared across calls: a thread-local error
 *     string and per-device caches of kernel occupancy queries (atomics).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 3

typedef struct CUstream_st *moe_stream_t;   /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,   /* shape outside the supported envelope */
    MOE_ERR_WORKSPACE = 3,     /* workspace or saved buffer too small */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    MOE_ERR_TIMEOUT = 5,       /* a bounded device wait ran out (device status) */
    MOE_ERR_INTERNAL = 6       /* a device-side consistency check failed */
} moe_status_t;

typedef enum {
    MOE_PRECISION_BF16 = 0,    /* bf16 operands, fp32 accumulation */
    MOE_PRECISION_MXFP8 = 1,   /* e4m3 operands, one e8m0 scale per 32 along K */
    MOE_PRECISION_NVFP4 = 2    /* NVFP4 expert weights (e2m1, one e4m3 scale per 16 along K,
                                  a power-of-two fp32 scale per expert matrix), bf16
                                  activations: the forward of at most 128 tokens in one
                                  macrobatch (the decode kernel); moe_backward and larger
                                  batches return MOE_ERR_UNSUPPORTED */
} moe_precision_t;

/* Layer shape and run options. Zero-initialise, then set the shape.
 *   T tokens, H hidden size, F expert FFN width, E experts, k experts per token.
 *   Supported: 1 <= k <= E <= 64, H and F multiples of 256, T >= 0.
 *   minibatch_rows: routed rows per grouped-GEMM step of the ring pipeline;
 *     0 = smallest multiple of 128 giving at least two full waves of GEMM1
 *     tiles on the device's SMs (article section 02: "at least two full SM
 *     waves per expert grouped GEMM").
 *   ring_bytes: size of the token ring: the dispatched token rows of the
 *     macrobatch in flight, padded to whole 128-row tiles per expert, in the
 *     layer's compute format (MXFP8: E4M3 along H plus scales, H + H/32 bytes a
 *     row, in the workspace; bf16: 2H bytes a row, written straight into the
 *     saved context, which the backward reads). The macrobatch's FFN hidden rows
 *     and expert outputs take workspace buffers of the same row count (article
 *     section 02: a fixed-size ring of tokens, each slot reused once the experts
 *     and the combine are done with it). 0 = large enough for all routed rows,
 *     i.e. one macrobatch.
 *   macrobatch_tokens: tokens per macrobatch; 0 = derived from ring_bytes.
 *   timeout_ms: budget of every device-side wait; 0 = 2000 ms.
 *   num_sms: SM count used for planning; 0 = query the current device.
 *   fault_mask: 0 in normal use; bits inject a failure from the host for tests
 *     of failure detection (no GPU fault, trap or unbounded wait):
 *     MOE_FAULT_GEMM1_READY: moe_forward sets GEMM1's first minibatch ready
 *     counter so that it never reaches its target; GEMM1's bounded wait runs
 *     out, the status word reports MOE_ERR_TIMEOUT, every other wait sees the
 *     status and returns, and the outputs of that call are undefined.
 *   forward_mode: MOE_FORWARD_PERSISTENT (0, default): after the router and the
 *     schedule, one persistent launch runs the dispatch, both expert GEMMs and
 *     the combine of every macrobatch, handing work on through device counters;
 *     MOE_FORWARD_PER_STAGE: one launch per stage and macrobatch. Both give the
 *     same bytes. (A bf16 forward of at most 128 tokens in one macrobatch runs
 *     the decode kernel in either mode.) */
typedef struct {
    int T, H, F, E, k;
    int precision;
    int minibatch_rows;
    int macrobatch_tokens;
    size_t ring_bytes;
    unsigned timeout_ms;
    int num_sms;
    unsigned fault_mask;
    int forward_mode;
} moe_config_t;

#define MOE_FORWARD_PERSISTENT 0
#define MOE_FORWARD_PER_STAGE 1

#define MOE_FAULT_GEMM1_READY 1u

/* Derived execution plan (host-only; no device access when cfg->num_sms > 0). */
typedef struct {
    int num_sms;             /* SMs the plan was made for */
    int minibatch_rows;      /* rows per grouped-GEMM step */
    int macrobatch_tokens;   /* tokens per macrobatch */
    int num_macrobatches;    /* ceil(T / macrobatch_tokens) */
    int rows_padded_max;     /* upper bound of padded expert-sorted rows */
    int ring_rows;           /* rows held by the ring (all halves) */
    size_t ring_bytes;       /* bytes the ring occupies in the workspace */
    size_t workspace_bytes;  /* = moe_workspace_size(cfg) */
    size_t saved_bytes;      /* = moe_saved_size(cfg) */
    size_t qweights_bytes;   /* = moe_qweights_size(cfg) */
} moe_plan_t;

/* Library ABI version (MOE_ABI_VERSION of the build). */
int moe_abi_version(void);

/* Fills *plan for cfg. Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a
 * shape the library does not run. */
moe_status_t moe_plan(const moe_config_t *cfg, moe_plan_t *plan);

/* Bytes of scratch memory needed by moe_schedule / moe_forward / moe_backward
 * (0 when cfg is invalid). Content is not preserved between calls. */
size_t moe_workspace_size(const moe_config_t *cfg);

/* Bytes of the forward->backward context written by moe_forward and read by
 * moe_backward (router ids/weights/probabilities, schedule maps, the bf16
 * FFN pre-activations a = x W1 and b = x W3 of every routed row; for bf16
 * configs also the expert-sorted x rows the dispatch gathered, which GEMM1 and
 * then the backward's dW1/dW3 read, so the backward never gathers them again). */
size_t moe_saved_size(const moe_config_t *cfg);

/* Bytes of the MXFP8 or NVFP4 weight copies made by moe_quantize_weights (0 for bf16). */
size_t moe_qweights_size(const moe_config_t *cfg);

/* Schedule only (article section 01: count, place, group).
 * topk_ids [T,k] int32 in [0,E). With macrobatch m = t / Mb (Mb = the plan's
 * macrobatch_tokens), the routed slots s = t*k + j are stably sorted by the key
 * (m, expert):
 *   counts [nM*E]          rows of (m, e)
 *   offsets [nM*(E+1)]     absolute sorted position where (m, e) starts; the
 *                          last entry of each macrobatch is where it ends
 *   sorted_to_slot [T*k]   slot at each sorted position
 *   slot_to_sorted [T*k]   inverse permutation
 * All outputs are bit-exact and deterministic. Ids outside [0,E) make the
 * device status MOE_ERR_INTERNAL (their slots are left out). */
moe_status_t moe_schedule(const moe_config_t *cfg, const int32_t *topk_ids,
                          int32_t *counts, int32_t *offsets,
                          int32_t *sorted_to_slot, int32_t *slot_to_sorted,
                          void *workspace, size_t workspace_bytes,
                          moe_stream_t stream);

/* moe_schedule for callers that cannot allocate device memory (a framework
 * callback whose pool owns all device memory, a deployment that forbids
 * allocation after start-up). Same arguments and results as moe_schedule,
 * minus the workspace: the scratch lives in a 1 MiB device array of the
 * library itself. The pages have no counterpart of this entry point.
 *   - Shapes whose schedule scratch (two histograms of (chunk, expert) counts
 *     plus the padded offsets, 256 routed slots per chunk) exceeds the array
 *     return MOE_ERR_UNSUPPORTED.
 *   - The first call on a device loads the array's module there (reserving
 *     its 1 MiB until the process exits; in a pool that owns every free byte
 *     this can fail with MOE_ERR_CUDA) and looks up the array's device address
 *     with that device current. Make that first call at start-up, before any
 *     stream capture.
 *   - The address is cached per device number for the life of the process:
 *     do not call cudaDeviceReset, or make another context current on the
 *     device, between calls.
 *   - All calls on a device share the array; calls that overlap on the GPU
 *     race and give undefined results. Each call clears what must start at 0.
 *   - Device-side id checks are not reported: pass ids in [0,E).
 *   - Calls no cudaMalloc, cudaFree or other allocating routine. */
moe_status_t moe_schedule_static(const moe_config_t *cfg, const int32_t *topk_ids,
                                 int32_t *counts, int32_t *offsets,
                                 int32_t *sorted_to_slot, int32_t *slot_to_sorted,
                                 moe_stream_t stream);

/* Quantised copies of the bf16 master weights, run once per weight update:
 * MXFP8: one copy per forward and backward GEMM, each along its contraction
 * axis; NVFP4: W1, W3 along H and W2 along F, in the tiles the decode kernel
 * streams. Returns MOE_ERR_UNSUPPORTED for a bf16 config. */
moe_status_t moe_quantize_weights(const moe_config_t *cfg, const void *W1,
                                  const void *W3, const void *W2,
                                  void *qweights, size_t qweights_bytes,
                                  moe_stream_t stream);

/* Forward (article section 03: Schedule, Dispatch, Expert FFN, Combine and the
 * final weighted fusion).
 *   x [T,H] bf16, W_r [H,E] bf16, bias [E] fp32 or NULL, W1/W3 [E,H,F] bf16,
 *   W2 [E,F,H] bf16, qweights: moe_quantize_weights output (MXFP8) or NULL.
 *   out [T,H] bf16: out[t] = sum_j w[t,j] * y_j, summed in fp32 in slot order j
 *     and rounded once; bit-reproducible run to run.
 *   topk_ids [T,k] int32, topk_w [T,k] fp32: the router's choice (descending
 *     probability) and renormalised weights.
 *   saved: moe_saved_size bytes, consumed by moe_backward. */
moe_status_t moe_forward(const moe_config_t *cfg, const void *x, const void *W_r,
                         const float *bias, const void *W1, const void *W3,
                         const void *W2, const void *qweights, void *out,
                         int32_t *topk_ids, float *topk_w, void *saved,
                         size_t saved_bytes, void *workspace,
                         size_t workspace_bytes, moe_stream_t stream);

/* Backward of sum(dout * out) with the top-k choice held fixed (article
 * section 02: pull reverse-combine and push reverse-dispatch).
 *   dout [T,H] bf16; x, W_r, W1, W3, W2, qweights and saved as given to the
 *   matching moe_forward.
 *   dx [T,H] bf16 (overwritten); dW_r [H,E], dW1/dW3 [E,H,F], dW2 [E,F,H] fp32:
 *   overwritten when accumulate == 0, added to when accumulate != 0. */
moe_status_t moe_backward(const moe_config_t *cfg, const void *dout,
                          const void *x, const void *W_r, const void *W1,
                          const void *W3, const void *W2, const void *qweights,
                          const void *saved, void *dx, float *dW_r, float *dW1,
                          float *dW3, float *dW2, int accumulate,
                          void *workspace, size_t workspace_bytes,
                          moe_stream_t stream);

/* Synchronises `stream`, returns the device status word of `workspace`
 * (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_INTERNAL) and clears it. */
moe_status_t moe_query_status(void *workspace, moe_stream_t stream);

/* Clears the device status word (enqueued on stream, no host sync). Call once
 * on a fresh workspace before its first use. */
moe_status_t moe_reset_status(void *workspace, moe_stream_t stream);

/* Intermediate buffers of the layer that moe_buffer_location can locate (a test
 * and debugging aid: the parity tests read them to compare the quantised
 * operands byte for byte with a reference quantiser). Rows are padded
 * expert-sorted rows: every (macrobatch, expert) run starts at a multiple of
 * 128 and is padded with zero rows; MOE_BUF_ROW_SLOT gives each row's routed
 * slot t*k + j (-1 = padding), MOE_BUF_PADDED_OFFSETS the run starts.
 * "_SCALES" buffers hold E8M0 scale bytes in 512-byte atoms (128 rows x 128
 * elements of the contraction axis; atom (r/128, k/128) in row-major order,
 * byte (r%32)*16 + ((r/32)%4)*4 + (k/32)%4 inside it).
 * Every kernel that follows ROW_SLOT or SLOT_ROW to a row checks the index
 * against its range (a slot in [-1, T*k), a row inside the padded rows, in the
 * combine inside the macrobatch's rows); an index outside it sets the device
 * status to MOE_ERR_INTERNAL and the access is skipped, so a corrupted saved
 * context is reported by moe_query_status instead of touching memory out of
 * bounds.
 *   saved buffer (written by moe_forward):
 *     PADDED_OFFSETS int32 [nM*E+1]; ROW_SLOT int32 [rows]; SLOT_ROW int32 [T*k]
 *     (each routed slot's padded row); A, B bf16 [rows][F]
 *     in 32 x 32 blocks of 2 KB (block (r/32, c/32) row-major, element (r, c) at
 *     ((c%32)/8*32 + r%32)*8 + c%8 inside it).
 *   workspace, valid after moe_forward until the next call on the workspace
 *   (the last macrobatch's rows; ring row = padded row - first padded row of
 *   that macrobatch):
 *     RING_X: dispatched x rows, E4M3 along H [ring_rows][H] (+ _SCALES); bf16:
 *       in saved, every macrobatch's rows at their padded rows [rows][H];
 *     RING_H: h rows of the macrobatch, bf16 [ring_rows][F] or E4M3 along F
 *       (+ _SCALES).
 *   workspace, valid after moe_backward until the next call on the workspace:
 *     DA, DB, HW: bf16 [rows][F] (dh.b.sigmoid'(a) terms, w.h), bf16 configurations
 *     only (MXFP8 quantises them straight into DA/DB/HW_TOKENS);
 *     MXFP8 only: DY_ROWS (dout rows, E4M3 along H), DA_ROWS, DB_ROWS (E4M3
 *     along F), each [rows][K] + _SCALES; X_TOKENS, DY_TOKENS (E4M3 [H][rows]
 *     along the rows) and HW_TOKENS, DA_TOKENS, DB_TOKENS ([F][rows]), + _SCALES. */
typedef enum {
    MOE_BUF_PADDED_OFFSETS = 0, MOE_BUF_ROW_SLOT, MOE_BUF_A, MOE_BUF_B,
    MOE_BUF_RING_X, MOE_BUF_RING_X_SCALES, MOE_BUF_RING_H, MOE_BUF_RING_H_SCALES,
    MOE_BUF_DA, MOE_BUF_DB, MOE_BUF_HW,
    MOE_BUF_DY_ROWS, MOE_BUF_DY_ROWS_SCALES, MOE_BUF_DA_ROWS, MOE_BUF_DA_ROWS_SCALES,
    MOE_BUF_DB_ROWS, MOE_BUF_DB_ROWS_SCALES,
    MOE_BUF_X_TOKENS, MOE_BUF_X_TOKENS_SCALES, MOE_BUF_DY_TOKENS, MOE_BUF_DY_TOKENS_SCALES,
    MOE_BUF_HW_TOKENS, MOE_BUF_HW_TOKENS_SCALES, MOE_BUF_DA_TOKENS, MOE_BUF_DA_TOKENS_SCALES,
    MOE_BUF_DB_TOKENS, MOE_BUF_DB_TOKENS_SCALES,
    MOE_BUF_SLOT_ROW,
    MOE_BUF_COUNT
} moe_buffer_t;

/* Where buffer `which` (a moe_buffer_t) lives: *in_saved = 1 for the saved
 * buffer, 0 for the workspace; *offset = bytes from the 1024-byte boundary at
 * or after the buffer's start (the base the library uses); *bytes = its size.
 * Host-only. MOE_ERR_UNSUPPORTED for a buffer the configuration does not have
 * (the MXFP8-only ones in a bf16 configuration). */
moe_status_t moe_buffer_location(const moe_config_t *cfg, int which, int *in_saved, size_t *offset,
                                 size_t *bytes);

/* Per-kernel timing of this host thread's calls (CUDA events recorded on the
 * launch stream around every kernel the library launches). */
typedef struct {
    char name[32];        /* kernel name, e.g. "grouped_gemm_fwd1" */
    int launches;         /* launches recorded since moe_profile_begin */
    double total_ms;      /* sum of their event-measured durations */
} moe_kernel_time_t;

/* Starts recording (clears earlier records of this thread). */
moe_status_t moe_profile_begin(void);

/* Stops recording, waits for the recorded events, writes up to max_entries
 * aggregated rows (one per kernel name, in first-launch order) and returns how
 * many there are (negative moe_status_t on a CUDA error). */
int moe_profile_end(moe_kernel_time_t *out, int max_entries);

/* Message of the last error returned on this host thread. */
const char *moe_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
