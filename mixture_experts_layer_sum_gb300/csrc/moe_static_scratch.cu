// moe_schedule_static: the schedule for callers that cannot allocate device
// memory.
//
// Some programs cannot hand this library a workspace: code that runs inside a
// framework callback whose memory pool owns every device byte, real-time or
// certified deployments that forbid allocation after start-up, and drivers of
// pre-planned memory where every buffer is fixed ahead of time. For them this
// entry point keeps its scratch (schedule chunk histograms, chunk bases,
// padded offsets and a status word) in one file-scope device array. The array
// belongs to this file's CUDA module; with lazy module loading (the default) the
// module, and with it the array's 1 MiB, is loaded on a device by the first
// call made there, and stays until the process exits. A pool that already owns
// every free byte can make that first call fail, so make it at start-up. The
// entry point computes exactly what moe_schedule computes, with the same kernels.
//
// Limits and rules:
//   - Capacity: kStaticScratchInts 32-bit words (1 MiB). A configuration whose
//     scratch does not fit is rejected with MOE_ERR_UNSUPPORTED.
//   - The array's host-side name is only a stand-in for the device object: its
//     device address is looked up once per device with cudaGetSymbolAddress
//     (with that device current) on the first call made on that device, so
//     make that first call before any stream capture begins.
//   - The looked-up addresses are cached per device number for the life of the
//     process. A cudaDeviceReset, or a different context made current on the
//     device, invalidates them: do neither between calls.
//   - Every call on a device uses the same array and leaves its contents
//     behind; each call clears the part that must start at zero. Calls whose
//     executions overlap on the GPU (different streams without ordering) race
//     on the array and give undefined results.
//   - No cudaMalloc, cudaFree or allocating library routine is called.
#include <mutex>
#include <string>

#include "../../include/moe.h"
#include "route_kernels.cuh"

namespace moe {
void set_last_error(const char *msg);
}

namespace {

constexpr size_t kStaticScratchInts = size_t(1) << 18;   // 1 MiB
constexpr int kMaxDevices = 64;
constexpr int kStatusInts = 64;

__device__ __align__(256) int g_static_scratch[kStaticScratchInts];

std::mutex g_mu;
int *g_dev_ptr[kMaxDevices] = {};
thread_local std::string g_last_msg;

moe_status_t fail(moe_status_t st, const char *msg) {
    moe::set_last_error(msg);
    return st;
}

}  // namespace

extern "C" moe_status_t moe_schedule_static(const moe_config_t *cfg, const int32_t *topk_ids, int32_t *counts,
                                            int32_t *offsets, int32_t *sorted_to_slot, int32_t *slot_to_sorted,
                                            moe_stream_t stream) {
    moe_plan_t plan;
    moe_status_t st = moe_plan(cfg, &plan);
    if (st != MOE_OK) return st;
    const int T = cfg->T, k = cfg->k, E = cfg->E;
    const long long R = (long long)T * k;
    if (!counts || !offsets || (R > 0 && (!topk_ids || !sorted_to_slot || !slot_to_sorted)))
        return fail(MOE_ERR_INVALID_ARG, "null pointer argument");
    const int Mb = plan.macrobatch_tokens, nM = plan.num_macrobatches;
    const int chunks_per_mb = std::max(1, moe::ceil_div(std::min(Mb, std::max(T, 1)) * k, moe::kSchedChunk));
    const int nchunks = T > 0 ? nM * chunks_per_mb : 0;
    const size_t need = kStatusInts + 2 * (size_t)std::max(nchunks, 1) * E + ((size_t)nM * E + 1);
    if (need > kStaticScratchInts)
        return fail(MOE_ERR_UNSUPPORTED,
                    "moe_schedule_static: the schedule scratch of this shape exceeds the 1 MiB static array");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(MOE_ERR_CUDA, "moe_schedule_static: no usable current device");
    int *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_dev_ptr[dev]) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
            if (e != cudaSuccess || !p) {
                // the failure (often an out-of-memory error while the module loads) stays
                // recorded as the runtime's last error; clear it so that it is not reported
                // again by the next launch check of this or another entry point
                cudaGetLastError();
                g_last_msg = std::string("moe_schedule_static: looking up the static scratch array failed: ") +
                             cudaGetErrorString(e);
                return fail(MOE_ERR_CUDA, g_last_msg.c_str());
            }
            g_dev_ptr[dev] = static_cast<int *>(p);
        }
        base = g_dev_ptr[dev];
    }
    cudaStream_t s = (cudaStream_t)stream;
    // the status word and its padding must start at zero on every call
    if (cudaMemsetAsync(base, 0, kStatusInts * sizeof(int), s) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "moe_schedule_static: clearing the status word failed");

    moe::SchedArgs a{};
    a.ids = topk_ids;
    a.T = T; a.k = k; a.E = E; a.Mb = Mb; a.nM = nM;
    a.chunks_per_mb = chunks_per_mb; a.nchunks = nchunks;
    a.status = base;
    a.chunk_counts = base + kStatusInts;
    a.chunk_base = a.chunk_counts + (size_t)std::max(nchunks, 1) * E;
    a.offp = a.chunk_base + (size_t)std::max(nchunks, 1) * E;
    a.counts = counts; a.offsets = offsets;
    a.sorted_to_slot = sorted_to_slot; a.slot_to_sorted = slot_to_sorted;
    a.slot_row = nullptr; a.row_slot = nullptr;
    if (moe::launch_schedule(a, s) != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_schedule_static: launch failed");
    return MOE_OK;
}
