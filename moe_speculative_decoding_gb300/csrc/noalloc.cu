// noalloc.cu -- the per-slot expert operation for callers that cannot allocate device memory.
//
// moe_expert_op_perslot needs a caller-allocated workspace.  Some callers cannot allocate:
// code that runs under a memory manager which owns every device byte (a serving
// framework's caching allocator, a fixed arena budgeted ahead of time), where a raw
// cudaMalloc would bypass its accounting, and code on a latency-critical path, where
// cudaMalloc and cudaFree synchronise the device.  This entry point runs the same
// kernels with the workspace replaced by a small array that lives in the library itself.
#include <mutex>

#include "common.cuh"
#include "expert_args.cuh"

namespace {

// The scratch of moe_expert_op_perslot_noalloc: a workspace (the device error word, then
// the gate/up partial sums of the tensor-core path) for every layer whose workspace fits
// 32 MiB, e.g. d = 4096, f = 14336, top-2 at 16 tokens (22 MB).  Every GPU that loads the
// library holds these bytes until the process exits, and every call of the entry point
// shares them.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static_assert(kNoAllocScratchBytes >= moe::kWorkspaceBytes, "scratch smaller than a workspace");
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device.  In host code the array's name
// only stands in for it, so the address is looked up once per device, with that device
// current, and cached.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status_t moe_expert_op_perslot_noalloc(const moe_layer_t *layer, const void *w_gate,
                                                      const void *w_up, const void *w_down, const void *x,
                                                      const int32_t *ids, const float *gates, int32_t n,
                                                      int32_t accumulate, float *y, int32_t *status_out,
                                                      moe_stream_t s) {
    // every argument is checked before any device work: a rejected call enqueues nothing
    const moe_status_t checked = moe::check_perslot_call(layer, w_gate, w_up, w_down, x, ids, gates, n, y);
    if (checked != MOE_OK) return checked;
    if (status_out != nullptr && (reinterpret_cast<uintptr_t>(status_out) & 3u) != 0) return MOE_ERR_ARG;
    // the per-slot calls launch at most MOE_PERSLOT_LAUNCH_TOKENS tokens at a time
    const int32_t nl = n < MOE_PERSLOT_LAUNCH_TOKENS ? n : MOE_PERSLOT_LAUNCH_TOKENS;
    if (moe_workspace_bytes(layer, nl) > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
    void *ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
    // the previous call's error word must not leak into this one.  Everything else in the
    // scratch carries the ticket of the call that wrote it (the epoch word after the error word
    // counts the calls), so a later call, of any layer shape, never takes it for its own: it
    // needs no clearing, and the array starts zeroed when the library loads.
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    const moe_status_t r = moe_expert_op_perslot(layer, w_gate, w_up, w_down, x, ids, gates, n, accumulate, y, ws,
                                                 kNoAllocScratchBytes, s);
    if (r != MOE_OK) return r;
    if (status_out != nullptr &&
        cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
