// probe.cu -- a read-only streaming probe of the memory the expert kernel streams from.
//
// Measurement only, not part of the method: it gives the read bandwidth a persistent grid of
// TMA bulk copies reaches on this GPU, beside the copy bandwidth (read + write) that the
// roofline takes as its peak.  Each CTA (one per SM) streams its contiguous share of the
// buffer through a ring of shared-memory slots with 1-D bulk copies (cp.async.bulk), one
// elected thread issuing and waiting; the bytes are not otherwise used.  Every wait is
// bounded, as in the expert kernel.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kProbeSlots = 6;
constexpr uint32_t kProbeChunk = 32768;   // bytes per copy

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}

__global__ void __launch_bounds__(32) read_probe_kernel(const uint8_t *buf, long long chunks, int32_t *err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 127u) & ~127u;
    const uint32_t bars = base + kProbeSlots * kProbeChunk;
    __shared__ int32_t abort_word;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kProbeSlots; ++s) mbar_init(bars + 8u * s, 1);
        abort_word = 0;
        fence_mbar_init();
    }
    __syncwarp();
    const long long lo = blockIdx.x * chunks / gridDim.x, hi = (blockIdx.x + 1) * chunks / gridDim.x;
    if (threadIdx.x == 0) {
        volatile int32_t *abort_flag = &abort_word;
        for (long long j = lo; j < hi; ++j) {
            const uint32_t k = static_cast<uint32_t>(j - lo), s = k % kProbeSlots;
            // the slot's previous copy has landed before it is reused
            if (k >= kProbeSlots && !mbar_wait(bars + 8u * s, ((k / kProbeSlots) - 1) & 1u, abort_flag, err)) break;
            mbar_arrive_expect_tx(bars + 8u * s, kProbeChunk);
            bulk_load(base + s * kProbeChunk, buf + j * static_cast<long long>(kProbeChunk), kProbeChunk, bars + 8u * s);
        }
        // the last copies land before the CTA exits
        const long long n = hi - lo;
        for (long long k = n > kProbeSlots ? n - kProbeSlots : 0; k < n; ++k)
            mbar_wait_drain(bars + 8u * (k % kProbeSlots), (k / kProbeSlots) & 1u, 400000000ll);
    }
    __syncwarp();
}

}  // namespace

cudaError_t launch_read_probe(const void *buf, size_t bytes, int32_t *err, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = kProbeSlots * kProbeChunk + 8 * kProbeSlots + 128;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(read_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long long chunks = static_cast<long long>(bytes / kProbeChunk);
    read_probe_kernel<<<sms, 32, smem, s>>>(static_cast<const uint8_t *>(buf), chunks, err);
    return cudaGetLastError();
}

}  // namespace moe
