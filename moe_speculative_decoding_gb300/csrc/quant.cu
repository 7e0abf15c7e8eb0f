// quant.cu -- per-row quantization to OCP FP8 E4M3, the operand format of the FP8 expert
// kernels: one fp32 scale per row, amax / 448 (1 for an all-zero row), codes rounded to
// nearest (ties to even) after an IEEE fp32 division, saturating at +-448.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;

__global__ void __launch_bounds__(kQThreads) quantize_rows_kernel(const void *src, int dtype, int rows, int cols,
                                                                  uint8_t *q, float *scale) {
    __shared__ float red[kQThreads / 32];
    pdl_wait();
    pdl_trigger();
    const float *const s32 = static_cast<const float *>(src);
    const __nv_bfloat16 *const s16 = static_cast<const __nv_bfloat16 *>(src);
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const size_t base = static_cast<size_t>(r) * cols;
        auto val = [&](int c) { return dtype == MOE_F32 ? s32[base + c] : __bfloat162float(s16[base + c]); };
        float mx = 0.0f;
        for (int c = threadIdx.x; c < cols; c += kQThreads) mx = fmaxf(mx, fabsf(val(c)));
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
        __syncthreads();
        float amax = 0.0f;
        for (int w = 0; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
        __syncthreads();   // red is rewritten for the next row
        const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        if (threadIdx.x == 0) scale[r] = sc;
        for (int c = threadIdx.x; c < cols; c += kQThreads) q[base + c] = f32_to_e4m3(val(c) / sc);
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const void *src, int dtype, int rows, int cols, uint8_t *q, float *scale,
                                 cudaStream_t s, bool pdl) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows < 65535 ? rows : 65535));
    cfg.blockDim = dim3(kQThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_rows_kernel, src, dtype, rows, cols, q, scale);
}

}  // namespace moe
