// expert_simt.cu -- generic CUDA-core kernel of the expert operation (fp32 or bf16).
//
// "Speculative Decoding for Mixture-of-Experts Models" (Lan), §1: the expert operation
// is the gate, up and down projections of each token of a pass with the weights of its
// selected experts; the per-slot form reads one expert per slot, the deduplicating form
// groups the pass's tokens by expert and reads each distinct expert once.
//
// One CTA per work item (group, tile of 64 rows of f).  A group is one slot (per-slot
// form) or one distinct expert with all of its tokens (deduplicating form).  The CTA
// computes h = silu(W_gate x) * (W_up x) for its 64 rows and every token of the group
// (warp-shuffle reductions), then the partial down projection W_down[:, rows] h over all
// d outputs and adds gate * partial into y with atomics, so the combine is fused and
// the f-split partial sums meet in y.  This kernel serves fp32 layers and is a second,
// independent GPU path for bf16 layers; the tensor-core kernel is the bf16 default.
#include "common.cuh"
#include "expert_args.cuh"

namespace moe {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int kWin = 16;   // tokens per window of accumulators

template <typename T>
__device__ __forceinline__ float ld_val(const T *p);
template <>
__device__ __forceinline__ float ld_val<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_val<__nv_bfloat16_raw>(const __nv_bfloat16_raw *p) {
    const unsigned short bits = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __uint_as_float(static_cast<uint32_t>(bits) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

template <typename WT, typename XT>
__global__ void __launch_bounds__(kSimtThreads) expert_simt_kernel(ExpertArgs a) {
    __shared__ float s_h[kMaxPassTokens][kFTile];
    __shared__ float s_gate[kMaxPassTokens];
    __shared__ int s_expert;
    __shared__ uint64_t s_mask;

    pdl_wait();
    const int tile = blockIdx.x;
    const int g = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        int e = -1;
        uint64_t mask = 0;
        for (int t = 0; t < kMaxPassTokens; ++t) s_gate[t] = 0.0f;
        if (a.mode == kModePerSlot) {
            e = a.ids[g];
            const int t = g / a.m;
            s_gate[t] = a.gates[g];
            mask = 1ull << t;
        } else if (g < a.num_distinct[0]) {   // g < min(N, n*m) by the launch shape
            e = a.expert_list[g];
            const int S = a.n * a.m;   // offsets are clamped to the slot buffer
            const int p0 = max(0, a.offsets[g]), p1 = min(S, a.offsets[g + 1]);
            for (int p = p0; p < p1; ++p) {
                const int slot = a.slot_order[p];
                const int t = slot / a.m;
                if (slot >= 0 && t < a.n) {
                    s_gate[t] += a.gates[slot];
                    mask |= 1ull << t;
                }
            }
        } else {
            e = -2;   // beyond the distinct experts of this pass: nothing to do
        }
        if (e != -2 && (e < 0 || e >= a.N)) {
            record_error(a.err, MOE_ERR_BAD_ID);
            e = -2;
        }
        s_expert = e;
        s_mask = mask;
    }
    __syncthreads();
    const int e = s_expert;
    const uint64_t mask = s_mask;
    if (e < 0) {
        pdl_trigger();
        return;
    }
    const int d = a.d, f = a.f;
    const int i0 = tile * kFTile;
    const WT *wg = static_cast<const WT *>(a.w_gate) + (static_cast<size_t>(e) * f + i0) * d;
    const WT *wu = static_cast<const WT *>(a.w_up) + (static_cast<size_t>(e) * f + i0) * d;
    const WT *wd = static_cast<const WT *>(a.w_down) + static_cast<size_t>(e) * d * f + i0;
    const XT *x = static_cast<const XT *>(a.x);

    // gate/up rows of this tile: warp w takes rows w, w + 8, ...; the group's tokens in
    // windows of 16 (a window's rows are read again from cache, not from memory)
    for (int r = warp; r < kFTile; r += kSimtWarps) {
        for (int t0 = 0; t0 < kMaxPassTokens; t0 += kWin) {
            const uint32_t wm = static_cast<uint32_t>(mask >> t0) & 0xFFFFu;
            if (wm == 0u) continue;
            float gacc[kWin], uacc[kWin];
#pragma unroll
            for (int t = 0; t < kWin; ++t) { gacc[t] = 0.0f; uacc[t] = 0.0f; }
            for (int k = lane; k < d; k += 32) {
                const float wgv = ld_val<WT>(wg + static_cast<size_t>(r) * d + k);
                const float wuv = ld_val<WT>(wu + static_cast<size_t>(r) * d + k);
#pragma unroll
                for (int t = 0; t < kWin; ++t) {
                    if ((wm >> t) & 1u) {
                        const float xv = ld_val<XT>(x + static_cast<size_t>(t0 + t) * d + k);
                        gacc[t] = fmaf(wgv, xv, gacc[t]);
                        uacc[t] = fmaf(wuv, xv, uacc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kWin; ++t) {
                if ((wm >> t) & 1u) {
                    const float gs = warp_sum(gacc[t]);
                    const float us = warp_sum(uacc[t]);
                    if (lane == 0) s_h[t0 + t][r] = silu(gs) * us;
                }
            }
        }
    }
    __syncthreads();

    // partial down projection over this tile's 64 columns, all d outputs
    for (int o = warp; o < d; o += kSimtWarps) {
        const float w0 = ld_val<WT>(wd + static_cast<size_t>(o) * f + lane);
        const float w1 = ld_val<WT>(wd + static_cast<size_t>(o) * f + lane + 32);
        for (int t0 = 0; t0 < kMaxPassTokens; t0 += kWin) {
            const uint32_t wm = static_cast<uint32_t>(mask >> t0) & 0xFFFFu;
            if (wm == 0u) continue;
#pragma unroll
            for (int t = 0; t < kWin; ++t) {
                if ((wm >> t) & 1u) {
                    const float p = warp_sum(w0 * s_h[t0 + t][lane] + w1 * s_h[t0 + t][lane + 32]);
                    if (lane == 0) atomicAdd(a.y + static_cast<size_t>(t0 + t) * d + o, s_gate[t0 + t] * p);
                }
            }
        }
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_expert_simt(const ExpertArgs &a, int groups, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.f / kFTile, groups);
    cfg.blockDim = dim3(kSimtThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.w_dtype == MOE_F32 && a.x_dtype == MOE_F32)
        return cudaLaunchKernelEx(&cfg, expert_simt_kernel<float, float>, a);
    if (a.w_dtype == MOE_BF16 && a.x_dtype == MOE_BF16)
        return cudaLaunchKernelEx(&cfg, expert_simt_kernel<__nv_bfloat16_raw, __nv_bfloat16_raw>, a);
    return cudaErrorInvalidValue;
}

}  // namespace moe
