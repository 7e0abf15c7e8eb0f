// route.cu -- top-m routing with softmax gates.
//
// "Speculative Decoding for Mixture-of-Experts Models" (Lan), §1 "Routing, union and
// reuse": the router selects a set of m of the N experts for each token; the gates are
// the softmax over the selected logits (the full softmax renormalised over the set), or
// the full softmax over all N when renormalisation is off.
//
// One warp per token.  Each lane owns the logits of experts lane, lane+32, ... (at most
// 32 per lane, N <= 1024) as order-preserving 64-bit keys (value, then lower id first);
// m rounds of a warp-wide max pick the experts in order.  Comparisons are exact, so the
// selected ids equal those of any exact sort with the same tie rule.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 4;
constexpr int kMaxPerLane = 32;   // N <= 1024

// Order-preserving 32-bit key of a float: larger float -> larger key; -0 == +0;
// NaN below every number (key 0).
__device__ __forceinline__ uint32_t float_key(float v) {
    if (v != v) return 0u;
    if (v == 0.0f) v = 0.0f;   // canonical zero
    uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint64_t make_key(float v, int e) {
    // ties: the lower id ranks first, so it gets the larger low word
    return (static_cast<uint64_t>(float_key(v)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

__global__ void __launch_bounds__(kRouteWarps * 32)
route_topm_kernel(const float *__restrict__ logits, int n, int N, int m, int renorm,
                  int32_t *__restrict__ ids, float *__restrict__ gates) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t < n) {
        const float *z = logits + static_cast<size_t>(t) * N;
        float v[kMaxPerLane];
        uint32_t taken = 0;   // bit k: expert lane + 32k already selected
#pragma unroll
        for (int k = 0; k < kMaxPerLane; ++k) {
            const int e = lane + 32 * k;
            v[k] = (e < N) ? z[e] : 0.0f;
        }
        float zmax = 0.0f, denom = 0.0f, my_z = 0.0f;
        int my_id = 0;
        for (int j = 0; j < m; ++j) {
            uint64_t best = 0;
#pragma unroll
            for (int k = 0; k < kMaxPerLane; ++k) {
                const int e = lane + 32 * k;
                if (e < N && !((taken >> k) & 1u)) {
                    const uint64_t key = make_key(v[k], e);
                    best = key > best ? key : best;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, best, off);
                best = other > best ? other : best;
            }
            int e_sel = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFu));
            e_sel = min(max(e_sel, 0), N - 1);   // unreachable guard: m <= N always leaves a candidate
            if ((e_sel & 31) == lane) taken |= 1u << (e_sel >> 5);
            const float z_sel = z[e_sel];
            if (j == 0) zmax = z_sel;
            if (j == lane) { my_z = z_sel; my_id = e_sel; }
            if (renorm) denom += expf(z_sel - zmax);
        }
        if (!renorm) {
            float part = 0.0f;
#pragma unroll
            for (int k = 0; k < kMaxPerLane; ++k) {
                const int e = lane + 32 * k;
                if (e < N) part += expf(v[k] - zmax);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
            denom = part;
        }
        if (lane < m) {
            ids[static_cast<size_t>(t) * m + lane] = my_id;
            gates[static_cast<size_t>(t) * m + lane] = expf(my_z - zmax) / denom;
        }
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_route_topm(const float *logits, int n, int N, int m, int renorm, int32_t *ids,
                              float *gates, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((n + kRouteWarps - 1) / kRouteWarps);
    cfg.blockDim = dim3(kRouteWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_topm_kernel, logits, n, N, m, renorm, ids, gates);
}

}  // namespace moe
