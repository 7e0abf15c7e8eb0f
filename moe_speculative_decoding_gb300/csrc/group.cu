// group.cu -- slot grouping by expert (counting sort).
//
// "Speculative Decoding for Mixture-of-Experts Models" (Lan), §1: a deduplicating kernel
// groups the pass's tokens by expert; App. E "Engine changes": the deduplicating engine
// sorts rows by expert.  Histogram over the N experts, exclusive scan over the bins
// (distinct experts in ascending id order), then a stable scatter of slot indices.
//
// One CTA of 1024 threads: thread e owns bin e during the scan (N <= 1024); the pass has
// at most 4096 slots, held in shared memory.  The rank of a slot inside its bin is the
// count of earlier slots with the same expert, which makes the scatter stable.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kGroupThreads = 1024;
constexpr int kGroupMaxSlots = 4096;
constexpr int kGroupMaxExperts = 1024;

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += y;
    }
    return v;
}

__global__ void __launch_bounds__(kGroupThreads)
group_slots_kernel(const int32_t *__restrict__ ids, int S, int N, int32_t *__restrict__ num_distinct,
                   int32_t *__restrict__ expert_list, int32_t *__restrict__ offsets,
                   int32_t *__restrict__ order, int32_t *err) {
    __shared__ int32_t s_ids[kGroupMaxSlots];
    __shared__ int32_t s_count[kGroupMaxExperts];
    __shared__ int32_t s_start[kGroupMaxExperts];
    __shared__ int32_t s_warp_cnt[32];
    __shared__ int32_t s_warp_flag[32];

    pdl_wait();
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < N; e += kGroupThreads) s_count[e] = 0;
    __syncthreads();
    for (int s = tid; s < S; s += kGroupThreads) {
        const int e = ids[s];
        const bool ok = (e >= 0) && (e < N);
        s_ids[s] = ok ? e : -1;
        if (ok) atomicAdd(&s_count[e], 1);
        else record_error(err, MOE_ERR_BAD_ID);
    }
    __syncthreads();

    // exclusive scans over the bins of (count) and (count > 0)
    const int c = (tid < N) ? s_count[tid] : 0;
    const int flag = c > 0 ? 1 : 0;
    const int inc_c = warp_inclusive_scan(c, lane);
    const int inc_f = warp_inclusive_scan(flag, lane);
    if (lane == 31) {
        s_warp_cnt[warp] = inc_c;
        s_warp_flag[warp] = inc_f;
    }
    __syncthreads();
    if (warp == 0) {
        const int a = warp_inclusive_scan(s_warp_cnt[lane], lane);
        const int b = warp_inclusive_scan(s_warp_flag[lane], lane);
        s_warp_cnt[lane] = a;
        s_warp_flag[lane] = b;
    }
    __syncthreads();
    const int base_c = warp > 0 ? s_warp_cnt[warp - 1] : 0;
    const int base_f = warp > 0 ? s_warp_flag[warp - 1] : 0;
    const int start = base_c + inc_c - c;
    const int idx = base_f + inc_f - flag;
    if (tid < N) {
        s_start[tid] = start;
        if (flag) {
            expert_list[idx] = tid;
            offsets[idx] = start;
        }
    }
    if (tid == 0) {
        const int U = s_warp_flag[31];
        num_distinct[0] = U;
        offsets[U] = s_warp_cnt[31];
    }
    __syncthreads();

    // stable scatter: rank = earlier slots naming the same expert
    for (int s = tid; s < S; s += kGroupThreads) {
        const int e = s_ids[s];
        if (e < 0) continue;
        int rank = 0;
        for (int s2 = 0; s2 < s; ++s2) rank += (s_ids[s2] == e) ? 1 : 0;
        order[s_start[e] + rank] = s;
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_group_slots(const int32_t *ids, int S, int N, int32_t *num_distinct,
                               int32_t *expert_list, int32_t *offsets, int32_t *order, int32_t *err,
                               cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kGroupThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, group_slots_kernel, ids, S, N, num_distinct, expert_list, offsets,
                              order, err);
}

}  // namespace moe
