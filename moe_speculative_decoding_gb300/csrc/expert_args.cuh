// expert_args.cuh -- arguments shared by the expert-operation kernels.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {

constexpr int kMaxPassTokens = MOE_MAX_PASS_TOKENS;   // tokens per pass (MMA N = 16, 32 or 64)
constexpr int kPerSlotLaunchTokens = MOE_PERSLOT_LAUNCH_TOKENS;   // tokens per launch of the per-slot calls
constexpr int kFTile = 64;                             // rows of f per work item

// kModeDedupIds: the deduplicating form from the slots' ids, the grouping built inside the
// tensor-core kernel (at most kMaxFusedSlots slots).
enum : int { kModePerSlot = 0, kModeDedup = 1, kModeDedupIds = 2 };
constexpr int kMaxFusedSlots = 256;

// One call of the expert operation.  Per-slot form: group g is slot g (expert ids[g],
// token g / m).  Deduplicating form: group g is expert_list[g] with the slots
// slot_order[offsets[g] .. offsets[g+1]); the number of groups is num_distinct[0].
struct ExpertArgs {
    const void *w_gate;
    const void *w_up;
    const void *w_down;
    const void *x;
    const int32_t *ids;
    const float *gates;
    const int32_t *num_distinct;
    const int32_t *expert_list;
    const int32_t *offsets;
    const int32_t *slot_order;
    float *y;
    int32_t *err;
    // e4m3 layers: fp32 scale of each weight row ([N, f], [N, f], [N, d]) and of each token
    // ([n]); null for bf16
    const float *s_gate, *s_up, *s_down, *s_x;
    // tensor-core path: the workspace's epoch word and CTA exit count ([0], [1]), and its
    // flags (expert_tc_flag_bytes)
    uint32_t *sync;
    uint32_t *flags;
    int d, f, N, m, n, mode, w_dtype, x_dtype;
    // cycles a pipeline wait may take before the call gives up with MOE_ERR_DEVICE_TIMEOUT
    long long wait_limit;
};

cudaError_t launch_expert_simt(const ExpertArgs &a, int groups, cudaStream_t s, bool pdl);

// Tensor-core path (bf16 or e4m3): one kernel, one CTA per SM.  Its CTAs share each
// (group, f tile) gate/up item's k blocks, at most kMaxSpan CTAs to an item, and hand their
// fp32 partial sums to the CTAs that form h through `part`: kMaxSpan * 128 tagged 64-bit words
// (value and the call's ticket) per (slot position, f tile), expert_tc_partial_bytes in all.
// `flags` (expert_tc_flag_bytes) holds the y-zeroing flags of each (CTA, epilogue warp).
// Neither region needs clearing between calls: everything in them carries a call's ticket,
// and the workspace is zeroed once when it is initialised.  zero_y: y is overwritten (zeroed
// inside the kernel) rather than added to.  Returns cudaErrorNotSupported when the shape is
// outside what it handles (the caller then reports MOE_ERR_UNSUPPORTED).
constexpr int kMaxSpan = 3;
constexpr int kMaxGrid = 256;   // CTAs of one call at most
inline size_t expert_tc_partial_bytes(int f, int m, int n) {
    return static_cast<size_t>(n) * m * (f / kFTile) * kMaxSpan * 128 * sizeof(uint64_t);
}
inline size_t expert_tc_flag_bytes(int f, int m, int n) {
    (void)f, (void)m, (void)n;
    return static_cast<size_t>(kMaxGrid) * 4 * sizeof(uint32_t);
}
inline size_t round256(size_t bytes) { return (bytes + 255) / 256 * 256; }
// The grouping the deduplicating call from ids keeps in the workspace for a pass of S >
// kMaxFusedSlots slots: the count, up to N experts, N + 1 offsets and the S-entry slot order.
inline size_t dedup_grouping_bytes(int N, int S) { return round256(static_cast<size_t>(4) * (2 * N + S + 2)); }
// The workspace's flag region: its size does not depend on the pass (the partial sums follow it).
inline size_t expert_tc_flag_region(int f, int m) { return round256(expert_tc_flag_bytes(f, m, kMaxPassTokens)); }
cudaError_t launch_expert_tc(const ExpertArgs &a, int max_groups, bool zero_y, uint64_t *part, cudaStream_t s,
                             bool pdl);
bool expert_tc_supports(int d, int f);

// Host checks shared by the per-slot entry points (api.cu): the status moe_expert_op_perslot
// returns for these arguments before any device work, leaving out the workspace, and whether
// a layer runs on the tensor-core path.
moe_status_t check_perslot_call(const moe_layer_t *L, const void *wg, const void *wu, const void *wd, const void *x,
                                const int32_t *ids, const float *gates, int32_t n, const float *y);
bool layer_uses_tc(const moe_layer_t *L);

}  // namespace moe
