// api.cu -- the C ABI of libmoeverify.so (declared in include/moe_verify.h).
//
// Host-side validation, dispatch to the kernels, and the host-only report math of
// "Speculative Decoding for Mixture-of-Experts Models" (Lan): requested bytes (§1
// "Bytes"), effective bandwidth, u_bar and r (§2), the saving and the crossover (§3.1,
// §2 "Testing the inputs"), E[U] under uniform routing (§1) and the best draft length
// (§1 "Speculative decoding").
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "common.cuh"
#include "expert_args.cuh"
#include "spec_args.cuh"

namespace moe {
cudaError_t launch_read_probe(const void *buf, size_t bytes, int32_t *err, cudaStream_t s);
}

namespace moe {
cudaError_t launch_route_topm(const float *logits, int n, int N, int m, int renorm, int32_t *ids, float *gates,
                              cudaStream_t s, bool pdl);
cudaError_t launch_group_slots(const int32_t *ids, int S, int N, int32_t *num_distinct, int32_t *expert_list,
                               int32_t *offsets, int32_t *order, int32_t *err, cudaStream_t s, bool pdl);
cudaError_t launch_quantize_rows(const void *src, int dtype, int rows, int cols, uint8_t *q, float *scale,
                                 cudaStream_t s, bool pdl);
}  // namespace moe

using namespace moe;

namespace {

constexpr bool kUsePdl = true;

// Cycles a device pipeline wait of the expert kernels may take (0: kWaitLimitCycles); set
// with moe_set_wait_limit.
std::atomic<long long> g_wait_limit{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// ids, gates, logits and groupings are read one element at a time: 4-byte alignment suffices
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool is_fp8(const moe_layer_t *L) { return L->w_dtype == MOE_E4M3 && L->x_dtype == MOE_E4M3; }

// the tensor-core path runs this layer (else the SIMT kernel): bf16 layers it supports, and
// every e4m3 layer (which has no other path)
bool uses_tc(const moe_layer_t *L) {
    if (is_fp8(L)) return true;
    return L->w_dtype == MOE_BF16 && L->x_dtype == MOE_BF16 && !(L->flags & MOE_FLAG_SIMT) &&
           expert_tc_supports(L->d, L->f);
}

moe_status_t check_layer(const moe_layer_t *L) {
    if (L == nullptr) return MOE_ERR_ARG;
    if (L->d <= 0 || L->f <= 0 || L->N <= 0 || L->m <= 0) return MOE_ERR_ARG;
    if (L->m > L->N || L->N > 1024) return MOE_ERR_UNSUPPORTED;
    if (L->d % 64 != 0 || L->f % 64 != 0 || L->d > 8192 || L->f > 65536) return MOE_ERR_UNSUPPORTED;
    const bool bf = L->w_dtype == MOE_BF16 && L->x_dtype == MOE_BF16;
    const bool fp = L->w_dtype == MOE_F32 && L->x_dtype == MOE_F32;
    if (!bf && !fp && !is_fp8(L)) return MOE_ERR_UNSUPPORTED;
    if (is_fp8(L) && (L->d % 128 != 0 || L->f % 128 != 0 || (L->flags & MOE_FLAG_SIMT))) return MOE_ERR_UNSUPPORTED;
    if ((L->flags & ~MOE_FLAG_SIMT) != 0) return MOE_ERR_ARG;
    return MOE_OK;
}

moe_status_t check_expert_common(const moe_layer_t *L, const void *wg, const void *wu, const void *wd,
                                 const void *x, const float *gates, int32_t n, const float *y, const void *ws,
                                 size_t ws_bytes) {
    moe_status_t st = check_layer(L);
    if (st != MOE_OK) return st;
    if (n < 1) return MOE_ERR_ARG;
    if (n > MOE_MAX_PASS_TOKENS) return MOE_ERR_UNSUPPORTED;
    const void *ptrs[] = {wg, wu, wd, x, y};
    for (const void *p : ptrs)
        if (p == nullptr || !aligned16(p)) return MOE_ERR_ARG;
    if (gates == nullptr || !aligned4(gates)) return MOE_ERR_ARG;
    if (ws == nullptr || ws_bytes < moe_workspace_bytes(L, n)) return MOE_ERR_WORKSPACE;
    if (!aligned16(ws)) return MOE_ERR_ARG;
    return MOE_OK;
}

ExpertArgs make_args(const moe_layer_t *L, const void *wg, const void *wu, const void *wd, const void *x,
                     const float *gates, int32_t n, float *y, void *ws, int mode) {
    ExpertArgs a;
    std::memset(&a, 0, sizeof a);
    a.w_gate = wg;
    a.w_up = wu;
    a.w_down = wd;
    a.x = x;
    a.gates = gates;
    a.y = y;
    a.err = &static_cast<DeviceWorkspace *>(ws)->error;
    a.d = L->d;
    a.f = L->f;
    a.N = L->N;
    a.m = L->m;
    a.n = n;
    a.mode = mode;
    a.w_dtype = L->w_dtype;
    a.x_dtype = L->x_dtype;
    const long long wl = g_wait_limit.load(std::memory_order_relaxed);
    a.wait_limit = wl > 0 ? wl : kWaitLimitCycles;
    return a;
}

moe_status_t run_expert(const moe_layer_t *L, const ExpertArgs &a, int max_groups, int32_t accumulate, void *ws,
                        cudaStream_t s) {
    cudaError_t e;
    if (uses_tc(L)) {
        // after the workspace header: the flags (sized for full passes, so that their place
        // does not depend on n), then the partial sums; the kernel zeroes y
        uint8_t *const w8 = static_cast<uint8_t *>(ws);
        ExpertArgs at = a;
        at.sync = &static_cast<DeviceWorkspace *>(ws)->sync[0];
        at.flags = reinterpret_cast<uint32_t *>(w8 + kWorkspaceBytes);
        uint64_t *part = reinterpret_cast<uint64_t *>(w8 + kWorkspaceBytes + expert_tc_flag_region(L->f, L->m));
        e = launch_expert_tc(at, max_groups, !accumulate, part, s, kUsePdl);
    } else {
        e = cudaSuccess;
        if (!accumulate) e = cudaMemsetAsync(a.y, 0, sizeof(float) * static_cast<size_t>(a.n) * a.d, s);
        if (e == cudaSuccess) e = launch_expert_simt(a, max_groups, s, kUsePdl);
    }
    if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_status(e);
}

// The deduplicating form from ids: the grouping built inside the kernel for up to
// kMaxFusedSlots slots, else by moe_group_slots' kernel into the workspace (after the partial
// sums of this pass), followed by the deduplicating kernel on it.
moe_status_t run_dedup_ids(const moe_layer_t *L, ExpertArgs a, int32_t n, int32_t accumulate, void *ws,
                           cudaStream_t s) {
    const int S = n * L->m;
    const int cap = S < L->N ? S : L->N;
    if (S <= kMaxFusedSlots) {
        a.mode = kModeDedupIds;
        return run_expert(L, a, cap, accumulate, ws, s);
    }
    uint8_t *const w8 = static_cast<uint8_t *>(ws);
    int32_t *const grp = reinterpret_cast<int32_t *>(w8 + kWorkspaceBytes + expert_tc_flag_region(L->f, L->m) +
                                                     round256(expert_tc_partial_bytes(L->f, L->m, n)));
    int32_t *const count = grp, *const list = grp + 1, *const offsets = list + L->N, *const order = offsets + L->N + 1;
    cudaError_t e = launch_group_slots(a.ids, S, L->N, count, list, offsets, order,
                                       &static_cast<DeviceWorkspace *>(ws)->error, s, kUsePdl);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    a.mode = kModeDedup;
    a.num_distinct = count;
    a.expert_list = list;
    a.offsets = offsets;
    a.slot_order = order;
    return run_expert(L, a, cap, accumulate, ws, s);
}

}  // namespace

namespace moe {
// The host checks of moe_expert_op_perslot that do not involve the workspace: the status it
// returns before any device work for these arguments (MOE_OK when they pass).
moe_status_t check_perslot_call(const moe_layer_t *L, const void *wg, const void *wu, const void *wd, const void *x,
                                const int32_t *ids, const float *gates, int32_t n, const float *y) {
    const moe_status_t st = check_layer(L);
    if (st != MOE_OK) return st;
    if (n < 1) return MOE_ERR_ARG;
    if (n > MOE_MAX_PASS_TOKENS) return MOE_ERR_UNSUPPORTED;
    const void *ptrs[] = {wg, wu, wd, x, y};
    for (const void *p : ptrs)
        if (p == nullptr || !aligned16(p)) return MOE_ERR_ARG;
    if (gates == nullptr || !aligned4(gates) || ids == nullptr || !aligned4(ids)) return MOE_ERR_ARG;
    if (is_fp8(L)) return MOE_ERR_UNSUPPORTED;   // e4m3 needs its scales: the _fp8 call
    return MOE_OK;
}

// The layer runs on the tensor-core path, whose workspace holds flags and partial sums.
bool layer_uses_tc(const moe_layer_t *L) { return check_layer(L) == MOE_OK && uses_tc(L); }
}  // namespace moe

namespace {
// Tokens per launch of a per-slot pass: the whole pass up to MOE_PERSLOT_LAUNCH_TOKENS; above,
// launches of up to 32 (one launch of the 32-token kernel is faster than two of 16) when the
// workspace holds that many, else of up to MOE_PERSLOT_LAUNCH_TOKENS, split evenly.  Passes are not
// run as launches of 64: the 64-token kernel streams a per-slot pass more slowly than two of 32.
int32_t perslot_launch_tokens(const moe_layer_t *L, int32_t n, size_t ws_bytes) {
    if (n <= MOE_PERSLOT_LAUNCH_TOKENS) return n;
    const int32_t wide = n < 32 ? n : 32;
    const int32_t cap = ws_bytes >= moe_workspace_bytes(L, wide) ? wide : MOE_PERSLOT_LAUNCH_TOKENS;
    const int32_t launches = (n + cap - 1) / cap;
    return (n + launches - 1) / launches;   // equal launches (40 tokens: two of 20, not 32 and 8)
}

// Element size of a layer's activations (bf16, fp32 or e4m3).
size_t x_elt_bytes(const moe_layer_t *L) { return L->x_dtype == MOE_BF16 ? 2u : (L->x_dtype == MOE_E4M3 ? 1u : 4u); }
}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

moe_status_t moe_set_wait_limit(int64_t cycles) {
    if (cycles < 0) return MOE_ERR_ARG;
    g_wait_limit.store(cycles, std::memory_order_relaxed);
    return MOE_OK;
}

const char *moe_status_str(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_ARG: return "invalid argument (null pointer, bad size or misaligned buffer)";
        case MOE_ERR_UNSUPPORTED: return "sizes or dtypes outside the supported range";
        case MOE_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_BAD_ID: return "an expert id outside [0, N) was skipped";
        case MOE_ERR_DEVICE_TIMEOUT: return "a device pipeline wait timed out";
    }
    return "unknown status";
}

size_t moe_workspace_bytes(const moe_layer_t *layer, int32_t n_max) {
    if (check_layer(layer) != MOE_OK || n_max < 1 || !uses_tc(layer)) return kWorkspaceBytes;
    const int n = n_max < MOE_MAX_PASS_TOKENS ? n_max : MOE_MAX_PASS_TOKENS;
    size_t bytes = kWorkspaceBytes + expert_tc_flag_region(layer->f, layer->m) +
                   round256(expert_tc_partial_bytes(layer->f, layer->m, n));
    if (n * layer->m > kMaxFusedSlots) bytes += dedup_grouping_bytes(layer->N, n * layer->m);
    return bytes;
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t s) {
    if (ws == nullptr || ws_bytes < kWorkspaceBytes) return MOE_ERR_WORKSPACE;
    if (!aligned16(ws)) return MOE_ERR_ARG;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(s)));
}

moe_status_t moe_route_topm(const float *logits, int32_t n, int32_t N, int32_t m, int32_t renorm, int32_t *ids,
                            float *gates, moe_stream_t s) {
    if (n < 0 || N < 1 || m < 1) return MOE_ERR_ARG;
    if (m > N || N > 1024 || m > 32) return MOE_ERR_UNSUPPORTED;
    if (n == 0) return MOE_OK;
    if (logits == nullptr || ids == nullptr || gates == nullptr) return MOE_ERR_ARG;
    if (!aligned4(logits) || !aligned4(ids) || !aligned4(gates)) return MOE_ERR_ARG;
    cudaError_t e = launch_route_topm(logits, n, N, m, renorm, ids, gates, reinterpret_cast<cudaStream_t>(s), kUsePdl);
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_status(e);
}

moe_status_t moe_group_slots(const int32_t *ids, int32_t n, int32_t m, int32_t N, int32_t *num_distinct,
                             int32_t *expert_list, int32_t *expert_offsets, int32_t *slot_order, void *ws,
                             moe_stream_t s) {
    if (n < 1 || m < 1 || N < 1) return MOE_ERR_ARG;
    if (static_cast<int64_t>(n) * m > 4096 || N > 1024) return MOE_ERR_UNSUPPORTED;
    const void *ptrs[] = {ids, num_distinct, expert_list, expert_offsets, slot_order};
    for (const void *p : ptrs)
        if (p == nullptr || !aligned4(p)) return MOE_ERR_ARG;
    if (ws != nullptr && !aligned16(ws)) return MOE_ERR_ARG;
    int32_t *err = ws ? &static_cast<DeviceWorkspace *>(ws)->error : nullptr;
    cudaError_t e = launch_group_slots(ids, n * m, N, num_distinct, expert_list, expert_offsets, slot_order, err,
                                       reinterpret_cast<cudaStream_t>(s), kUsePdl);
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_status(e);
}

moe_status_t moe_expert_op_perslot(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                   const void *w_down, const void *x, const int32_t *ids, const float *gates,
                                   int32_t n, int32_t accumulate, float *y, void *ws, size_t ws_bytes,
                                   moe_stream_t s) {
    moe_status_t st0 = check_perslot_call(layer, w_gate, w_up, w_down, x, ids, gates, n, y);
    if (st0 != MOE_OK) return st0;
    const int32_t cap = perslot_launch_tokens(layer, n, ws_bytes);
    if (cap < n && n <= MOE_MAX_PASS_TOKENS) {
        // consecutive launches of up to cap tokens (each validates its part)
        moe_status_t st = check_layer(layer);
        if (st != MOE_OK) return st;
        if (x == nullptr || ids == nullptr || gates == nullptr || y == nullptr) return MOE_ERR_ARG;
        const size_t xrow = static_cast<size_t>(layer->d) * x_elt_bytes(layer);
        for (int32_t t0 = 0; t0 < n; t0 += cap) {
            const int32_t nc = n - t0 < cap ? n - t0 : cap;
            const size_t so = static_cast<size_t>(t0) * layer->m;
            st = moe_expert_op_perslot(layer, w_gate, w_up, w_down, static_cast<const uint8_t *>(x) + t0 * xrow,
                                       ids + so, gates + so, nc, accumulate, y + static_cast<size_t>(t0) * layer->d,
                                       ws, ws_bytes, s);
            if (st != MOE_OK) return st;
        }
        return MOE_OK;
    }
    moe_status_t st = check_expert_common(layer, w_gate, w_up, w_down, x, gates, n, y, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (is_fp8(layer)) return MOE_ERR_UNSUPPORTED;   // e4m3 needs its scales: the _fp8 call
    if (ids == nullptr || !aligned4(ids)) return MOE_ERR_ARG;
    ExpertArgs a = make_args(layer, w_gate, w_up, w_down, x, gates, n, y, ws, kModePerSlot);
    a.ids = ids;
    return run_expert(layer, a, n * layer->m, accumulate, ws, reinterpret_cast<cudaStream_t>(s));
}

moe_status_t moe_expert_op_dedup(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                 const void *w_down, const void *x, const float *gates, int32_t n,
                                 const int32_t *num_distinct, const int32_t *expert_list,
                                 const int32_t *expert_offsets, const int32_t *slot_order, int32_t accumulate,
                                 float *y, void *ws, size_t ws_bytes, moe_stream_t s) {
    moe_status_t st = check_expert_common(layer, w_gate, w_up, w_down, x, gates, n, y, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (is_fp8(layer)) return MOE_ERR_UNSUPPORTED;   // e4m3 needs its scales: the _fp8 call
    const void *ptrs[] = {num_distinct, expert_list, expert_offsets, slot_order};
    for (const void *p : ptrs)
        if (p == nullptr || !aligned4(p)) return MOE_ERR_ARG;
    ExpertArgs a = make_args(layer, w_gate, w_up, w_down, x, gates, n, y, ws, kModeDedup);
    a.num_distinct = num_distinct;
    a.expert_list = expert_list;
    a.offsets = expert_offsets;
    a.slot_order = slot_order;
    const int cap = n * layer->m < layer->N ? n * layer->m : layer->N;
    return run_expert(layer, a, cap, accumulate, ws, reinterpret_cast<cudaStream_t>(s));
}

moe_status_t moe_expert_op_dedup_ids(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                     const void *w_down, const void *x, const int32_t *ids, const float *gates,
                                     int32_t n, int32_t accumulate, float *y, void *ws, size_t ws_bytes,
                                     moe_stream_t s) {
    moe_status_t st = check_expert_common(layer, w_gate, w_up, w_down, x, gates, n, y, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (is_fp8(layer) || !uses_tc(layer)) return MOE_ERR_UNSUPPORTED;
    if (ids == nullptr || !aligned4(ids)) return MOE_ERR_ARG;
    ExpertArgs a = make_args(layer, w_gate, w_up, w_down, x, gates, n, y, ws, kModeDedupIds);
    a.ids = ids;
    return run_dedup_ids(layer, a, n, accumulate, ws, reinterpret_cast<cudaStream_t>(s));
}

namespace {
// the kernels read scales one fp32 at a time: 4-byte alignment suffices
bool fp8_scales_ok(const moe_weight_scales_t *sc, const float *x_scale) {
    return sc != nullptr && sc->gate != nullptr && sc->up != nullptr && sc->down != nullptr && x_scale != nullptr &&
           aligned4(sc->gate) && aligned4(sc->up) && aligned4(sc->down) && aligned4(x_scale);
}
}  // namespace

moe_status_t moe_expert_op_perslot_fp8(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                       const void *w_down, const moe_weight_scales_t *scales, const void *x,
                                       const float *x_scale, const int32_t *ids, const float *gates, int32_t n,
                                       int32_t accumulate, float *y, void *ws, size_t ws_bytes, moe_stream_t s) {
    const int32_t cap = perslot_launch_tokens(layer, n, ws_bytes);
    if (cap < n && n <= MOE_MAX_PASS_TOKENS) {
        // consecutive launches of up to cap tokens (each validates its part)
        moe_status_t st = check_layer(layer);
        if (st != MOE_OK) return st;
        if (x == nullptr || x_scale == nullptr || ids == nullptr || gates == nullptr || y == nullptr) return MOE_ERR_ARG;
        const size_t xrow = static_cast<size_t>(layer->d) * x_elt_bytes(layer);
        for (int32_t t0 = 0; t0 < n; t0 += cap) {
            const int32_t nc = n - t0 < cap ? n - t0 : cap;
            const size_t so = static_cast<size_t>(t0) * layer->m;
            st = moe_expert_op_perslot_fp8(layer, w_gate, w_up, w_down, scales,
                                           static_cast<const uint8_t *>(x) + t0 * xrow, x_scale + t0, ids + so,
                                           gates + so, nc, accumulate, y + static_cast<size_t>(t0) * layer->d, ws,
                                           ws_bytes, s);
            if (st != MOE_OK) return st;
        }
        return MOE_OK;
    }
    moe_status_t st = check_expert_common(layer, w_gate, w_up, w_down, x, gates, n, y, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (!is_fp8(layer)) return MOE_ERR_UNSUPPORTED;
    if (ids == nullptr || !aligned4(ids) || !fp8_scales_ok(scales, x_scale)) return MOE_ERR_ARG;
    ExpertArgs a = make_args(layer, w_gate, w_up, w_down, x, gates, n, y, ws, kModePerSlot);
    a.ids = ids;
    a.s_gate = scales->gate;
    a.s_up = scales->up;
    a.s_down = scales->down;
    a.s_x = x_scale;
    return run_expert(layer, a, n * layer->m, accumulate, ws, reinterpret_cast<cudaStream_t>(s));
}

moe_status_t moe_expert_op_dedup_ids_fp8(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                         const void *w_down, const moe_weight_scales_t *scales, const void *x,
                                         const float *x_scale, const int32_t *ids, const float *gates, int32_t n,
                                         int32_t accumulate, float *y, void *ws, size_t ws_bytes, moe_stream_t s) {
    moe_status_t st = check_expert_common(layer, w_gate, w_up, w_down, x, gates, n, y, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (!is_fp8(layer)) return MOE_ERR_UNSUPPORTED;
    if (ids == nullptr || !aligned4(ids) || !fp8_scales_ok(scales, x_scale)) return MOE_ERR_ARG;
    ExpertArgs a = make_args(layer, w_gate, w_up, w_down, x, gates, n, y, ws, kModeDedupIds);
    a.ids = ids;
    a.s_gate = scales->gate;
    a.s_up = scales->up;
    a.s_down = scales->down;
    a.s_x = x_scale;
    return run_dedup_ids(layer, a, n, accumulate, ws, reinterpret_cast<cudaStream_t>(s));
}

moe_status_t moe_expert_op_dedup_fp8(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                     const void *w_down, const moe_weight_scales_t *scales, const void *x,
                                     const float *x_scale, const float *gates, int32_t n, const int32_t *num_distinct,
                                     const int32_t *expert_list, const int32_t *expert_offsets,
                                     const int32_t *slot_order, int32_t accumulate, float *y, void *ws,
                                     size_t ws_bytes, moe_stream_t s) {
    moe_status_t st = check_expert_common(layer, w_gate, w_up, w_down, x, gates, n, y, ws, ws_bytes);
    if (st != MOE_OK) return st;
    if (!is_fp8(layer)) return MOE_ERR_UNSUPPORTED;
    const void *ptrs[] = {num_distinct, expert_list, expert_offsets, slot_order};
    for (const void *p : ptrs)
        if (p == nullptr || !aligned4(p)) return MOE_ERR_ARG;
    if (!fp8_scales_ok(scales, x_scale)) return MOE_ERR_ARG;
    ExpertArgs a = make_args(layer, w_gate, w_up, w_down, x, gates, n, y, ws, kModeDedup);
    a.num_distinct = num_distinct;
    a.expert_list = expert_list;
    a.offsets = expert_offsets;
    a.slot_order = slot_order;
    a.s_gate = scales->gate;
    a.s_up = scales->up;
    a.s_down = scales->down;
    a.s_x = x_scale;
    const int cap = n * layer->m < layer->N ? n * layer->m : layer->N;
    return run_expert(layer, a, cap, accumulate, ws, reinterpret_cast<cudaStream_t>(s));
}

moe_status_t moe_quantize_rows_e4m3(const void *src, int32_t src_dtype, int32_t rows, int32_t cols, uint8_t *q,
                                    float *scale, moe_stream_t s) {
    if (src_dtype != MOE_F32 && src_dtype != MOE_BF16) return MOE_ERR_ARG;
    if (rows < 0 || cols < 1) return MOE_ERR_ARG;
    if (rows == 0) return MOE_OK;
    if (src == nullptr || q == nullptr || scale == nullptr) return MOE_ERR_ARG;
    cudaError_t e = launch_quantize_rows(src, src_dtype, rows, cols, q, scale, reinterpret_cast<cudaStream_t>(s),
                                         kUsePdl);
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_status(e);
}

moe_status_t moe_pass_bytes(const moe_layer_t *layer, const int32_t *ids_host, int32_t n, moe_pass_bytes_t *out) {
    moe_status_t st = check_layer(layer);
    if (st != MOE_OK) return st;
    if (ids_host == nullptr || out == nullptr || n < 0) return MOE_ERR_ARG;
    std::vector<uint8_t> seen(static_cast<size_t>(layer->N), 0);
    int32_t U = 0;
    const int64_t S = static_cast<int64_t>(n) * layer->m;
    for (int64_t s = 0; s < S; ++s) {
        const int32_t e = ids_host[s];
        if (e < 0 || e >= layer->N) return MOE_ERR_BAD_ID;
        if (!seen[e]) {
            seen[e] = 1;
            ++U;
        }
    }
    const uint64_t wsz = layer->w_dtype == MOE_BF16 ? 2u : (layer->w_dtype == MOE_E4M3 ? 1u : 4u);
    const uint64_t xsz = layer->x_dtype == MOE_BF16 ? 2u : (layer->x_dtype == MOE_E4M3 ? 1u : 4u);
    out->expert_bytes = 3ull * static_cast<uint64_t>(layer->d) * static_cast<uint64_t>(layer->f) * wsz;
    // an e4m3 expert also reads its fp32 row scales: 2f (gate, up) + d (down)
    if (layer->w_dtype == MOE_E4M3) out->expert_bytes += 4ull * (2ull * layer->f + layer->d);
    out->slot_bytes = static_cast<uint64_t>(S) * out->expert_bytes;
    out->dedup_bytes = static_cast<uint64_t>(U) * out->expert_bytes;
    out->act_bytes = static_cast<uint64_t>(n) * layer->d * xsz + static_cast<uint64_t>(n) * layer->d * 4ull +
                     (layer->x_dtype == MOE_E4M3 ? 4ull * n : 0ull);
    out->n = n;
    out->m = layer->m;
    out->U = U;
    out->reserved = 0;
    out->ubar = S > 0 ? static_cast<double>(U) / static_cast<double>(S) : 0.0;
    return MOE_OK;
}

moe_status_t moe_bandwidth_report(int32_t n_lo, int32_t count, const double *slot_bytes, const double *dedup_bytes,
                                  const double *t_slot, const double *t_dedup, double *beta_slot,
                                  double *beta_dedup, double *ubar, double *r, double *saving,
                                  int32_t *crossover) {
    if (count < 1 || !slot_bytes || !dedup_bytes || !t_slot || !t_dedup || !beta_slot || !beta_dedup || !ubar ||
        !r || !saving || !crossover)
        return MOE_ERR_ARG;
    for (int32_t i = 0; i < count; ++i) {
        if (!(t_slot[i] > 0.0) || !(t_dedup[i] > 0.0) || !(slot_bytes[i] > 0.0) || !(dedup_bytes[i] >= 0.0))
            return MOE_ERR_ARG;
    }
    for (int32_t i = 0; i < count; ++i) {
        beta_slot[i] = slot_bytes[i] / t_slot[i];
        beta_dedup[i] = dedup_bytes[i] / t_dedup[i];
        ubar[i] = dedup_bytes[i] / slot_bytes[i];
        r[i] = beta_dedup[i] / beta_slot[i];
        saving[i] = t_slot[i] - t_dedup[i];
    }
    // the smallest n from which the saving stays positive
    int32_t cross = -1;
    for (int32_t i = count - 1; i >= 0; --i) {
        if (saving[i] > 0.0) cross = n_lo + i;
        else break;
    }
    *crossover = cross;
    return MOE_OK;
}

double moe_expected_union(int32_t N, int32_t m, int32_t n) {
    if (N < 1 || m < 0 || m > N || n < 0) return NAN;
    const double q = 1.0 - static_cast<double>(m) / static_cast<double>(N);
    return static_cast<double>(N) * (1.0 - std::pow(q, static_cast<double>(n)));
}

int32_t moe_best_draft_length(const double *V, int32_t kmax, double a) {
    if (V == nullptr || kmax < 0 || !(a >= 0.0) || !(a < 1.0)) return -1;
    int32_t best = -1;
    double best_T = 0.0, G = 0.0, p = 1.0;
    for (int32_t k = 0; k <= kmax; ++k) {
        if (!(V[k] > 0.0)) return -1;
        G += p;   // G_a(k) = 1 + a + ... + a^k
        p *= a;
        const double T = G / V[k];
        if (best < 0 || T > best_T) {
            best = k;
            best_T = T;
        }
    }
    return best;
}

// ---------------------------------------------------------------- step-time theory

namespace {

// G_a(k) = 1 + a + ... + a^k by Horner's rule.
double expected_tokens(double a, int k) {
    double g = 1.0;
    for (int i = 0; i < k; ++i) g = 1.0 + a * g;
    return g;
}

// q(a) > 0 exactly when T_a(k) > T_a(i) (i < k): G_a(k) V(i) - G_a(i) V(k), written as
// V(i) a^{i+1} G_a(k-i-1) - G_a(i) (V(k) - V(i)) so that equal step times do not cancel.
double faster_margin(const double *V, int k, int i, double a) {
    return V[i] * std::pow(a, i + 1) * expected_tokens(a, k - i - 1) - expected_tokens(a, i) * (V[k] - V[i]);
}

// alpha_{k,i}: the boundary of {a in [0,1) : q(a) > 0}, an upward-closed set (G_a(k)/G_a(i)
// rises with a towards (k+1)/(i+1)); bracketed regula falsi with the Illinois step.
double alpha_of(const double *V, int k, int i) {
    if (V[k] < V[i]) return 0.0;                                          // q(0) = V(i) - V(k)
    if ((k + 1) * V[i] <= (i + 1) * V[k]) return 1.0;                     // q(a) <= 0 below a = 1
    double lo = 0.0, hi = 1.0, qlo = faster_margin(V, k, i, 0.0), qhi = (k + 1) * V[i] - (i + 1) * V[k];
    int side = 0;
    for (int it = 0; it < 400 && hi - lo > 1e-17; ++it) {
        double x = (qhi - qlo) != 0.0 ? (lo * qhi - hi * qlo) / (qhi - qlo) : 0.5 * (lo + hi);
        if (!(x > lo && x < hi)) x = 0.5 * (lo + hi);
        const double qx = faster_margin(V, k, i, x);
        if (qx > 0.0) {
            hi = x;
            qhi = qx;
            if (side == 1) qlo *= 0.5;
            side = 1;
        } else {
            lo = x;
            qlo = qx;
            if (side == -1) qhi *= 0.5;
            side = -1;
        }
    }
    return hi;
}

bool valid_times(const double *V, int kmax) {
    if (V == nullptr || kmax < 0) return false;
    for (int k = 0; k <= kmax; ++k)
        if (!(V[k] > 0.0) || !std::isfinite(V[k])) return false;
    return true;
}

}  // namespace

moe_status_t moe_staircase(const double *V, int32_t kmax, double *a0, double *a_step, double *alpha,
                           int32_t *convex) {
    if (kmax < 1 || kmax > 64 || !valid_times(V, kmax) || a0 == nullptr || a_step == nullptr || convex == nullptr)
        return MOE_ERR_ARG;
    const int K = kmax + 1;
    std::vector<double> al(static_cast<size_t>(K) * K, 0.0);
    for (int k = 1; k <= kmax; ++k)
        for (int i = 0; i < k; ++i) al[static_cast<size_t>(k) * K + i] = alpha_of(V, k, i);
    a_step[0] = 0.0;
    for (int j = 1; j <= kmax; ++j) {
        double best = 0.0;
        for (int i = 0; i < j; ++i) {
            double mn = 1.0;
            for (int k = j; k <= kmax; ++k) mn = std::min(mn, al[static_cast<size_t>(k) * K + i]);
            best = i == 0 ? mn : std::max(best, mn);
        }
        a_step[j] = best;
    }
    if (alpha != nullptr) std::memcpy(alpha, al.data(), al.size() * sizeof(double));
    *a0 = V[1] / V[0] - 1.0;
    int cv = 1;
    double c_prev = 0.0;
    for (int i = 1; i <= kmax; ++i) {
        const double c = V[i] - V[i - 1];
        if (c < c_prev) cv = 0;
        c_prev = c;
    }
    *convex = cv;
    return MOE_OK;
}

double moe_speedup(const double *V, int32_t kmax, int32_t k, double a) {
    if (!valid_times(V, kmax) || k < 0 || k > kmax || !(a >= 0.0) || !(a < 1.0)) return NAN;
    return expected_tokens(a, k) * V[0] / V[k];
}

double moe_reuse_threshold(int32_t k, double a, const moe_threshold_in_t *in) {
    if (in == nullptr || k < 1 || !(a >= 0.0) || !(a < 1.0) || !(in->mW > 0.0) || !(in->B_k > 0.0) ||
        !(in->beta_1 > 0.0))
        return NAN;
    const double bracket = (expected_tokens(a, k) - 1.0) * in->tau_1 - in->dD_over_betaD - in->dphi;
    return 1.0 - in->B_k / (in->mW * k) * bracket - (in->B_k / in->beta_1 - 1.0) / k;
}

double moe_reuse_threshold_bytes(int32_t k, double a, double mW, double D_1, double D_k1) {
    if (k < 1 || !(a >= 0.0) || !(a < 1.0) || !(mW > 0.0)) return NAN;
    return 1.0 - ((expected_tokens(a, k) - 1.0) * (D_1 + mW) - (D_k1 - D_1)) / (mW * k);
}

moe_status_t moe_error_bounds(double eps, moe_error_bounds_t *out) {
    if (out == nullptr || !(eps >= 0.0) || !(eps < 0.5)) return MOE_ERR_ARG;
    const double d = eps / (1.0 - eps);
    out->delta = d;
    out->verify_factor = d;
    out->decision_log_margin = std::log1p(eps) - std::log1p(-eps);
    out->regret_factor = (1.0 - d) / (1.0 + d);
    out->speedup_lo = (1.0 - d) / (1.0 + d);
    out->speedup_hi = (1.0 + d) / (1.0 - d);
    return MOE_OK;
}

int32_t moe_kstar_separated(const double *V, int32_t kmax, double a, double delta) {
    if (!(delta >= 0.0) || !(delta < 1.0)) return -1;
    const int32_t ks = moe_best_draft_length(V, kmax, a);
    if (ks < 0) return -1;
    const double top = expected_tokens(a, ks) / V[ks];
    const double f = (1.0 + delta) / (1.0 - delta);
    for (int32_t i = 0; i <= kmax; ++i)
        if (i != ks && !(f * expected_tokens(a, i) / V[i] < top)) return 0;
    return 1;
}

moe_status_t moe_fit_op_times(int32_t count, const int32_t *n, const int32_t *U, const double *t, int32_t m,
                              double b, int32_t form, double *coef) {
    if (count < 3 || n == nullptr || U == nullptr || t == nullptr || coef == nullptr || m < 1 || !(b > 0.0) ||
        (form != 0 && form != 1))
        return MOE_ERR_ARG;
    // columns of the design matrix, each scaled to unit norm, then a modified Gram-Schmidt QR
    const size_t C = static_cast<size_t>(count);
    std::vector<double> A(3 * C);
    for (size_t r = 0; r < C; ++r) {
        if (n[r] < 1 || U[r] < 0 || !std::isfinite(t[r])) return MOE_ERR_ARG;
        A[r] = 1.0;
        A[C + r] = static_cast<double>(U[r]) * b;
        A[2 * C + r] = form == 0 ? (static_cast<double>(n[r]) * m - U[r]) * b : static_cast<double>(n[r]);
    }
    double scale[3], R[3][3] = {{0.0}}, qt[3];
    for (int j = 0; j < 3; ++j) {
        double nn = 0.0;
        for (size_t r = 0; r < C; ++r) nn += A[j * C + r] * A[j * C + r];
        scale[j] = std::sqrt(nn);
        if (!(scale[j] > 0.0)) return MOE_ERR_ARG;
        for (size_t r = 0; r < C; ++r) A[j * C + r] /= scale[j];
    }
    std::vector<double> y(t, t + C);
    for (int j = 0; j < 3; ++j) {
        for (int i = 0; i < j; ++i) {
            double dot = 0.0;
            for (size_t r = 0; r < C; ++r) dot += A[i * C + r] * A[j * C + r];
            R[i][j] = dot;
            for (size_t r = 0; r < C; ++r) A[j * C + r] -= dot * A[i * C + r];
        }
        double nn = 0.0;
        for (size_t r = 0; r < C; ++r) nn += A[j * C + r] * A[j * C + r];
        R[j][j] = std::sqrt(nn);
        if (!(R[j][j] > 1e-10)) return MOE_ERR_ARG;   // rank below 3
        for (size_t r = 0; r < C; ++r) A[j * C + r] /= R[j][j];
        double dot = 0.0;
        for (size_t r = 0; r < C; ++r) dot += A[j * C + r] * y[r];
        qt[j] = dot;
        for (size_t r = 0; r < C; ++r) y[r] -= dot * A[j * C + r];
    }
    double x[3];
    for (int j = 2; j >= 0; --j) {
        double v = qt[j];
        for (int k = j + 1; k < 3; ++k) v -= R[j][k] * x[k];
        x[j] = v / R[j][j];
    }
    for (int j = 0; j < 3; ++j) coef[j] = x[j] / scale[j];
    return MOE_OK;
}

moe_status_t moe_spec_accept(const int32_t *draft, const float *q, const float *p, const float *r, const float *u,
                             int32_t B, int32_t K, int32_t V, int32_t greedy, int32_t *n_accepted, int32_t *token,
                             moe_stream_t s) {
    if (B < 0 || K < 0 || V < 1) return MOE_ERR_ARG;
    if (K > kMaxSpecK || V > kMaxSpecV) return MOE_ERR_UNSUPPORTED;
    if (B == 0) return MOE_OK;
    auto al4 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
    if (p == nullptr || n_accepted == nullptr || token == nullptr || !al4(p) || !al4(n_accepted) || !al4(token))
        return MOE_ERR_ARG;
    if (K > 0 && (draft == nullptr || !al4(draft))) return MOE_ERR_ARG;
    if (!greedy) {
        if (u == nullptr || !al4(u)) return MOE_ERR_ARG;
        if (K > 0 && (q == nullptr || r == nullptr || !al4(q) || !al4(r))) return MOE_ERR_ARG;
    }
    SpecArgs a;
    a.draft = draft;
    a.q = q;
    a.p = p;
    a.r = r;
    a.u = u;
    a.n_acc = n_accepted;
    a.token = token;
    a.B = B;
    a.K = K;
    a.V = V;
    a.greedy = greedy ? 1 : 0;
    a.seg = spec_segment(V);
    a.vec = (V % 4 == 0 && aligned16(p) && (greedy || K == 0 || aligned16(q))) ? 1 : 0;
    cudaError_t e = launch_spec_accept(a, reinterpret_cast<cudaStream_t>(s), kUsePdl);
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_status(e);
}

size_t moe_union_cost_workspace_bytes(int32_t count) {
    return count < 1 ? 16 : round256(union_cost_scratch_bytes(count));
}

moe_status_t moe_union_cost(const uint64_t *bitmaps, int32_t nodes, int32_t L, int32_t W, const uint32_t *subsets,
                            int32_t count, const double *pv, const double *bcoef, double beta, int32_t *F,
                            int32_t *size, double *R, double *T, int32_t *best, void *ws, size_t ws_bytes,
                            moe_stream_t s) {
    if (nodes < 0 || L < 1 || W < 1 || count < 0) return MOE_ERR_ARG;
    if (nodes > 32 || static_cast<size_t>(nodes + 1) * L * W * sizeof(uint64_t) > kMaxUnionSmem)
        return MOE_ERR_UNSUPPORTED;
    if (best == nullptr || (reinterpret_cast<uintptr_t>(best) & 3u) != 0) return MOE_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
    if (count == 0) return cuda_status(cudaMemsetAsync(best, 0xFF, sizeof(int32_t), st));
    auto al = [](const void *ptr, uintptr_t m) { return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & m) == 0; };
    if (!al(bitmaps, 7) || !al(subsets, 3) || !al(bcoef, 7) || !al(F, 3) || !al(size, 3) || !al(R, 7) || !al(T, 7))
        return MOE_ERR_ARG;
    if (nodes > 0 && !al(pv, 7)) return MOE_ERR_ARG;
    if (ws == nullptr || !aligned16(ws)) return MOE_ERR_ARG;
    if (ws_bytes < moe_union_cost_workspace_bytes(count)) return MOE_ERR_WORKSPACE;
    UnionArgs a;
    a.bitmaps = bitmaps;
    a.subsets = subsets;
    a.pv = pv;
    a.bcoef = bcoef;
    a.beta = beta;
    a.F = F;
    a.size = size;
    a.R = R;
    a.T = T;
    a.best = best;
    a.nodes = nodes;
    a.L = L;
    a.W = W;
    a.count = count;
    cudaError_t e = launch_union_cost(a, ws, st, kUsePdl);
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_status(e);
}

moe_status_t moe_read_probe(const void *buf, size_t bytes, void *ws, moe_stream_t s) {
    if (buf == nullptr || !aligned16(buf) || ws == nullptr || !aligned16(ws)) return MOE_ERR_ARG;
    if (bytes < 32768) return MOE_ERR_ARG;
    cudaError_t e = launch_read_probe(buf, bytes, &static_cast<DeviceWorkspace *>(ws)->error,
                                      reinterpret_cast<cudaStream_t>(s));
    return cuda_status(e);
}

moe_status_t moe_last_device_error(void *ws, moe_stream_t s, int32_t *code) {
    if (ws == nullptr || code == nullptr) return MOE_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(ws, 0, sizeof v) != cudaSuccess) return MOE_ERR_CUDA;
    *code = v;
    return MOE_OK;
}

}  // extern "C"
