/*
 * moe_verify.h -- C ABI of libmoeverify.so: the MoE expert operation of a
 * speculative-decoding verification pass on one NVIDIA GB300 (sm_103a).
 *
 * Source of the method: "Speculative Decoding for Mixture-of-Experts Models: Expert
 * Bytes, Kernel Bandwidth and the Best Draft Length" (Lan), cited as [Lan] with the
 * section, equation or appendix that defines each operation.
 *
 * Conventions shared by every call
 * --------------------------------
 *  * Ownership: the caller owns every buffer (device or host).  The library never
 *    allocates or frees device memory; scratch comes from a caller-provided workspace
 *    of moe_workspace_bytes() bytes.
 *  * Pointers marked [dev] are device pointers, [host] host pointers.  Weights, x, y and
 *    workspaces must be 16-byte aligned; routing arrays (logits, ids, gates, the grouping)
 *    and scale arrays, which the kernels read one element at a time, need only 4-byte
 *    alignment (so per-layer slices of one ids array stay valid for any n and m).  Weight
 *    and activation buffers must also be contiguous row-major in the layouts stated below.
 *  * Asynchrony: a call that takes a stream enqueues its kernels on that stream and
 *    returns without synchronising.  The host-only calls and moe_last_device_error (which
 *    synchronises the stream) are the exceptions.
 *  * Errors: every call returns a moe_status_t.  Arguments are validated on the host
 *    before anything is launched (MOE_ERR_ARG / MOE_ERR_UNSUPPORTED, nothing enqueued).
 *    A failed launch returns MOE_ERR_CUDA.  Problems only the device can see (an expert
 *    id outside [0, N), a pipeline wait that timed out) are recorded in the workspace and
 *    read back with moe_last_device_error; the offending slots are skipped, never
 *    dereferenced.  Nothing throws across the ABI.
 *  * Threading: calls are re-entrant; calls that share a workspace must be ordered on
 *    one stream.
 */
#ifndef MOE_VERIFY_H
#define MOE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *moe_stream_t;

#define MOE_ABI_VERSION 2

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = 1,            /* null pointer, bad size or misaligned buffer */
    MOE_ERR_UNSUPPORTED = 2,    /* sizes or dtypes outside the supported range */
    MOE_ERR_CUDA = 3,           /* a CUDA runtime call or a launch failed */
    MOE_ERR_WORKSPACE = 4,      /* workspace missing or smaller than moe_workspace_bytes() */
    MOE_ERR_BAD_ID = 5,         /* (device) an expert id outside [0, N) was skipped */
    MOE_ERR_DEVICE_TIMEOUT = 6  /* (device) a pipeline wait gave up after its time limit */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2 } moe_dtype_t;

/*
 * One MoE layer [Lan, §1: N experts, each token routed to m of them].
 *   d  hidden size; f  expert intermediate size; N  experts; m  experts per token.
 *   w_dtype  dtype of the expert weights; x_dtype  dtype of the pass activations.
 * Weight layouts (row-major, one contiguous block per expert, nn.Linear convention):
 *   w_gate, w_up  [N, f, d];   w_down  [N, d, f].
 * Supported: 1 <= m <= N <= 1024, d and f multiples of 64, d <= 8192, f <= 65536;
 * (w_dtype, x_dtype) = (MOE_BF16, MOE_BF16), (MOE_F32, MOE_F32) or (MOE_E4M3, MOE_E4M3).
 * The tensor-core kernels take bf16 layers with d a multiple of 128; other bf16 shapes run
 * on the CUDA-core kernel.  e4m3 layers (OCP FP8 E4M3 codes, one fp32 scale per weight row
 * and per token, see moe_quantize_rows_e4m3) run only through the _fp8 calls, on the
 * tensor cores, with d and f multiples of 128.
 */
typedef struct {
    int32_t d, f, N, m;
    int32_t w_dtype, x_dtype;
    int32_t flags;   /* 0, or MOE_FLAG_SIMT */
} moe_layer_t;

/* flags: run the expert operation on the CUDA-core kernel even for bf16 layers (the
 * tensor-core kernel is the default for bf16; fp32 layers always use the CUDA cores). */
#define MOE_FLAG_SIMT 1

/* Largest pass size (tokens per verification pass) every expert-operation call accepts. */
#define MOE_MAX_PASS_TOKENS 64
/* The per-slot calls run a pass above this many tokens as consecutive launches of equal size, up
 * to 32 tokens when the workspace holds moe_workspace_bytes(layer, min(n, 32)), else up to this many
 * (the per-slot form reads every slot's expert either way), so their workspace needs only
 * moe_workspace_bytes(layer, MOE_PERSLOT_LAUNCH_TOKENS).  The deduplicating calls run a pass of
 * up to MOE_MAX_PASS_TOKENS in one launch: a distinct expert is read once for all of its tokens. */
#define MOE_PERSLOT_LAUNCH_TOKENS 16
/* The per-slot calls' pass limit (the same as every call's). */
#define MOE_MAX_PERSLOT_TOKENS 64

/* Returns MOE_ABI_VERSION.  Library infrastructure: no passage of the pages defines it. */
int32_t moe_abi_version(void);

/* Static description of a status code (never NULL).  Library infrastructure: no passage of the
 * pages defines it. */
const char *moe_status_str(moe_status_t status);

/*
 * Bytes of device workspace the expert-operation calls need for this layer and passes
 * of up to n_max tokens: 256 bytes holding the device error word and, for layers the
 * tensor-core kernel runs, a flag region of 4096 bytes (the per-call flags with which the
 * kernel's CTAs publish their zeroing of y) and the gate/up partial sums the CTAs hand to
 * each other, 3 * 128 tagged 64-bit words (an fp32 value and the call's ticket) per (slot,
 * 64-row tile of f): 256 + 4096 + round256(n_max*m*(f/64)*3072) bytes (4.72 MB for d = 2048,
 * f = 768, top-8 at 16 tokens).
 * Zero it once with moe_workspace_init before its first use.  Calls never clear it: every
 * call takes a new ticket (the workspace counts its calls), and a flag or a partial sum counts
 * only when it carries the reading call's ticket, so a workspace may move between layers of
 * any shape without being zeroed again.  Tickets are 32-bit: zero a workspace again at least
 * once in 2^32 calls.
 * n_max above MOE_MAX_PASS_TOKENS counts as MOE_MAX_PASS_TOKENS.  For a pass of more than
 * 256 slots (n_max*m > 256) the deduplicating call from ids also keeps the pass's grouping
 * there: round256(4 * (2*N + n_max*m + 2)) bytes more.
 */
size_t moe_workspace_bytes(const moe_layer_t *layer, int32_t n_max);

/* Zeroes all ws_bytes of the workspace [dev] on stream s.  Library infrastructure: no passage of
 * the pages defines it. */
moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t s);

/*
 * Top-m routing [Lan, §1 "Routing, union and reuse": the router selects a set of m of
 * the N experts for each token; the MoE layer combines the m expert outputs with the
 * router's gate weights].
 *   logits [dev] fp32 [n, N]   router logits of the pass's n tokens.
 *   ids    [dev] int32 [n, m]  out: the m experts with the largest logits, in order of
 *                              descending logit; an equal logit goes to the lower id.
 *   gates  [dev] fp32 [n, m]   out: renorm != 0 -> softmax over the m selected logits
 *                              (the full softmax renormalised over the selected set);
 *                              renorm == 0 -> the full softmax over all N logits.
 * NaN logits are not supported: they rank below every number, and the ids stay distinct
 * and inside [0, N).  Supported: 0 <= n, 1 <= m <= min(N, 32), N <= 1024.
 * n == 0 enqueues nothing.
 */
moe_status_t moe_route_topm(const float *logits, int32_t n, int32_t N, int32_t m, int32_t renorm,
                            int32_t *ids, float *gates, moe_stream_t s);

/*
 * Slot grouping by expert, a counting sort [Lan, §1: a deduplicating kernel groups the
 * pass's tokens by expert; App. E "Engine changes": the deduplicating engine sorts rows by
 * expert].  Slot s = t*m + j names expert ids[s].
 *   ids            [dev] int32 [n*m]
 *   num_distinct   [dev] int32 [1]            out: U, the distinct experts of the pass
 *   expert_list    [dev] int32 [min(N, n*m)]  out: the U distinct ids, ascending
 *   expert_offsets [dev] int32 [min(N, n*m)+1] out: slots of expert_list[u] are
 *                                             slot_order[offsets[u] .. offsets[u+1])
 *   slot_order     [dev] int32 [n*m]          out: slot indices grouped by expert,
 *                                             ascending slot index within an expert
 *   ws             [dev] workspace or NULL.   Ids outside [0, N) are left out of every
 *                                             group; with a workspace they set
 *                                             MOE_ERR_BAD_ID there.
 * Supported: 1 <= n*m <= 4096, N <= 1024.  Entries past U are left unspecified.
 */
moe_status_t moe_group_slots(const int32_t *ids, int32_t n, int32_t m, int32_t N,
                             int32_t *num_distinct, int32_t *expert_list, int32_t *expert_offsets,
                             int32_t *slot_order, void *ws, moe_stream_t s);

/*
 * Per-slot expert operation [Lan, §1: a per-slot kernel multiplies each token by each
 * of its selected experts separately, with one expert read per slot; it requests m*n*w
 * expert bytes per pass], fused with the weighted combine of the MoE layer:
 *   for every slot (t, j), e = ids[t, j]:
 *     h = silu(W_gate[e] x_t) * (W_up[e] x_t),   silu(z) = z / (1 + exp(-z))
 *     y_t += gates[t, j] * W_down[e] h
 *   w_gate, w_up, w_down [dev] layer weights in the layouts of moe_layer_t.
 *   x     [dev] [n, d] in layer->x_dtype.
 *   ids   [dev] int32 [n, m];  gates [dev] fp32 [n, m].
 *   y     [dev] fp32 [n, d]    accumulate == 0: y is overwritten; != 0: added to.
 *   ws    [dev] workspace of ws_bytes >= moe_workspace_bytes(layer, n).
 * Supported: 1 <= n <= MOE_MAX_PASS_TOKENS.  A pass above MOE_PERSLOT_LAUNCH_TOKENS runs as
 * consecutive launches on s of equal size, up to 32 tokens when ws_bytes >= moe_workspace_bytes(layer,
 * min(n, 32)), else up to MOE_PERSLOT_LAUNCH_TOKENS (the per-slot form reads every slot's
 * expert either way; the launches write disjoint rows of y and share ws, which needs only
 * moe_workspace_bytes(layer, MOE_PERSLOT_LAUNCH_TOKENS)).  Each launch is validated
 * before it is enqueued and the first error ends the call; the chunks share the layer and
 * the pointers' alignment, so an argument error is found before the first launch.
 * Summation order inside y is not fixed (results may differ in the last bits between runs).
 */
moe_status_t moe_expert_op_perslot(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                   const void *w_down, const void *x, const int32_t *ids,
                                   const float *gates, int32_t n, int32_t accumulate, float *y,
                                   void *ws, size_t ws_bytes, moe_stream_t s);

/*
 * Deduplicating expert operation [Lan, §1: a deduplicating kernel groups the pass's
 * tokens by expert and reads each distinct expert once; it requests w * X(n) expert bytes
 * for a pass whose slots name X(n) distinct experts], fused with the same combine.  The
 * grouping is the output of moe_group_slots on the same ids (it stays on the device; the
 * host never reads U).  Every distinct expert's weights are streamed from memory once
 * for all of its tokens.
 *   gates [dev] fp32 [n, m];  num_distinct, expert_list, expert_offsets, slot_order [dev]
 *   as written by moe_group_slots for this pass; other arguments as the per-slot call.
 * Shared (always-on) experts run through this call with their own weight block: ids
 * listing all of them for every token, gates of 1 and accumulate = 1.
 */
moe_status_t moe_expert_op_dedup(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                 const void *w_down, const void *x, const float *gates, int32_t n,
                                 const int32_t *num_distinct, const int32_t *expert_list,
                                 const int32_t *expert_offsets, const int32_t *slot_order,
                                 int32_t accumulate, float *y, void *ws, size_t ws_bytes,
                                 moe_stream_t s);

/*
 * The deduplicating form from the slots' ids in one launch: the same result as
 * moe_group_slots followed by moe_expert_op_dedup ([Lan] §1: each distinct expert of the pass
 * read once, its tokens batched), with the grouping (the counting sort on expert id) built
 * inside the kernel, once per CTA in shared memory, instead of by a launch of its own.
 *   Arguments as moe_expert_op_perslot (ids [dev] int32 [n*m] as there).  Ids outside
 *   [0, N) are left out of every group and set MOE_ERR_BAD_ID in the workspace.
 * A pass of more than 256 slots (n*m > 256, e.g. top-8 above 32 tokens) has its grouping built
 * by moe_group_slots into the workspace first (two launches, the same result; the workspace
 * then holds it, see moe_workspace_bytes).
 * Supported: the layers the tensor-core kernel runs (bf16, d a multiple of 128), 1 <= n <=
 * MOE_MAX_PASS_TOKENS; otherwise MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_expert_op_dedup_ids(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                     const void *w_down, const void *x, const int32_t *ids, const float *gates,
                                     int32_t n, int32_t accumulate, float *y, void *ws, size_t ws_bytes,
                                     moe_stream_t s);

/*
 * The per-slot expert operation without a caller workspace.  The paper has no
 * counterpart: this is a service to callers that cannot allocate device memory -- code
 * running under a memory manager that owns every device byte (a serving framework's
 * caching allocator, a fixed arena budgeted ahead of time), where a raw cudaMalloc would
 * bypass its accounting, and code on a latency-critical path, where cudaMalloc and
 * cudaFree synchronise the device.  It allocates nothing and calls no allocating routine.
 *   Arguments and results as moe_expert_op_perslot, without ws/ws_bytes, plus
 *   status_out [dev] int32 [1] or NULL: receives the call's device error word (MOE_OK,
 *   MOE_ERR_BAD_ID or MOE_ERR_DEVICE_TIMEOUT), written on stream s after the kernels.
 * Scratch: a 32 MiB array inside the library, held by every GPU that loads it until the
 * process exits.  A layer or pass whose workspace (moe_workspace_bytes) would exceed it is
 * rejected with MOE_ERR_WORKSPACE.  Every argument is checked first (the same checks and
 * statuses as moe_expert_op_perslot): a rejected call enqueues no device work.  Its error
 * word is cleared at the start of every call,
 * and the array keeps the last call's contents after it.  All calls on a GPU share it, so calls that
 * overlap on that GPU (on different streams, or from different host threads) race: order
 * them on one stream.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current and caches it; make that first call before any stream capture.
 */
moe_status_t moe_expert_op_perslot_noalloc(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                           const void *w_down, const void *x, const int32_t *ids,
                                           const float *gates, int32_t n, int32_t accumulate, float *y,
                                           int32_t *status_out, moe_stream_t s);

/*
 * FP8 expert weights: the fp32 scale of every weight row [dev]: gate [N, f], up [N, f],
 * down [N, d] (value = code * scale; see moe_quantize_rows_e4m3).
 */
typedef struct {
    const float *gate, *up, *down;
} moe_weight_scales_t;

/*
 * The per-slot and the deduplicating expert operation of an e4m3 layer (the quantized
 * experts of [Lan, App. E Table 6], in GB300's FP8 tensor-core format): as
 * moe_expert_op_perslot / moe_expert_op_dedup, with
 *   w_gate, w_up, w_down [dev] e4m3 codes in the layouts of moe_layer_t, scales their row scales;
 *   x [dev] uint8 [n, d] e4m3 codes, x_scale [dev] fp32 [n] the token scales (alignment as
 *   stated at the top: scale arrays 4 bytes).
 * h is rounded to e4m3 as the down projection's operand, with one scale per token and
 * 256-wide block of f (amax / 448; the last block is 128 wide when f % 256 = 128).  layer->w_dtype = layer->x_dtype = MOE_E4M3, d and f
 * multiples of 128; requested bytes per expert w = 3 d f + 4 (2 f + d) (moe_pass_bytes).
 * Returns MOE_ERR_UNSUPPORTED for a layer that is not e4m3.
 */
moe_status_t moe_expert_op_perslot_fp8(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                       const void *w_down, const moe_weight_scales_t *scales, const void *x,
                                       const float *x_scale, const int32_t *ids, const float *gates, int32_t n,
                                       int32_t accumulate, float *y, void *ws, size_t ws_bytes, moe_stream_t s);

moe_status_t moe_expert_op_dedup_fp8(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                     const void *w_down, const moe_weight_scales_t *scales, const void *x,
                                     const float *x_scale, const float *gates, int32_t n, const int32_t *num_distinct,
                                     const int32_t *expert_list, const int32_t *expert_offsets,
                                     const int32_t *slot_order, int32_t accumulate, float *y, void *ws,
                                     size_t ws_bytes, moe_stream_t s);

/* The e4m3 form of moe_expert_op_dedup_ids (scales as moe_expert_op_perslot_fp8). */
moe_status_t moe_expert_op_dedup_ids_fp8(const moe_layer_t *layer, const void *w_gate, const void *w_up,
                                         const void *w_down, const moe_weight_scales_t *scales, const void *x,
                                         const float *x_scale, const int32_t *ids, const float *gates, int32_t n,
                                         int32_t accumulate, float *y, void *ws, size_t ws_bytes, moe_stream_t s);

/*
 * Per-row quantization to e4m3 on the device (the operand format of the _fp8 calls): for each
 * row r of src [rows, cols] (fp32 or bf16 by src_dtype), scale[r] = amax_r / 448 in fp32 (1 if
 * the row is all zero) and q[r][c] = e4m3(src[r][c] / scale[r]), the division in IEEE fp32,
 * rounded to nearest with ties to even and saturated at +-448.
 *   src [dev], q [dev] uint8 [rows, cols], scale [dev] fp32 [rows].  rows == 0 enqueues nothing.
 */
moe_status_t moe_quantize_rows_e4m3(const void *src, int32_t src_dtype, int32_t rows, int32_t cols, uint8_t *q,
                                    float *scale, moe_stream_t s);

/*
 * Requested bytes of one pass [Lan, §1 "Bytes": E_slot = m*n*w, E_dedup = w * X(n);
 * §2 "Effective bandwidth": u_bar(n) = E_dedup / E_slot].  Host only.
 *   ids_host [host] int32 [n*m].
 *   out: expert_bytes w = 3*d*f*sizeof(weight) (+ 4*(2f + d) row-scale bytes for e4m3);
 *        slot_bytes = n*m*w; dedup_bytes = U*w;
 *        act_bytes = n*d*sizeof(x) + n*d*4 (activations read, output written; reported
 *        apart and never part of E_slot, E_dedup or u_bar); U; ubar = U / (n*m).
 * Returns MOE_ERR_BAD_ID if an id is outside [0, N).
 */
typedef struct {
    uint64_t expert_bytes, slot_bytes, dedup_bytes, act_bytes;
    int32_t n, m, U, reserved;
    double ubar;
} moe_pass_bytes_t;

moe_status_t moe_pass_bytes(const moe_layer_t *layer, const int32_t *ids_host, int32_t n,
                            moe_pass_bytes_t *out);

/*
 * Bandwidth report over pass sizes n = n_lo .. n_lo+count-1 [Lan, §2 "Effective
 * bandwidth": beta_p(n) = requested expert bytes of kernel p over its time,
 * r(n) = beta_dedup / beta_slot, u_bar(n) = E_dedup / E_slot; §3.1 eq. (6): the saving
 * S(n) = t_slot(n) - t_dedup(n), and (7): dedup is faster exactly where u_bar < r;
 * §2 "Testing the inputs": the crossover is the smallest n from which the saving stays
 * positive].  Host only; all arrays [host] of length count.
 *   slot_bytes, dedup_bytes  requested bytes summed over the passes timed at each n.
 *   t_slot, t_dedup          the matching summed times (any unit; beta is bytes/unit).
 *   out: beta_slot, beta_dedup, ubar, r, saving; *crossover = the crossover n, or -1.
 */
moe_status_t moe_bandwidth_report(int32_t n_lo, int32_t count, const double *slot_bytes,
                                  const double *dedup_bytes, const double *t_slot,
                                  const double *t_dedup, double *beta_slot, double *beta_dedup,
                                  double *ubar, double *r, double *saving, int32_t *crossover);

/*
 * Expected distinct experts of n tokens under independent uniform routing,
 * N * (1 - q^n) with q = 1 - m/N [Lan, §1, after MoESD].  Host only.
 */
double moe_expected_union(int32_t N, int32_t m, int32_t n);

/*
 * Best draft length under geometric acceptance [Lan, §1 "Speculative decoding": the
 * throughput T_a(k) = G_a(k) / V(k) with G_a(k) = 1 + a + ... + a^k; k*(a) is the
 * smallest maximiser over k = 0..kmax].  V [host] double [kmax+1], the step time of a
 * step that drafts k tokens.  Returns k*, or -1 if a is outside [0, 1) or some V <= 0.
 */
int32_t moe_best_draft_length(const double *V, int32_t kmax, double a);

/*
 * Staircase of a step time [Lan, §3.2 (8)-(9) and App. B.1 (B.4): a0 = V(1)/V(0) - 1 is the
 * acceptance above which one draft beats none; §3.3 and App. B.3 (B.26)-(B.31): alpha_{k,i}
 * = inf {a in [0,1) : T_a(k) > T_a(i)} (1 if empty) and the step points
 * a_j = max_{i<j} min_{k>=j} alpha_{k,i}, so that k*(a) >= j for a in (a_j, 1) and k*(a) < j
 * for a in [0, a_j); (10): with 0 <= c_1 <= ... <= c_kmax, c_i = V(i) - V(i-1), j - 1 and j
 * alone decide whether k*(a) reaches j].  Host only.
 *   V      [host] double [kmax+1], the step time of a step drafting k tokens, all > 0;
 *          1 <= kmax <= 64.
 *   a0     out: V(1)/V(0) - 1 (may be negative, or >= 1).
 *   a_step [host] double [kmax+1] out: a_step[0] = 0, a_step[j] the j-th step point.
 *   alpha  [host] double [(kmax+1)*(kmax+1)] out, or NULL: alpha[k*(kmax+1) + i] for i < k,
 *          0 elsewhere.
 *   convex out: 1 if V is convex and non-decreasing (the hypothesis of (10)), else 0.
 * Returns MOE_ERR_ARG for a NULL output, kmax outside [1, 64] or a V <= 0 or not finite.
 */
moe_status_t moe_staircase(const double *V, int32_t kmax, double *a0, double *a_step, double *alpha,
                           int32_t *convex);

/*
 * Speedup of draft length k over plain decoding [Lan, §3.2 (9)]:
 * T_a(k)/T_a(0) = G_a(k) V(0) / V(k).  Host only; NAN for k outside [0, kmax], a outside
 * [0, 1) or a V <= 0.
 */
double moe_speedup(const double *V, int32_t kmax, int32_t k, double a);

/*
 * Reuse threshold of a deduplicating engine in time [Lan, §3.4 (14), App. B.2 (B.12)-(B.14)]:
 * a draft of length k is faster than plain decoding exactly when the byte-weighted mean reuse
 * rho_bar_k of the k drafted tokens (11) exceeds
 *   rho*_k(a) = 1 - (B_k / (m W k)) [ (G_a(k) - 1) tau(1) - dD_k / beta_D - dphi_k ]
 *                 - (B_k / beta(1) - 1) / k.
 * Host only.  in: mW = m W (expert bytes of a one-token pass), B_k = beta_dedup(k+1),
 * beta_1 = beta(1), tau_1 = tau(1) = V(0), dD_over_betaD = (D(k+1) - D(1)) / beta_D,
 * dphi = phi_dedup(k+1) - phi(1) (any consistent units).  NAN for k < 1, a outside [0, 1),
 * or mW, B_k, beta_1 not > 0.
 */
typedef struct {
    double mW, B_k, beta_1, tau_1, dD_over_betaD, dphi;
} moe_threshold_in_t;

double moe_reuse_threshold(int32_t k, double a, const moe_threshold_in_t *in);

/*
 * The same threshold with one bandwidth and no fixed time [Lan, §3.4 (16), (B.16)]:
 *   rho*_k(a) = 1 - [ (G_a(k) - 1)(D(1) + m W) - (D(k+1) - D(1)) ] / (m W k),
 * D(n) = D + kv(n-1) the bytes read once per pass.  Host only; NAN for k < 1, a outside
 * [0, 1) or mW not > 0.
 */
double moe_reuse_threshold_bytes(int32_t k, double a, double mW, double D_1, double D_k1);

/*
 * Error bounds for a relative bandwidth error |e| <= eps < 1/2 [Lan, §3.5, Table 2, App. C]:
 *   delta         = eps / (1 - eps), the relative error of a predicted step time;
 *   verify_factor = eps / (1 - eps): |tau_hat - tau| <= verify_factor * M_p(n) (17), and
 *                   |S_hat - S| <= verify_factor * (M^e_slot + M^e_dedup) (18);
 *   decision_log_margin = ln((1+eps)/(1-eps)): the predicted and true faster kernel agree
 *                   when |ln r(n) - ln u_bar(n)| exceeds it (19);
 *   regret_factor = (1-delta)/(1+delta): T_a(k_hat*) >= regret_factor * T_a(k*) (20);
 *   speedup_lo, speedup_hi = (1-delta)/(1+delta), (1+delta)/(1-delta): the best predicted
 *                   speedup over the true one (21) ((1+delta)/(1-delta) = 1/(1-2 eps), (C.7)).
 * Host only.  Returns MOE_ERR_ARG for eps outside [0, 1/2) or a NULL out.
 */
typedef struct {
    double delta, verify_factor, decision_log_margin, regret_factor, speedup_lo, speedup_hi;
} moe_error_bounds_t;

moe_status_t moe_error_bounds(double eps, moe_error_bounds_t *out);

/*
 * The separation condition of (20) [Lan, §3.5, Table 2]: with step-time errors within
 * delta, the predicted best draft length equals the true one when
 * (1+delta)/(1-delta) T_a(i) < T_a(k*) for every i != k*.  Host only.  Returns 1 if it holds
 * for V at acceptance a, 0 if not, -1 for bad arguments (as moe_best_draft_length, or
 * delta outside [0, 1)).
 */
int32_t moe_kstar_separated(const double *V, int32_t kmax, double a, double delta);

/*
 * Least-squares fit of one layer's expert-operation time on passes with chosen ids
 * [Lan, §2 "Effective bandwidth", fit (4): t_slot = t_op + c_u U b + c_re (n m - U) b, with
 * c_re / c_u the re-read cost; App. E "Deduplicating fit", (E.1): t_dedup = t_op + c_g U b +
 * c_t n].  Host only.
 *   count          passes (>= 3); n, U [host] int32 [count]: tokens and distinct experts of
 *                  each pass; t [host] double [count]: its (median) operation time.
 *   m, b           experts per token, bytes of one expert of the timed layer.
 *   form           0: per-slot fit (4), coef = {t_op, c_u, c_re};
 *                  1: deduplicating fit (E.1), coef = {t_op, c_g, c_t}.
 *   coef           [host] double [3] out.
 * Returns MOE_ERR_ARG for bad arguments or a design matrix of rank below 3 (e.g. every pass
 * with the same n and U).
 */
moe_status_t moe_fit_op_times(int32_t count, const int32_t *n, const int32_t *U, const double *t, int32_t m,
                              double b, int32_t form, double *coef);

/*
 * Synchronises stream s, reads the device error word of the workspace [dev] into *code
 * (a moe_status_t value; MOE_OK if nothing was recorded) and clears it.  Library
 * infrastructure: no passage of the pages defines it.
 */
moe_status_t moe_last_device_error(void *ws, moe_stream_t s, int32_t *code);

/*
 * Sets, for the expert-operation calls issued after it by this process, how many SM clock
 * cycles one device pipeline wait (a shared-memory barrier, or another CTA's flag) may take
 * before the call gives up: it then records MOE_ERR_DEVICE_TIMEOUT in the workspace's error
 * word, waits (bounded) for its copies and tensor-core operations in flight, frees its
 * tensor memory and returns, leaving the CUDA context usable.  cycles = 0 restores the
 * default, about two seconds at the maximum clock.  A limit shorter than the call's normal
 * waits makes it time out: failure detection is tested this way, without a GPU fault.
 * Library infrastructure: no passage of the pages defines it.  Host only; returns
 * MOE_ERR_ARG for cycles < 0.
 */
moe_status_t moe_set_wait_limit(int64_t cycles);

/*
 * Measurement helper, not part of the method: a read-only streaming probe, the read side of the
 * bandwidth the expert operation is measured against ([Lan] §2 "Effective bandwidth": requested
 * bytes over time, against the memory's bandwidth).  One CTA per SM
 * streams its contiguous share of buf through 1-D TMA bulk copies into shared memory and
 * discards it: floor(bytes / 32768) * 32768 bytes are read.  Time it on the stream to get the
 * read bandwidth the expert kernel's weight stream can reach, beside a copy's (read + write).
 *   buf [dev] 16-byte aligned, bytes >= 32768; ws [dev] a workspace (its error word records a
 *   wait that timed out).  Asynchronous on s.
 */
moe_status_t moe_read_probe(const void *buf, size_t bytes, void *ws, moe_stream_t s);

/* ---------------------------------------------------------------- verify-side neighbours */

/*
 * One round of speculative sampling for B sequences at once ("Lossless but Not Free: An
 * Empirical Anatomy of Speculative Decoding on Consumer Hardware", §3.1 steps 3-4, eqs (1) and
 * (2), Algorithm 1; §3.2 the greedy special case).  For each sequence b, drafts x_1..x_K are
 * accepted while r_i < min(1, p_i(x_i)/q_i(x_i)) (single precision; q_i(x_i) = 0 accepts iff
 * p_i(x_i) > 0; an id outside [0, V) is rejected); a = the number accepted.  The emitted token
 * is drawn with u from p'_{a+1} ~ max(0, p_{a+1} - q_{a+1}) when a < K, from p_{K+1} (the
 * bonus) when a = K; if those weights are all zero, from p_{a+1} itself, and if that is all
 * zero, its argmax.  Greedy (temperature 0): accept iff argmax p_i = x_i, emit argmax p_{a+1}
 * (lowest index among equal maxima); q, r and u are not read.
 * The draw: W(x) = floor(w(x) * 2^46) of each weight clamped to [0, 1], Z = sum W, and the
 * token is the smallest x with W(0) + ... + W(x) > floor(Z * floor(u * 2^24) / 2^24) (exact
 * integer sums: the same token in any summation order).
 *   draft [dev] int32 [B, K]; q [dev] fp32 [B, K, V]; p [dev] fp32 [B, K+1, V] (rows without
 *   NaN); r [dev] fp32 [B, K], u [dev] fp32 [B] uniform draws in [0, 1);
 *   n_accepted [dev] int32 [B] (a), token [dev] int32 [B].  All pointers 4-byte aligned.
 * Supported: 0 <= K <= 31, 1 <= V <= 262144.  B == 0 enqueues nothing.  Asynchronous on s;
 * no workspace.  Reads one row pair per sequence (p and q at the first rejection, or p_{K+1})
 * in sampling mode, the K+1 target rows in greedy mode.
 */
moe_status_t moe_spec_accept(const int32_t *draft, const float *q, const float *p, const float *r, const float *u,
                             int32_t B, int32_t K, int32_t V, int32_t greedy, int32_t *n_accepted, int32_t *token,
                             moe_stream_t s);

/*
 * Expert-union cost of candidate draft subtrees ("SpecFit: Not All Draft Tokens Cost the Same
 * in Offloaded MoE Inference", §3.2 eqs (3)-(5)).  A pool of `nodes` draft nodes (<= 32) plus
 * the root s; for each candidate subset S (a node mask, bit v-1 for node v; bits beyond the
 * pool are ignored):
 *   F(S) = sum_{l < L} |E_{l,s} u U_{v in S} E_{l,v}|,  size = |S|,
 *   R(S) = 1 + sum_{v in S} p_v (summed in node order),  T(S) = bcoef[|S|] + beta * F(S),
 * and *best = the lowest index of the largest R/T (-1 when count == 0).  R, T in double.
 *   bitmaps [dev] uint64 [nodes+1][L][W] (node 0 the root; expert e at bit e % 64 of word e / 64;
 *   (nodes+1)*L*W*8 <= 200 KB); subsets [dev] uint32 [count]; pv [dev] double [nodes];
 *   bcoef [dev] double [nodes+1]; F, size [dev] int32 [count]; R, T [dev] double [count];
 *   best [dev] int32 [1]; ws [dev] of moe_union_cost_workspace_bytes(count) bytes (16-byte
 *   aligned).  Asynchronous on s.
 */
size_t moe_union_cost_workspace_bytes(int32_t count);
moe_status_t moe_union_cost(const uint64_t *bitmaps, int32_t nodes, int32_t L, int32_t W, const uint32_t *subsets,
                            int32_t count, const double *pv, const double *bcoef, double beta, int32_t *F,
                            int32_t *size, double *R, double *T, int32_t *best, void *ws, size_t ws_bytes,
                            moe_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_VERIFY_H */
