/*
 * moe_oracle.c -- plain, slow CPU oracle for the MoE verify-pass expert operation.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file: only the tests, the smoke check of __graft_entry__ and the CPU-baseline leg of
 * bench.py use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Source of every definition: "Speculative Decoding for Mixture-of-Experts Models:
 * Expert Bytes, Kernel Bandwidth and the Best Draft Length" (Lan), cited below as [Lan]
 * with the section, equation or appendix the function follows.
 *
 * Precision: every floating-point value is widened exactly to double (bf16 bits are
 * shifted into the top half of an IEEE single; fp32 widens exactly) and all arithmetic
 * runs in double, one term at a time, in the order the definition is written.
 *
 * dtype codes: 0 = fp32, 1 = bf16 (raw 16-bit patterns).
 *
 * Parity pins (what each function is checked against, in tests/test_oracle_pins.py):
 *   oracle_route_topm        brute-force selection property + scipy softmax, hand cases
 *   oracle_group_slots       numpy stable argsort / bincount
 *   oracle_expert_*          numpy float64 matmul (one SwiGLU FFN), linearity in gates
 *   oracle_pass_bytes        brute-force set union, bounds m <= U <= min(N, nm)
 *   oracle_expected_union    exact enumeration on tiny N, Monte-Carlo on the configs
 *   oracle_union_size        identity (B.5) per window, Python set union
 *   oracle_reuse_estimate    closed form of the synthetic trace law
 *   oracle_best_draft_length the pages' jump example, exact rational brute force
 *   oracle_crossover         hand cases of the definition
 *   oracle_alpha / oracle_step_points / oracle_convex_step_point
 *                            closed forms (k, i) = (1,0), (2,0), (2,1); polynomial roots;
 *                            the brute-force staircase k*(a) on fine grids; the jump example
 *   oracle_reuse_threshold*  the pages' counterexample (rho*_1 = 7/20, rho*_2 = 371/800 and
 *                            its three patterns); identity (B.13); brute-force speedups
 *   oracle_err_*             random perturbations of every bandwidth within the bound
 *   oracle_e4m3_*            every code against torch.float8_e4m3fn; nearest-value search
 *   oracle_quantize_rows_e4m3 the definition: scale = amax/448, codes round to nearest
 *   oracle_expert_op_token_fp8 the fp64 SwiGLU of the dequantized weights within the
 *                            rounding bound of the quantized h (2^-4 relative)
 *   oracle_spec_accept       Proposition 1 of [Anatomy] by exact enumeration of draw grids
 *                            (the emitted token is distributed as p), the one-hot / greedy
 *                            equivalence, the expected yield (1 - a^{K+1})/(1 - a), hand cases
 *   oracle_fx_draw           draw frequencies on a uniform u grid equal the weights' shares
 *   oracle_union_cost        Python set unions per layer, monotone and submodular F,
 *                            brute-force argmax of R/T
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ helpers */

/*
 * Threads of the expert-operation loops (OpenMP over output rows; 1 when built without
 * OpenMP).  Returns the count now in force.
 */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

static double widen(const void *base, int dtype, size_t idx)
{
    if (dtype == 0) {
        return (double)((const float *)base)[idx];
    }
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float v;
    memcpy(&v, &bits, sizeof v);
    return (double)v;
}

static size_t dtype_size(int dtype) { return dtype == 0 ? 4u : 2u; }

/* ------------------------------------------------------------------ routing */

/*
 * Top-m routing [Lan, §1 "Routing, union and reuse": the router selects a set S of m
 * of the N experts for each token].  The m selected experts are the first m of the
 * experts ordered by (logit descending, expert id ascending); ids[t, j] lists them in
 * that order.  Gates are the softmax over the selected logits (renorm != 0), i.e. the
 * full softmax renormalised over S, or the full softmax over all N (renorm == 0).
 * Returns 0, or -1 for bad arguments or a NaN logit.
 */
int oracle_route_topm(const float *logits, int n, int N, int m, int renorm,
                      int32_t *ids, double *gates)
{
    if (n < 0 || N < 1 || m < 1 || m > N) return -1;
    int *order = (int *)malloc(sizeof(int) * (size_t)N);
    if (!order) return -1;
    for (int t = 0; t < n; ++t) {
        const float *z = logits + (size_t)t * N;
        for (int e = 0; e < N; ++e) {
            if (isnan(z[e])) { free(order); return -1; }
            order[e] = e;
        }
        /* insertion sort of expert ids by (logit desc, id asc) */
        for (int a = 1; a < N; ++a) {
            int cur = order[a];
            int b = a - 1;
            while (b >= 0) {
                int prev = order[b];
                int cur_first = (z[cur] > z[prev]) || (z[cur] == z[prev] && cur < prev);
                if (!cur_first) break;
                order[b + 1] = prev;
                --b;
            }
            order[b + 1] = cur;
        }
        double zmax = (double)z[order[0]];
        double denom = 0.0;
        if (renorm) {
            for (int j = 0; j < m; ++j) denom += exp((double)z[order[j]] - zmax);
        } else {
            for (int e = 0; e < N; ++e) denom += exp((double)z[e] - zmax);
        }
        for (int j = 0; j < m; ++j) {
            ids[(size_t)t * m + j] = order[j];
            gates[(size_t)t * m + j] = exp((double)z[order[j]] - zmax) / denom;
        }
    }
    free(order);
    return 0;
}

/* ----------------------------------------------------------------- grouping */

/*
 * Slot grouping by expert [Lan, App. E "Engine changes": the deduplicating MLX engine
 * sorts rows by expert; §1: a deduplicating kernel groups the pass's tokens by expert].
 * Counting sort over the n*m slots (slot s = t*m + j): histogram over N experts,
 * exclusive prefix sum over the non-empty experts in ascending id order, then a stable
 * scatter of slot indices (ascending s within each expert).
 * Outputs: *U = number of distinct experts; expert_list[0..U); offsets[0..U];
 * order[0..n*m).  Returns 0, or -1 if an id is outside [0, N).
 */
int oracle_group_slots(const int32_t *ids, int n, int m, int N, int32_t *U,
                       int32_t *expert_list, int32_t *offsets, int32_t *order)
{
    int S = n * m;
    int32_t *count = (int32_t *)calloc((size_t)N, sizeof(int32_t));
    int32_t *start = (int32_t *)calloc((size_t)N, sizeof(int32_t));
    if (!count || !start) { free(count); free(start); return -1; }
    for (int s = 0; s < S; ++s) {
        if (ids[s] < 0 || ids[s] >= N) { free(count); free(start); return -1; }
        count[ids[s]] += 1;
    }
    int u = 0, acc = 0;
    for (int e = 0; e < N; ++e) {
        if (count[e] == 0) continue;
        expert_list[u] = e;
        offsets[u] = acc;
        start[e] = acc;
        acc += count[e];
        ++u;
    }
    offsets[u] = acc;
    for (int s = 0; s < S; ++s) {
        int e = ids[s];
        order[start[e]] = s;
        start[e] += 1;
    }
    *U = u;
    free(count);
    free(start);
    return 0;
}

/* --------------------------------------------------------- one expert, one token */

/*
 * The expert operation for one (token, expert) pair [Lan, §1: the gate, up and down
 * projections of a token with the weights of a selected expert], as a SwiGLU:
 *   g = W_gate[e] x,  u = W_up[e] x  (f values each),
 *   h_i = silu(g_i) * u_i with silu(z) = z / (1 + exp(-z)),
 *   out = W_down[e] h  (d values).
 * Layouts (row-major): W_gate, W_up [N, f, d]; W_down [N, d, f]; x [n, d].
 */
static void swiglu_expert(int d, int f, int wdt, int xdt, const void *wg, const void *wu,
                          const void *wd, const void *x, int t, int e, double *h, double *out)
{
    size_t wbase_gu = (size_t)e * (size_t)f * (size_t)d;
    size_t wbase_d = (size_t)e * (size_t)d * (size_t)f;
    size_t xbase = (size_t)t * (size_t)d;
    /* Output rows are independent and each is summed by one thread in k (or i) order, so
     * the thread count (oracle_set_threads) never changes a result bit. */
    #pragma omp parallel for schedule(static)
    for (int i = 0; i < f; ++i) {
        double g = 0.0, u = 0.0;
        for (int k = 0; k < d; ++k) {
            double xv = widen(x, xdt, xbase + (size_t)k);
            g += widen(wg, wdt, wbase_gu + (size_t)i * d + k) * xv;
            u += widen(wu, wdt, wbase_gu + (size_t)i * d + k) * xv;
        }
        h[i] = g / (1.0 + exp(-g)) * u;
    }
    #pragma omp parallel for schedule(static)
    for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int i = 0; i < f; ++i) acc += widen(wd, wdt, wbase_d + (size_t)o * f + i) * h[i];
        out[o] = acc;
    }
}

/*
 * Per-slot expert operation [Lan, §1: a per-slot kernel multiplies each token by each
 * of its selected experts separately, one expert read per slot], followed by the
 * weighted combine of the MoE layer: y_t = sum_{j ascending} gates[t,j] * E_{ids[t,j]}(x_t).
 * y is [n, d] in double.  Returns 0, or -1 for an id outside [0, N).
 */
int oracle_expert_op_perslot(int d, int f, int N, int m, int wdt, int xdt, const void *wg,
                             const void *wu, const void *wd, const void *x, const int32_t *ids,
                             const double *gates, int n, double *y)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
    double *ys = (double *)malloc(sizeof(double) * (size_t)d);
    if (!h || !ys) { free(h); free(ys); return -1; }
    for (size_t i = 0; i < (size_t)n * d; ++i) y[i] = 0.0;
    for (int t = 0; t < n; ++t) {
        for (int j = 0; j < m; ++j) {
            int e = ids[(size_t)t * m + j];
            if (e < 0 || e >= N) { free(h); free(ys); return -1; }
            swiglu_expert(d, f, wdt, xdt, wg, wu, wd, x, t, e, h, ys);
            double gate = gates[(size_t)t * m + j];
            for (int o = 0; o < d; ++o) y[(size_t)t * d + o] += gate * ys[o];
        }
    }
    free(h);
    free(ys);
    return 0;
}

/*
 * Deduplicating expert operation [Lan, §1: a deduplicating kernel groups the pass's
 * tokens by expert and reads each distinct expert once].  Loops expert-major over the
 * grouping (expert_list, offsets, order); each slot's product is kept, then the same
 * combine as the per-slot form runs in (t, j ascending) order, so the two forms give
 * bit-identical results here.
 */
int oracle_expert_op_dedup(int d, int f, int N, int m, int wdt, int xdt, const void *wg,
                           const void *wu, const void *wd, const void *x, const double *gates,
                           int n, int U, const int32_t *expert_list, const int32_t *offsets,
                           const int32_t *order, double *y)
{
    size_t S = (size_t)n * m;
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
    double *ys = (double *)calloc(S * (size_t)d, sizeof(double));
    if (!h || !ys) { free(h); free(ys); return -1; }
    for (int u = 0; u < U; ++u) {
        int e = expert_list[u];
        if (e < 0 || e >= N) { free(h); free(ys); return -1; }
        for (int p = offsets[u]; p < offsets[u + 1]; ++p) {
            int s = order[p];
            int t = s / m;
            swiglu_expert(d, f, wdt, xdt, wg, wu, wd, x, t, e, h, ys + (size_t)s * d);
        }
    }
    for (size_t i = 0; i < (size_t)n * d; ++i) y[i] = 0.0;
    for (int t = 0; t < n; ++t)
        for (int j = 0; j < m; ++j) {
            size_t s = (size_t)t * m + j;
            for (int o = 0; o < d; ++o) y[(size_t)t * d + o] += gates[s] * ys[s * d + o];
        }
    free(h);
    free(ys);
    return 0;
}

/*
 * The layer output for one token only (all its m experts, combined), for spot checks
 * of large passes: the same arithmetic as oracle_expert_op_perslot restricted to t.
 */
int oracle_expert_op_token(int d, int f, int N, int m, int wdt, int xdt, const void *wg,
                           const void *wu, const void *wd, const void *x, const int32_t *ids,
                           const double *gates, int t, double *y_t)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
    double *ys = (double *)malloc(sizeof(double) * (size_t)d);
    if (!h || !ys) { free(h); free(ys); return -1; }
    for (int o = 0; o < d; ++o) y_t[o] = 0.0;
    for (int j = 0; j < m; ++j) {
        int e = ids[(size_t)t * m + j];
        if (e < 0 || e >= N) { free(h); free(ys); return -1; }
        swiglu_expert(d, f, wdt, xdt, wg, wu, wd, x, t, e, h, ys);
        for (int o = 0; o < d; ++o) y_t[o] += gates[(size_t)t * m + j] * ys[o];
    }
    free(h);
    free(ys);
    return 0;
}

/* --------------------------------------------------------------------- bytes */

/*
 * Requested expert bytes of one pass [Lan, §1 "Bytes": a per-slot kernel requests m*n*w,
 * one request per slot; a deduplicating kernel requests w * X(n), X(n) the number of
 * distinct experts of the pass; §2: u_bar(n) = E_dedup / E_slot].
 * w = 3*d*f*sizeof(weight).  out[0..3] = {w, slot_bytes, dedup_bytes, act_bytes} where
 * act_bytes = x read (n*d*sizeof(x)) + y written (n*d*4); *U_out = distinct experts;
 * *ubar = U / (n*m).  Returns 0, or -1 for an id outside [0, N).
 */
int oracle_pass_bytes(int d, int f, int N, int m, int wdt, int xdt, const int32_t *ids, int n,
                      uint64_t *out, int32_t *U_out, double *ubar)
{
    unsigned char *seen = (unsigned char *)calloc((size_t)N, 1);
    if (!seen) return -1;
    int U = 0;
    for (int s = 0; s < n * m; ++s) {
        if (ids[s] < 0 || ids[s] >= N) { free(seen); return -1; }
        if (!seen[ids[s]]) { seen[ids[s]] = 1; ++U; }
    }
    free(seen);
    /* dtype 2 = e4m3: one byte per weight, plus the fp32 scale of each of the expert's
     * 2f + d rows; the activations add their n fp32 token scales */
    uint64_t wb = wdt == 2 ? 1u : (uint64_t)dtype_size(wdt);
    uint64_t xb = xdt == 2 ? 1u : (uint64_t)dtype_size(xdt);
    uint64_t w = 3ull * (uint64_t)d * (uint64_t)f * wb + (wdt == 2 ? 4ull * (2ull * f + d) : 0ull);
    out[0] = w;
    out[1] = (uint64_t)n * (uint64_t)m * w;
    out[2] = (uint64_t)U * w;
    out[3] = (uint64_t)n * (uint64_t)d * xb + (uint64_t)n * (uint64_t)d * 4ull + (xdt == 2 ? 4ull * n : 0ull);
    *U_out = U;
    *ubar = (n * m) > 0 ? (double)U / (double)(n * m) : 0.0;
    return 0;
}

/* ------------------------------------------------------- union and reuse on traces */

/*
 * X_t(n) = |S_t u ... u S_{t+n-1}| [Lan, §1 "Routing, union and reuse"] on a trace
 * sets[T, m] of expert ids.  Returns the count, or -1 for bad arguments.
 */
int oracle_union_size(const int32_t *sets, int T, int m, int N, int t0, int n)
{
    if (t0 < 0 || n < 0 || t0 + n > T) return -1;
    unsigned char *seen = (unsigned char *)calloc((size_t)N, 1);
    if (!seen) return -1;
    int X = 0;
    for (int t = t0; t < t0 + n; ++t)
        for (int j = 0; j < m; ++j) {
            int e = sets[(size_t)t * m + j];
            if (e < 0 || e >= N) { free(seen); return -1; }
            if (!seen[e]) { seen[e] = 1; ++X; }
        }
    free(seen);
    return X;
}

/*
 * Reuse estimate rho_hat(n) [Lan, eq. (1) and App. D.2 "Models and prompts"]: over every
 * window of n consecutive tokens of the trace, count the last token's experts that an
 * earlier token of the window also selected; divide the sum by m times the number of
 * windows.  rho_hat(1) = 0.  Returns -1.0 for bad arguments.
 */
double oracle_reuse_estimate(const int32_t *sets, int T, int m, int N, int n)
{
    if (n < 1 || n > T) return -1.0;
    unsigned char *seen = (unsigned char *)calloc((size_t)N, 1);
    if (!seen) return -1.0;
    double hits = 0.0;
    int windows = 0;
    for (int t0 = 0; t0 + n <= T; ++t0) {
        memset(seen, 0, (size_t)N);
        for (int t = t0; t < t0 + n - 1; ++t)
            for (int j = 0; j < m; ++j) seen[sets[(size_t)t * m + j]] = 1;
        const int32_t *last = sets + (size_t)(t0 + n - 1) * m;
        for (int j = 0; j < m; ++j) hits += seen[last[j]] ? 1.0 : 0.0;
        ++windows;
    }
    free(seen);
    return hits / ((double)m * (double)windows);
}

/* ----------------------------------------------------------------- report math */

/*
 * Expected distinct experts of n tokens under independent uniform routing,
 * N (1 - q^n) with q = 1 - m/N [Lan, §1, citing MoESD].
 */
double oracle_expected_union(int N, int m, int n)
{
    double q = 1.0 - (double)m / (double)N;
    return (double)N * (1.0 - pow(q, (double)n));
}

/* G_a(k) = 1 + a + ... + a^k, the expected tokens a step emits [Lan, §1 "Speculative decoding"]. */
double oracle_expected_tokens(double a, int k)
{
    double g = 0.0, p = 1.0;
    for (int i = 0; i <= k; ++i) { g += p; p *= a; }
    return g;
}

/*
 * Best draft length k*(a) [Lan, §1: the smallest maximiser over k in {0..kmax} of the
 * throughput T_a(k) = G_a(k) / V(k), V(k) the step time].  Comparison is strict, so the
 * first (smallest) maximiser wins.  Returns -1 if some V(k) <= 0.
 */
int oracle_best_draft_length(const double *V, int kmax, double a)
{
    int best = -1;
    double best_T = 0.0;
    for (int k = 0; k <= kmax; ++k) {
        if (!(V[k] > 0.0)) return -1;
        double T = oracle_expected_tokens(a, k) / V[k];
        if (best < 0 || T > best_T) { best = k; best_T = T; }
    }
    return best;
}

/*
 * Crossover [Lan, §2 "Testing the inputs": the smallest pass size from which the
 * measured saving S(n) = t_slot(n) - t_dedup(n) stays positive].  t_slot and t_dedup
 * are indexed by n - n_lo for n in [n_lo, n_hi].  Returns the crossover n, or -1 when
 * S(n_hi) <= 0 (no pass size in range from which the saving stays positive).
 */
int oracle_crossover(const double *t_slot, const double *t_dedup, int n_lo, int n_hi)
{
    int ans = -1;
    for (int n = n_hi; n >= n_lo; --n) {
        double S = t_slot[n - n_lo] - t_dedup[n - n_lo];
        if (S > 0.0) ans = n;
        else break;
    }
    return ans;
}

/*
 * Bandwidth report [Lan, §2 "Effective bandwidth": beta_p(n) = requested expert bytes of
 * kernel p over its time; r(n) = beta_dedup / beta_slot; u_bar(n) = E_dedup / E_slot;
 * §3.1: the saving S(n) = tau_slot(n) - tau_dedup(n)].  Arrays of length count for
 * n = n_lo .. n_lo+count-1; *cross = oracle_crossover over the same range.
 */
int oracle_bandwidth_report(int n_lo, int count, const double *slot_bytes,
                            const double *dedup_bytes, const double *t_slot,
                            const double *t_dedup, double *beta_slot, double *beta_dedup,
                            double *ubar, double *r, double *saving, int *cross)
{
    for (int i = 0; i < count; ++i) {
        if (!(t_slot[i] > 0.0) || !(t_dedup[i] > 0.0) || !(slot_bytes[i] > 0.0)) return -1;
        beta_slot[i] = slot_bytes[i] / t_slot[i];
        beta_dedup[i] = dedup_bytes[i] / t_dedup[i];
        ubar[i] = dedup_bytes[i] / slot_bytes[i];
        r[i] = beta_dedup[i] / beta_slot[i];
        saving[i] = t_slot[i] - t_dedup[i];
    }
    *cross = oracle_crossover(t_slot, t_dedup, n_lo, n_lo + count - 1);
    return 0;
}

/* ------------------------------------------------------------------ step-time theory */

/* T_a(k) = G_a(k) / V(k), the throughput of draft length k [Lan, §1 "Speculative decoding"]. */
double oracle_throughput(const double *V, int k, double a)
{
    return oracle_expected_tokens(a, k) / V[k];
}

/*
 * a0 = V(1)/V(0) - 1 [Lan, §3.2 and App. B.1 (B.4)]: one draft is faster than none exactly
 * when a > a0.
 */
double oracle_first_threshold(const double *V)
{
    return V[1] / V[0] - 1.0;
}

/* The speedup T_a(k)/T_a(0) = G_a(k) V(0) / V(k) [Lan, §3.2 (9)]. */
double oracle_speedup(const double *V, int k, double a)
{
    return oracle_throughput(V, k, a) / oracle_throughput(V, 0, a);
}

/*
 * alpha_{k,i} [Lan, App. B.3]: the infimum of J_{k,i} = {a in [0,1) : T_a(k) > T_a(i)},
 * taken as 1 when J_{k,i} is empty (0 <= i < k).  J_{k,i} is closed upward in [0,1)
 * ((B.26)-(B.27)): G_a(k)/G_a(i) rises with a from 1 at a = 0 towards (k+1)/(i+1) as
 * a -> 1.  So: if T_0(k) > T_0(i) the infimum is 0; if (k+1)/(i+1) <= V(k)/V(i) no a < 1
 * qualifies and the value is 1; otherwise the boundary is found by halving an interval
 * [lo, hi] with lo outside and hi inside J_{k,i}, testing T_a(k) > T_a(i) directly.
 */
/*
 * T_a(k) > T_a(i) for i < k, multiplied through by V(k) V(i) > 0 and with G_a(k) split as
 * G_a(i) + a^{i+1} + ... + a^k: V(i) (a^{i+1} + ... + a^k) > G_a(i) (V(k) - V(i)).  The
 * same inequality, without the cancellation of comparing two nearly equal throughputs.
 */
static int oracle_faster(const double *V, int k, int i, double a)
{
    double tail = 0.0, p = 1.0;
    for (int s = 0; s <= k; ++s) {
        if (s > i) tail += p;
        p *= a;
    }
    return V[i] * tail > oracle_expected_tokens(a, i) * (V[k] - V[i]) ? 1 : 0;
}

double oracle_alpha(const double *V, int k, int i)
{
    if (oracle_faster(V, k, i, 0.0)) return 0.0;
    if ((double)(k + 1) * V[i] <= (double)(i + 1) * V[k]) return 1.0;
    double lo = 0.0, hi = 1.0;
    for (int it = 0; it < 200; ++it) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (oracle_faster(V, k, i, mid)) hi = mid;
        else lo = mid;
    }
    return hi;
}

/*
 * Step points a_j = max over i < j of min over k >= j of alpha_{k,i}, j = 1..kmax
 * [Lan, §3.3 and App. B.3 (B.31)]: k*(a) >= j for every a in (a_j, 1) and k*(a) < j for
 * every a in [0, a_j).  a_step[0] = 0.  Returns 0, or -1 if kmax < 1 or some V <= 0.
 */
int oracle_step_points(const double *V, int kmax, double *a_step)
{
    if (kmax < 1) return -1;
    for (int k = 0; k <= kmax; ++k)
        if (!(V[k] > 0.0)) return -1;
    a_step[0] = 0.0;
    for (int j = 1; j <= kmax; ++j) {
        double mx = 0.0;
        for (int i = 0; i < j; ++i) {
            double mn = 1.0;
            for (int k = j; k <= kmax; ++k) {
                double al = oracle_alpha(V, k, i);
                if (al < mn) mn = al;
            }
            if (i == 0 || mn > mx) mx = mn;
        }
        a_step[j] = mx;
    }
    return 0;
}

/*
 * Convex and non-decreasing step time [Lan, §3.3 (10)]: c_i = V(i) - V(i-1) with
 * 0 <= c_1 <= c_2 <= ... <= c_kmax.  Returns 1 if so, else 0.
 */
int oracle_convex_nondecreasing(const double *V, int kmax)
{
    double prev = 0.0;
    for (int i = 1; i <= kmax; ++i) {
        double c = V[i] - V[i - 1];
        if (c < prev) return 0;
        prev = c;
    }
    return 1;
}

/*
 * The step point a_j of a convex non-decreasing step time [Lan, App. B.3 (B.36)]:
 * a_j = inf {a in [0,1) : h_j(a) > c_j / V(j-1)} with h_j(a) = a^j / G_a(j-1), strictly
 * increasing on [0,1); a_1 = min(c_1/V(0), 1).  The infimum is found by halving, testing
 * the defining inequality a^j V(j-1) > G_a(j-1) c_j of (10).  Returns 1 when the set is
 * empty (h_j never exceeds the bound below a = 1).
 */
double oracle_convex_step_point(const double *V, int j)
{
    double c = V[j] - V[j - 1];
    if (j == 1) {
        double v = c / V[0];
        return v < 1.0 ? v : 1.0;
    }
    /* at a = 0 the left side is 0 and never exceeds a non-negative right side */
    double hi_lim = 1.0, lo = 0.0, hi = 1.0;
    /* as a -> 1, a^j V(j-1) -> V(j-1) and G_a(j-1) c_j -> j c_j */
    if (V[j - 1] <= (double)j * c) return hi_lim;
    for (int it = 0; it < 200; ++it) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (pow(mid, (double)j) * V[j - 1] > oracle_expected_tokens(mid, j - 1) * c) hi = mid;
        else lo = mid;
    }
    return hi;
}

/*
 * Byte-weighted mean reuse of the k drafted tokens [Lan, §3.4 (11)]:
 * rho_bar_k = (1/(k W)) sum_{j=2}^{k+1} sum_l w_l rho_l(j), W = sum_l w_l.
 * rho [L][jmax+1] row-major (rho[l][j] for j = 0..jmax), w [L].  Requires k+1 <= jmax.
 */
double oracle_mean_reuse(int L, const double *w, const double *rho, int jmax, int k)
{
    double W = 0.0, acc = 0.0;
    for (int l = 0; l < L; ++l) W += w[l];
    for (int j = 2; j <= k + 1; ++j)
        for (int l = 0; l < L; ++l) acc += w[l] * rho[l * (jmax + 1) + j];
    return acc / ((double)k * W);
}

/*
 * Reuse threshold in time [Lan, §3.4 (14), App. B.2 (B.12)-(B.14)]:
 *   rho*_k(a) = 1 - (1/k) [ B_k Y / (m W) + B_k / beta(1) - 1 ],
 *   Y = (G_a(k) - 1) tau(1) - dD_k / beta_D - dphi_k,
 * the bracket of (14) written out; a draft of length k is faster than plain decoding
 * exactly when rho_bar_k > rho*_k(a).
 *   mW = m W, Bk = beta_dedup(k+1), beta1 = beta(1), tau1 = tau(1),
 *   dD_bD = (D(k+1) - D(1)) / beta_D, dphi = phi_dedup(k+1) - phi(1).
 */
double oracle_reuse_threshold(int k, double a, double mW, double Bk, double beta1, double tau1,
                              double dD_bD, double dphi)
{
    double Y = (oracle_expected_tokens(a, k) - 1.0) * tau1 - dD_bD - dphi;
    return 1.0 - (Bk * Y / mW + Bk / beta1 - 1.0) / (double)k;
}

/*
 * Reuse threshold in bytes, one bandwidth and t0 = phi = 0 [Lan, §3.4 (16), (B.16)]:
 *   rho*_k(a) = 1 - [ (G_a(k) - 1)(D(1) + m W) - (D(k+1) - D(1)) ] / (m W k).
 */
double oracle_reuse_threshold_bytes(int k, double a, double mW, double D1, double Dk1)
{
    return 1.0 - ((oracle_expected_tokens(a, k) - 1.0) * (D1 + mW) - (Dk1 - D1)) / (mW * (double)k);
}

/*
 * Error bounds [Lan, §3.5, Table 2, App. C], for a relative bandwidth error |e| <= eps < 1
 * (each bandwidth estimated as beta (1 + e)), and delta = eps / (1 - eps) for the step time.
 */
/* (17): |tau_hat - tau| <= eps/(1-eps) M_p(n); returns the factor eps/(1-eps). */
double oracle_err_verify_factor(double eps) { return eps / (1.0 - eps); }

/* (18): |S_hat - S| <= eps/(1-eps) (M^e_slot + M^e_dedup). */
double oracle_err_saving_bound(double eps, double Me_slot, double Me_dedup)
{
    return eps / (1.0 - eps) * (Me_slot + Me_dedup);
}

/* (19): the predicted and the true faster kernel agree if |ln r - ln u_bar| > ln((1+eps)/(1-eps)). */
int oracle_err_decision_agrees(double r, double ubar, double eps)
{
    return fabs(log(r) - log(ubar)) > log((1.0 + eps) / (1.0 - eps)) ? 1 : 0;
}

/* (20): T_a(k_hat*) >= (1-delta)/(1+delta) T_a(k*); returns (1-delta)/(1+delta). */
double oracle_err_regret_factor(double delta) { return (1.0 - delta) / (1.0 + delta); }

/*
 * (20) separation: k_hat* = k* if (1+delta)/(1-delta) T_a(i) < T_a(k*) for every i != k*.
 * Returns 1 if the separation holds for step time V at acceptance a, else 0.
 */
int oracle_err_kstar_separated(const double *V, int kmax, double a, double delta)
{
    int ks = oracle_best_draft_length(V, kmax, a);
    if (ks < 0) return 0;
    double Tk = oracle_throughput(V, ks, a);
    for (int i = 0; i <= kmax; ++i) {
        if (i == ks) continue;
        if (!((1.0 + delta) / (1.0 - delta) * oracle_throughput(V, i, a) < Tk)) return 0;
    }
    return 1;
}

/* (21): the best predicted speedup lies in [(1-delta)/(1+delta), (1+delta)/(1-delta)] times the true one. */
void oracle_err_speedup_interval(double delta, double *lo, double *hi)
{
    *lo = (1.0 - delta) / (1.0 + delta);
    *hi = (1.0 + delta) / (1.0 - delta);
}

/* ------------------------------------------------------------------ FP8 (e4m3) experts */

/*
 * OCP FP8 E4M3 ("FN": no infinities): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits.  Exponent 0: subnormal, m * 2^-9.  Exponent 1..15: 2^(e-7) (1 + m/8), except
 * exponent 15 with mantissa 7, which is NaN.  Largest finite value 448.
 */
double oracle_e4m3_decode(uint8_t c)
{
    int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = (double)m * ldexp(1.0, -9);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/*
 * The e4m3 code nearest to v: a search over every finite code, ties to the even mantissa
 * (the code with the lower mantissa bit clear); |v| above 448 saturates to +-448 (the
 * saturating conversion).  v must not be NaN.
 */
uint8_t oracle_e4m3_encode(double v)
{
    int sgn = v < 0.0 || (v == 0.0 && signbit(v));
    double a = fabs(v);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 127; ++c) {   /* codes 0..126: +0 .. 448, 127 is NaN */
        double d = fabs(oracle_e4m3_decode((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = c; }
    }
    return (uint8_t)(best | (sgn << 7));
}

/*
 * Per-row quantization to e4m3 (the format the tensor-core FP8 path reads): for each row,
 * amax = max |v|, scale = amax / 448 in fp32 (1 when amax = 0), codes = e4m3(v / scale)
 * with the division in fp32.  The division and the scale are taken in the kernel's
 * precision, fp32, because they decide integer codes.
 *   src [rows, cols] fp32 (dtype 0) or bf16 bits (dtype 1); q [rows, cols]; scale [rows].
 */
int oracle_quantize_rows_e4m3(const void *src, int dtype, int rows, int cols, uint8_t *q, float *scale)
{
    for (int r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) {
            float v = (float)widen(src, dtype, (size_t)r * cols + c);
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[r] = sc;
        for (int c = 0; c < cols; ++c) {
            float v = (float)widen(src, dtype, (size_t)r * cols + c);
            q[(size_t)r * cols + c] = oracle_e4m3_encode((double)(v / sc));
        }
    }
    return 0;
}

/*
 * The expert operation of one token with e4m3 weights and activations (the quantized
 * experts of [Lan], App. E Table 6, on GB300's FP8 format).  For each of token t's m
 * experts e:
 *   g_i = sg[e][i] sx[t] sum_k W_g[e][i][k] x[t][k],  u_i the same with W_u, sigma = silu;
 *   h_i = silu(g_i) u_i, quantized per block of 128 consecutive i: s_b = amax_b / 448 in
 *   fp32, h~_i = e4m3(h_i / s_b) s_b (the down projection's operand);
 *   y_t[o] += gates[t][j] sd[e][o] sum_i W_d[e][o][i] h~_i.
 * W_g, W_u [N][f][d], W_d [N][d][f] e4m3 codes; sg, su [N][f], sd [N][d] fp32; x [n][d]
 * codes, sx [n].  f must be a multiple of 128.  Returns 0, or -1 for bad arguments.
 */
int oracle_expert_op_token_fp8(int d, int f, int N, int m, const uint8_t *wg, const uint8_t *wu,
                               const uint8_t *wd, const float *sg, const float *su, const float *sd,
                               const uint8_t *x, const float *sx, const int32_t *ids, const double *gates,
                               int t, double *y_t)
{
    if (f % 128 != 0) return -1;
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
    double *hq = (double *)malloc(sizeof(double) * (size_t)f);
    if (!h || !hq) { free(h); free(hq); return -1; }
    for (int o = 0; o < d; ++o) y_t[o] = 0.0;
    for (int j = 0; j < m; ++j) {
        int e = ids[(size_t)t * m + j];
        if (e < 0 || e >= N) { free(h); free(hq); return -1; }
        for (int i = 0; i < f; ++i) {
            double g = 0.0, u = 0.0;
            for (int k = 0; k < d; ++k) {
                double xv = oracle_e4m3_decode(x[(size_t)t * d + k]);
                g += oracle_e4m3_decode(wg[((size_t)e * f + i) * d + k]) * xv;
                u += oracle_e4m3_decode(wu[((size_t)e * f + i) * d + k]) * xv;
            }
            g *= (double)sg[(size_t)e * f + i] * (double)sx[t];
            u *= (double)su[(size_t)e * f + i] * (double)sx[t];
            h[i] = g / (1.0 + exp(-g)) * u;
        }
        /* h rounded to e4m3 per span of 256 columns of f (the last one 128 when f is not a
         * multiple of 256), one scale amax / 448 per token and span */
        for (int b0 = 0; b0 < f; b0 += 256) {
            const int b1 = b0 + 256 < f ? b0 + 256 : f;
            float amax = 0.0f;
            for (int i = b0; i < b1; ++i)
                if (fabsf((float)h[i]) > amax) amax = fabsf((float)h[i]);
            float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            for (int i = b0; i < b1; ++i)
                hq[i] = oracle_e4m3_decode(oracle_e4m3_encode((double)((float)h[i] / sc))) * (double)sc;
        }
        for (int o = 0; o < d; ++o) {
            double acc = 0.0;
            for (int i = 0; i < f; ++i) acc += oracle_e4m3_decode(wd[((size_t)e * d + o) * f + i]) * hq[i];
            y_t[o] += gates[(size_t)t * m + j] * (double)sd[(size_t)e * d + o] * acc;
        }
    }
    free(h);
    free(hq);
    return 0;
}

/* ================================================================ verify-side neighbours
 *
 * Speculative sampling: "Lossless but Not Free: An Empirical Anatomy of Speculative
 * Decoding on Consumer Hardware", cited as [Anatomy]: §3.1 steps 3-4 (the accept test, eq.
 * (1); the adjusted resample, eq. (2); the bonus token; Algorithm 1) and the greedy special
 * case of §3.2.  The uniform draws r_i and u are inputs.  Single-precision arithmetic where
 * the page fixes it ("sampling arithmetic is CPU float32"): the ratio p/q and its minimum
 * with 1, and p - q.
 *
 * Reading for the draw from a distribution over V tokens: every weight w (clamped to [0, 1])
 * becomes the integer W = floor(w * 2^46), Z = the exact sum of the W, and the drawn token is
 * the smallest x whose running sum W(0) + ... + W(x) exceeds t = floor(Z * U / 2^24) with
 * U = floor(u * 2^24).  Integer sums make the index independent of the summation order; each
 * weight moves by less than 2^-46.
 */

static uint64_t fx_weight(float w)
{
    if (!(w > 0.0f)) return 0;                 /* zero, negative or NaN */
    if (w >= 1.0f) return (uint64_t)1 << 46;
    return (uint64_t)((double)w * 70368744177664.0);   /* exact product, truncated */
}

static uint32_t fx_u24(float u)
{
    if (!(u > 0.0f)) return 0;
    if (u >= 1.0f) return (1u << 24) - 1u;
    return (uint32_t)((double)u * 16777216.0);
}

/* The inverse-CDF draw above; -1 when every weight is zero. */
static int32_t fx_draw(const uint64_t *W, int V, float u)
{
    uint64_t Z = 0;
    for (int x = 0; x < V; ++x) Z += W[x];
    if (Z == 0) return -1;
    __extension__ unsigned __int128 prod = (unsigned __int128)Z * fx_u24(u);
    const uint64_t t = (uint64_t)(prod >> 24);
    uint64_t c = 0;
    for (int x = 0; x < V; ++x) {
        c += W[x];
        if (c > t) return x;
    }
    return V - 1;   /* not reached: t < Z */
}

/* Lowest index of the largest value (a NaN never wins). */
static int32_t argmax_row(const float *row, int V)
{
    int32_t best = 0;
    for (int x = 1; x < V; ++x)
        if (row[x] > row[best]) best = x;
    return best;
}

/* The accept test of eq. (1): r < min(1, p(x)/q(x)) in single precision.  Reading for
 * q(x) = 0 (a draft never samples such a token): accept iff p(x) > 0. */
static int accept_draft(float px, float qx, float r)
{
    if (qx > 0.0f) {
        const float ratio = px / qx;
        const float thr = ratio < 1.0f ? ratio : 1.0f;
        return r < thr;
    }
    return px > 0.0f;
}

/* One round of Algorithm 1 for each of B sequences.  draft [B, K] token ids x_1..x_K;
 * q [B, K, V] the draft's distributions q_1..q_K; p [B, K+1, V] the target's p_1..p_{K+1};
 * r [B, K] and u [B] uniform draws (ignored when greedy).  Out: n_acc[b] = a, the number of
 * leading accepted drafts, and token[b] = the emitted token: a draw from p'_{a+1} of eq. (2)
 * when a < K, the bonus draw from p_{K+1} when a = K.  Greedy (temperature 0): accept iff
 * argmax p_i = x_i, and emit argmax p_{a+1}.  Readings: a draft id outside [0, V) is
 * rejected; when the adjusted weights of eq. (2) are all zero the draw falls back to the
 * target row p_{a+1} itself, and when that is all zero too, to its argmax. */
int oracle_spec_accept(const int32_t *draft, const float *q, const float *p, const float *r, const float *u,
                       int B, int K, int V, int greedy, int32_t *n_acc, int32_t *token)
{
    if (B < 0 || K < 0 || V < 1) return -1;
    uint64_t *W = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
    if (W == NULL) return -1;
    for (int b = 0; b < B; ++b) {
        int a = 0;
        for (; a < K; ++a) {
            const int32_t x = draft[(size_t)b * K + a];
            const float *pa = p + ((size_t)b * (K + 1) + a) * V;
            if (x < 0 || x >= V) break;
            if (greedy) {
                if (argmax_row(pa, V) != x) break;
            } else {
                const float *qa = q + ((size_t)b * K + a) * V;
                if (!accept_draft(pa[x], qa[x], r[(size_t)b * K + a])) break;
            }
        }
        const float *prow = p + ((size_t)b * (K + 1) + a) * V;
        int32_t y;
        if (greedy) {
            y = argmax_row(prow, V);
        } else {
            if (a < K) {
                const float *qrow = q + ((size_t)b * K + a) * V;
                for (int x = 0; x < V; ++x) {
                    const float dlt = prow[x] - qrow[x];
                    W[x] = fx_weight(dlt > 0.0f ? dlt : 0.0f);
                }
                y = fx_draw(W, V, u[b]);
            } else {
                y = -1;
            }
            if (y < 0) {
                for (int x = 0; x < V; ++x) W[x] = fx_weight(prow[x]);
                y = fx_draw(W, V, u[b]);
            }
            if (y < 0) y = argmax_row(prow, V);
        }
        n_acc[b] = a;
        token[b] = y;
    }
    free(W);
    return 0;
}

/* Exposed for the pins: the draw alone, on caller weights in [0, 1]. */
int32_t oracle_fx_draw(const float *w, int V, float u)
{
    uint64_t *W = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(V > 0 ? V : 1));
    if (W == NULL || V < 1) { free(W); return -2; }
    for (int x = 0; x < V; ++x) W[x] = fx_weight(w[x]);
    const int32_t y = fx_draw(W, V, u);
    free(W);
    return y;
}

/*
 * Expert-union cost of a draft subtree: "SpecFit: Not All Draft Tokens Cost the Same in
 * Offloaded MoE Inference", §3.2 eqs (3) and (4): F(S) = sum over layers l of
 * |E_{l,s} u U_{v in S} E_{l,v}| with E_{l,v} the experts node v routes to in layer l (s the
 * root), R(S) = 1 + sum_{v in S} p_v, T(S) = b_{|S|} + beta F(S).  bitmaps [nodes+1][L][W]
 * 64-bit words, node 0 the root, expert e at bit e % 64 of word e / 64; subsets [count] node
 * masks (bit v-1 for node v = 1..nodes <= 32; higher bits ignored); pv [nodes] (index v-1);
 * bcoef [nodes+1].
 * Out: F, size |S|, R, T per subset, and *best = the lowest index of the largest R/T ([SpecFit]
 * eq. (5) over the given candidates).  R and T in double, p_v summed in node order.
 */
int oracle_union_cost(const uint64_t *bitmaps, int nodes, int L, int W, const uint32_t *subsets, int count,
                      const double *pv, const double *bcoef, double beta, int32_t *F, int32_t *size, double *R,
                      double *T, int32_t *best)
{
    if (nodes < 0 || nodes > 32 || L < 1 || W < 1 || count < 0) return -1;
    int32_t bi = -1;
    double bR = 0.0, bT = 1.0;
    for (int c = 0; c < count; ++c) {
        /* bits beyond the pool name no node and are ignored */
        const uint32_t mask = subsets[c] & (nodes >= 32 ? 0xFFFFFFFFu : ((1u << nodes) - 1u));
        int32_t f = 0;
        for (int l = 0; l < L; ++l) {
            for (int w = 0; w < W; ++w) {
                uint64_t acc = bitmaps[((size_t)0 * L + l) * W + w];
                for (int v = 1; v <= nodes; ++v)
                    if ((mask >> (v - 1)) & 1u) acc |= bitmaps[((size_t)v * L + l) * W + w];
                for (int bit = 0; bit < 64; ++bit) f += (int32_t)((acc >> bit) & 1u);
            }
        }
        int32_t k = 0;
        double rr = 1.0;
        for (int v = 1; v <= nodes; ++v)
            if ((mask >> (v - 1)) & 1u) {
                ++k;
                rr += pv[v - 1];
            }
        const double tt = bcoef[k] + beta * (double)f;
        F[c] = f;
        size[c] = k;
        R[c] = rr;
        T[c] = tt;
        if (bi < 0 || rr / tt > bR / bT) {
            bi = c;
            bR = rr;
            bT = tt;
        }
    }
    *best = bi;
    return 0;
}
