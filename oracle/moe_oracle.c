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
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ helpers */

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
    for (int i = 0; i < f; ++i) {
        double g = 0.0, u = 0.0;
        for (int k = 0; k < d; ++k) {
            double xv = widen(x, xdt, xbase + (size_t)k);
            g += widen(wg, wdt, wbase_gu + (size_t)i * d + k) * xv;
            u += widen(wu, wdt, wbase_gu + (size_t)i * d + k) * xv;
        }
        h[i] = g / (1.0 + exp(-g)) * u;
    }
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
    uint64_t w = 3ull * (uint64_t)d * (uint64_t)f * (uint64_t)dtype_size(wdt);
    out[0] = w;
    out[1] = (uint64_t)n * (uint64_t)m * w;
    out[2] = (uint64_t)U * w;
    out[3] = (uint64_t)n * (uint64_t)d * (uint64_t)dtype_size(xdt) + (uint64_t)n * (uint64_t)d * 4ull;
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
