// spec.cu -- the verify-side neighbours of the verification pass.
//
// Speculative sampling, "Lossless but Not Free: An Empirical Anatomy of Speculative Decoding
// on Consumer Hardware" §3.1 (steps 3-4, eqs (1) and (2), Algorithm 1) and §3.2 (the greedy
// special case): for B sequences at once, the walk over the K drafts with the accept test
// r_i < min(1, p_i(x_i)/q_i(x_i)), then one token drawn from the adjusted distribution
// max(0, p_{a+1} - q_{a+1}) (normalised) at the first rejection, or the bonus token from
// p_{K+1} when every draft is accepted.  The uniform draws are inputs.
//
// The draw is an inverse-CDF search with exact integer weights: W = floor(w * 2^46) of each
// weight w clamped to [0, 1], Z = sum W, threshold t = floor(Z * floor(u * 2^24) / 2^24), the
// token the smallest x whose running sum exceeds t.  Integer sums make the drawn index the
// same in any summation order.
//
// One cluster of kSpecCluster CTAs per sequence splits the vocabulary: every warp of the
// cluster owns a contiguous segment of the row and keeps one sum per 128-element step (lane s
// holds step s).  Warp sums are reduced in the CTA, CTA sums exchanged through distributed
// shared memory, and the one warp whose segment holds the threshold re-reads a single step
// to find the token.  A sequence therefore reads the one row pair it needs (p and q at the
// first rejection, or p_{K+1}) once, plus 1 KB.  The greedy rule reads all K+1 target rows
// (the walk needs argmax p_i of each) in one pass.
//
// Expert-union cost, "SpecFit: Not All Draft Tokens Cost the Same in Offloaded MoE Inference"
// §3.2 eqs (3)-(5): for a batch of candidate subtrees S (node masks over a pool of <= 32 draft
// nodes), F(S) = sum over layers of |E_{l,s} u U_{v in S} E_{l,v}| from per-node, per-layer
// expert bitmaps (OR and popcount), R(S) = 1 + sum_{v in S} p_v, T(S) = b_{|S|} + beta F(S),
// and the lowest index of the largest R/T.
#include "common.cuh"
#include "spec_args.cuh"

namespace moe {
namespace {

constexpr int kSpecThreads = 256;
constexpr int kSpecWarps = kSpecThreads / 32;
constexpr int kSpecCluster = 8;           // CTAs per sequence
constexpr int kStepElems = 128;           // elements of one warp step: 32 lanes x 4

__device__ __forceinline__ uint64_t fx_weight(float w) {
    if (!(w > 0.0f)) return 0ull;                   // zero, negative or NaN
    if (w >= 1.0f) return 1ull << 46;
    return __float2ull_rz(w * 70368744177664.0f);   // w * 2^46 is exact in fp32
}

__device__ __forceinline__ uint32_t fx_u24(float u) {
    if (!(u > 0.0f)) return 0u;
    if (u >= 1.0f) return (1u << 24) - 1u;
    return __float2uint_rz(u * 16777216.0f);
}

// floor(Z * U / 2^24) with the 88-bit product
__device__ __forceinline__ uint64_t fx_threshold(uint64_t Z, uint32_t U) {
    const uint64_t lo = Z * static_cast<uint64_t>(U);
    const uint64_t hi = __umul64hi(Z, static_cast<uint64_t>(U));
    return (hi << 40) | (lo >> 24);
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}
__device__ __forceinline__ uint64_t warp_incl_scan_u64(uint64_t v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

// (value, index) with the larger value winning and, among equal values, the lower index
__device__ __forceinline__ void argmax_combine(float &v, int &i, float ov, int oi) {
    if (ov > v || (ov == v && oi < i)) {
        v = ov;
        i = oi;
    }
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared-memory address of `local` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ uint64_t ld_cluster_u64(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Weight of element x of the active row: mode 0 max(0, p - q), mode 1 p.
__device__ __forceinline__ uint64_t row_weight(const float *prow, const float *qrow, int mode, int x) {
    const float pv = __ldg(prow + x);
    float w = pv;
    if (mode == 0) {
        const float dlt = pv - __ldg(qrow + x);
        w = dlt > 0.0f ? dlt : 0.0f;
    }
    return fx_weight(w);
}

// Lane `lane`'s partial of step s of a segment [s0, s1): its 4 elements' weights.
__device__ __forceinline__ uint64_t step_partial(const float *prow, const float *qrow, int mode, int s0, int s1,
                                                 int s, int lane) {
    uint64_t acc = 0;
    const int x0 = s0 + s * kStepElems + 4 * lane;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (x0 + k < s1) acc += row_weight(prow, qrow, mode, x0 + k);
    return acc;
}

constexpr int kVecSteps = 10;   // steps a lane loads at once on the vector path (float4 per step and row)

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ uint64_t pair_weight(float pv, float qv, int mode) {
    float w = pv;
    if (mode == 0) {
        const float dlt = pv - qv;
        w = dlt > 0.0f ? dlt : 0.0f;
    }
    return fx_weight(w);
}

// The warp's (largest value, lowest index) over its segment [s0, s1) of `row`, reduced over
// the warp.  Vector path (vec: the row's base and V are 16-byte multiples): float4 loads, 20
// steps in flight per lane; otherwise 8 independent scalar loads per lane.
__device__ __forceinline__ void seg_argmax(const float *row, int s0, int s1, int nsteps, int lane, bool vec,
                                           float &bv, int &bi) {
    bv = neg_inf();
    bi = 0x7fffffff;
    if (vec) {
        for (int s = 0; s < nsteps; s += 2 * kVecSteps) {
            float4 v[2 * kVecSteps];
#pragma unroll
            for (int j = 0; j < 2 * kVecSteps; ++j) {
                const int x0 = s0 + (s + j) * kStepElems + 4 * lane;
                v[j] = (s + j < nsteps && x0 < s1) ? __ldg(reinterpret_cast<const float4 *>(row + x0))
                                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int j = 0; j < 2 * kVecSteps; ++j) {
                const int x0 = s0 + (s + j) * kStepElems + 4 * lane;
                if (s + j < nsteps && x0 < s1) {
                    argmax_combine(bv, bi, v[j].x, x0);
                    argmax_combine(bv, bi, v[j].y, x0 + 1);
                    argmax_combine(bv, bi, v[j].z, x0 + 2);
                    argmax_combine(bv, bi, v[j].w, x0 + 3);
                }
            }
        }
    } else {
        for (int x = s0 + lane; x < s1; x += 32 * 8) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = (x + 32 * j < s1) ? __ldg(row + x + 32 * j) : 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (x + 32 * j < s1) argmax_combine(bv, bi, v[j], x + 32 * j);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
        argmax_combine(bv, bi, ov, oi);
    }
}

// The sum of each step of the warp's segment, returned in lane s for step s.
__device__ __forceinline__ uint64_t seg_step_sums(const float *prow, const float *qrow, int mode, int s0, int s1,
                                                  int nsteps, int lane, bool vec) {
    uint64_t mine = 0;
    if (vec) {
        for (int s = 0; s < nsteps; s += kVecSteps) {
            float4 pv[kVecSteps], qv[kVecSteps];
#pragma unroll
            for (int j = 0; j < kVecSteps; ++j) {
                const int x0 = s0 + (s + j) * kStepElems + 4 * lane;
                const bool on = s + j < nsteps && x0 < s1;
                pv[j] = on ? __ldg(reinterpret_cast<const float4 *>(prow + x0)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                qv[j] = (on && mode == 0) ? __ldg(reinterpret_cast<const float4 *>(qrow + x0))
                                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int j = 0; j < kVecSteps; ++j) {
                const uint64_t part = pair_weight(pv[j].x, qv[j].x, mode) + pair_weight(pv[j].y, qv[j].y, mode) +
                                      pair_weight(pv[j].z, qv[j].z, mode) + pair_weight(pv[j].w, qv[j].w, mode);
                const uint64_t tot = warp_sum_u64(part);
                if (lane == s + j) mine = tot;
            }
        }
    } else {
        for (int s = 0; s < nsteps; s += 4) {
            uint64_t part[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) part[j] = (s + j < nsteps) ? step_partial(prow, qrow, mode, s0, s1, s + j, lane) : 0ull;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint64_t tot = warp_sum_u64(part[j]);
                if (lane == s + j) mine = tot;
            }
        }
    }
    return mine;
}

__global__ void __launch_bounds__(kSpecThreads) spec_accept_kernel(const SpecArgs a) {
    __shared__ uint64_t warp_tot[kSpecWarps];
    __shared__ uint64_t cta_tot;
    __shared__ float wmax_v[kSpecWarps][kMaxSpecK + 1];
    __shared__ int wmax_i[kSpecWarps][kMaxSpecK + 1];
    __shared__ float cmax_v[kMaxSpecK + 1];
    __shared__ int cmax_i[kMaxSpecK + 1];
    __shared__ int s_acc;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / kSpecCluster;
    const int K = a.K, V = a.V;
    const int g = static_cast<int>(rank) * kSpecWarps + warp;   // warp of the cluster
    const int s0 = min(V, g * a.seg), s1 = min(V, s0 + a.seg);
    const int nsteps = (s1 - s0 + kStepElems - 1) / kStepElems;   // <= 32
    const float *const pseq = a.p + static_cast<size_t>(b) * (K + 1) * V;

    pdl_wait();
    pdl_trigger();

    if (a.greedy) {
        // argmax of every target row over this warp's segment, then the CTA, then the cluster
        for (int i = 0; i <= K; ++i) {
            float bv;
            int bi;
            seg_argmax(pseq + static_cast<size_t>(i) * V, s0, s1, nsteps, lane, a.vec != 0, bv, bi);
            if (lane == 0) {
                wmax_v[warp][i] = bv;
                wmax_i[warp][i] = bi;
            }
        }
        __syncthreads();
        if (threadIdx.x <= K) {
            float bv = wmax_v[0][threadIdx.x];
            int bi = wmax_i[0][threadIdx.x];
            for (int w = 1; w < kSpecWarps; ++w) argmax_combine(bv, bi, wmax_v[w][threadIdx.x], wmax_i[w][threadIdx.x]);
            cmax_v[threadIdx.x] = bv;
            cmax_i[threadIdx.x] = bi;
        }
        cluster_sync();
        if (rank == 0 && warp == 0) {
            // lane i < K+1: row i's argmax over the cluster; then the walk
            int am = 0;
            if (lane <= K) {
                float bv = cmax_v[lane];
                int bi = cmax_i[lane];
                for (uint32_t c = 1; c < kSpecCluster; ++c) {
                    const float ov = __uint_as_float(ld_cluster_u32(cluster_map(smem_u32(&cmax_v[lane]), c)));
                    const int oi = static_cast<int>(ld_cluster_u32(cluster_map(smem_u32(&cmax_i[lane]), c)));
                    argmax_combine(bv, bi, ov, oi);
                }
                am = bi;
            }
            const int x = lane < K ? a.draft[static_cast<size_t>(b) * K + lane] : -1;
            const uint32_t match = __ballot_sync(0xFFFFFFFFu, lane < K && x == am);
            const uint32_t miss = ~match;
            const int acc = min(K, __ffs(miss) - 1);   // leading matches
            const int tok = __shfl_sync(0xFFFFFFFFu, am, acc);
            if (lane == 0) {
                a.n_acc[b] = acc;
                a.token[b] = tok;
            }
        }
        cluster_sync();   // no CTA leaves while its shared memory may still be read
        return;
    }

    // ---------------------------------------------------------------- sampling
    // the walk: lane i < K tests draft i (every CTA of the cluster, redundantly)
    if (warp == 0) {
        bool ok = false;
        if (lane < K) {
            const int x = a.draft[static_cast<size_t>(b) * K + lane];
            if (x >= 0 && x < V) {
                const float px = __ldg(pseq + static_cast<size_t>(lane) * V + x);
                const float qx = __ldg(a.q + (static_cast<size_t>(b) * K + lane) * V + x);
                const float r = __ldg(a.r + static_cast<size_t>(b) * K + lane);
                if (qx > 0.0f) {
                    const float ratio = px / qx;
                    const float thr = ratio < 1.0f ? ratio : 1.0f;
                    ok = r < thr;
                } else {
                    ok = px > 0.0f;
                }
            }
        }
        const uint32_t miss = ~__ballot_sync(0xFFFFFFFFu, ok);
        if (lane == 0) s_acc = min(K, __ffs(miss) - 1);
    }
    __syncthreads();
    const int acc = s_acc;
    const float *const prow = pseq + static_cast<size_t>(acc) * V;
    const float *const qrow = acc < K ? a.q + (static_cast<size_t>(b) * K + acc) * V : prow;
    const uint32_t U = fx_u24(__ldg(a.u + b));

    int token = -1;
    // attempt 0: eq. (2) at a rejection, the bonus row otherwise; attempt 1: the row p itself
    for (int attempt = (acc < K ? 0 : 1); attempt < 2; ++attempt) {
        const int mode = attempt;
        // per step: the warp's sum, kept by lane s
        const uint64_t mine = seg_step_sums(prow, qrow, mode, s0, s1, nsteps, lane, a.vec != 0);
        const uint64_t wtot = warp_sum_u64(mine);
        if (lane == 0) warp_tot[warp] = wtot;
        __syncthreads();
        uint64_t pre_w = 0, ctot = 0;
        for (int w = 0; w < kSpecWarps; ++w) {
            if (w < warp) pre_w += warp_tot[w];
            ctot += warp_tot[w];
        }
        if (threadIdx.x == 0) cta_tot = ctot;
        cluster_sync();
        uint64_t Z = 0, pre_c = 0;
        for (uint32_t c = 0; c < kSpecCluster; ++c) {
            const uint64_t v = ld_cluster_u64(cluster_map(smem_u32(&cta_tot), c));
            if (c < rank) pre_c += v;
            Z += v;
        }
        if (Z != 0) {
            const uint64_t t = fx_threshold(Z, U);
            const uint64_t base = pre_c + pre_w;
            if (wtot != 0 && base <= t && t < base + wtot) {
                // this warp holds the threshold: the step, then the lane, then the element
                const uint64_t incl = warp_incl_scan_u64(mine, lane);
                const uint32_t over = __ballot_sync(0xFFFFFFFFu, base + incl > t);
                const int s = __ffs(over) - 1;
                const uint64_t sbase = base + __shfl_sync(0xFFFFFFFFu, incl - mine, s);
                const uint64_t lp = step_partial(prow, qrow, mode, s0, s1, s, lane);
                const uint64_t lincl = warp_incl_scan_u64(lp, lane);
                const uint32_t lover = __ballot_sync(0xFFFFFFFFu, sbase + lincl > t);
                const int l = __ffs(lover) - 1;
                if (lane == l) {
                    uint64_t c = sbase + lincl - lp;
                    const int x0 = s0 + s * kStepElems + 4 * lane;
                    int x = x0;
                    for (int k = 0; k < 4 && x0 + k < s1; ++k) {
                        c += row_weight(prow, qrow, mode, x0 + k);
                        if (c > t) {
                            x = x0 + k;
                            break;
                        }
                    }
                    a.n_acc[b] = acc;
                    a.token[b] = x;
                }
            }
            token = 0;   // drawn (by the owning warp)
        }
        cluster_sync();   // every CTA is done reading this round's totals
        if (token >= 0) break;
    }
    if (token >= 0) return;

    // every weight of the row is zero: the row's argmax (lowest index of the largest value)
    {
        float bv;
        int bi;
        seg_argmax(prow, s0, s1, nsteps, lane, a.vec != 0, bv, bi);
        if (lane == 0) {
            wmax_v[warp][0] = bv;
            wmax_i[warp][0] = bi;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < kSpecWarps; ++w) argmax_combine(bv, bi, wmax_v[w][0], wmax_i[w][0]);
            cmax_v[0] = bv;
            cmax_i[0] = bi;
        }
        cluster_sync();
        if (rank == 0 && threadIdx.x == 0) {
            float v = cmax_v[0];
            int i = cmax_i[0];
            for (uint32_t c = 1; c < kSpecCluster; ++c)
                argmax_combine(v, i, __uint_as_float(ld_cluster_u32(cluster_map(smem_u32(&cmax_v[0]), c))),
                               static_cast<int>(ld_cluster_u32(cluster_map(smem_u32(&cmax_i[0]), c))));
            a.n_acc[b] = acc;
            a.token[b] = i;
        }
        cluster_sync();
    }
}

// ------------------------------------------------------------------ union cost

// 256 subsets per CTA, kUcPer per thread.  One per thread (256 threads) measured fastest:
// 2 or 4 per thread let one broadcast word serve several subsets but leave fewer warps to
// hide the chains of dependent ORs (70 vs 77 and 83 us for 2^18 subsets of 18 nodes).
constexpr int kUcThreads = 256;
constexpr int kUcPer = 1;
constexpr int kUcChunk = 16;   // words of a subset's accumulator held in registers at a time
constexpr int kUcTabChunk = 8;   // the same for the node-triple table
constexpr int kUcMinBlocks = 5;  // CTAs per SM the registers must allow

// 8-byte asynchronous copy global -> shared (no register staging, all in flight at once)
__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}

__global__ void __launch_bounds__(kUcThreads, kUcMinBlocks) union_cost_kernel(const UnionArgs a,
                                                                             double *const blk_ratio,
                                                                             int *const blk_index) {
    // [nodes+1][L][W] bitmaps, or with the node-triple table only the root's row before it
    extern __shared__ uint64_t sbm[];
    const int words = (a.tab ? 1 : a.nodes + 1) * a.L * a.W;
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i < words; i += blockDim.x) cp_async8(sbm + i, a.bitmaps + i);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    const uint32_t pool = a.nodes >= 32 ? 0xFFFFFFFFu : ((1u << a.nodes) - 1u);
    int cs[kUcPer];
    uint32_t mask[kUcPer];
    int f[kUcPer];
#pragma unroll
    for (int k = 0; k < kUcPer; ++k) {
        cs[k] = blockIdx.x * (kUcThreads * kUcPer) + k * kUcThreads + threadIdx.x;
        mask[k] = cs[k] < a.count ? a.subsets[cs[k]] & pool : 0u;
        f[k] = 0;
    }
    const int LW = a.L * a.W;
    int lw0 = 0;
    if (a.tab) {
        // Node triples: entry ((g * LW/2 + p) * 8 + c) holds word pair p of the OR of the nodes
        // 3g+1..3g+3 selected by the bits of c (nodes past the pool count as empty), so the 8
        // entries of one (triple, pair) fill 128 contiguous bytes and a warp's loads of them are
        // conflict-free.  A lane then ORs one entry per triple, two triples per 3-input op.
        const int NG = (a.nodes + 2) / 3, LW2 = LW >> 1;
        uint4 *const tab = reinterpret_cast<uint4 *>(sbm + words);
        for (int e = threadIdx.x; e < NG * LW2 * 8; e += blockDim.x) {
            const int c = e & 7, gp = e >> 3, g = gp / LW2, pr = gp - g * LW2;
            uint64_t w0 = 0, w1 = 0;
#pragma unroll
            for (int bb = 0; bb < 3; ++bb) {
                const int v = 3 * g + 1 + bb;
                if (v <= a.nodes && ((c >> bb) & 1)) {
                    w0 |= __ldg(a.bitmaps + v * LW + 2 * pr);
                    w1 |= __ldg(a.bitmaps + v * LW + 2 * pr + 1);
                }
            }
            tab[e] = make_uint4(static_cast<uint32_t>(w0), static_cast<uint32_t>(w0 >> 32), static_cast<uint32_t>(w1),
                                static_cast<uint32_t>(w1 >> 32));
        }
        __syncthreads();
        for (int p0 = 0; p0 < LW2; p0 += kUcTabChunk / 2) {
            const int np = min(kUcTabChunk / 2, LW2 - p0);
            const uint4 *const r0 = reinterpret_cast<const uint4 *>(sbm) + p0;   // the root
#pragma unroll
            for (int k = 0; k < kUcPer; ++k) {
                uint32_t acc[2 * kUcTabChunk];
#pragma unroll
                for (int j = 0; j < kUcTabChunk / 2; ++j) {
                    const uint4 b = j < np ? r0[j] : make_uint4(0u, 0u, 0u, 0u);
                    acc[4 * j] = b.x;
                    acc[4 * j + 1] = b.y;
                    acc[4 * j + 2] = b.z;
                    acc[4 * j + 3] = b.w;
                }
                int g = 0;
                for (; g + 1 < NG; g += 2) {
                    const uint4 *const ta = tab + (g * LW2 + p0) * 8 + ((mask[k] >> (3 * g)) & 7u);
                    const uint4 *const tb = tab + ((g + 1) * LW2 + p0) * 8 + ((mask[k] >> (3 * g + 3)) & 7u);
#pragma unroll
                    for (int j = 0; j < kUcTabChunk / 2; ++j) {
                        if (j >= np) break;
                        const uint4 x = ta[8 * j], y = tb[8 * j];
                        acc[4 * j] |= x.x | y.x;
                        acc[4 * j + 1] |= x.y | y.y;
                        acc[4 * j + 2] |= x.z | y.z;
                        acc[4 * j + 3] |= x.w | y.w;
                    }
                }
                if (g < NG) {
                    const uint4 *const ta = tab + (g * LW2 + p0) * 8 + ((mask[k] >> (3 * g)) & 7u);
#pragma unroll
                    for (int j = 0; j < kUcTabChunk / 2; ++j) {
                        if (j >= np) break;
                        const uint4 x = ta[8 * j];
                        acc[4 * j] |= x.x;
                        acc[4 * j + 1] |= x.y;
                        acc[4 * j + 2] |= x.z;
                        acc[4 * j + 3] |= x.w;
                    }
                }
#pragma unroll
                for (int j = 0; j < 2 * kUcTabChunk; ++j) f[k] += __popc(acc[j]);
            }
        }
        lw0 = LW;
    }
    // F(S) = popc of the OR of the root's and the selected nodes' bitmaps, per (layer, word).
    // The node loop is the same in every lane: all lanes read the same word (a broadcast, no
    // bank conflicts), and each ORs it into its subsets' accumulators under their subset bits.
    if (!a.tab && (LW & 1) == 0) {
        for (; lw0 + kUcChunk <= LW; lw0 += kUcChunk) {
            uint32_t acc[kUcPer][2 * kUcChunk];
            const uint4 *const r0 = reinterpret_cast<const uint4 *>(sbm + lw0);   // the root
#pragma unroll
            for (int j = 0; j < kUcChunk / 2; ++j) {
                const uint4 b = r0[j];
#pragma unroll
                for (int k = 0; k < kUcPer; ++k) {
                    acc[k][4 * j] = b.x;
                    acc[k][4 * j + 1] = b.y;
                    acc[k][4 * j + 2] = b.z;
                    acc[k][4 * j + 3] = b.w;
                }
            }
            for (int v = 1; v <= a.nodes; ++v) {
                const uint4 *const rv = reinterpret_cast<const uint4 *>(sbm + v * LW + lw0);
                uint32_t mv[kUcPer];
#pragma unroll
                for (int k = 0; k < kUcPer; ++k) mv[k] = 0u - ((mask[k] >> (v - 1)) & 1u);
#pragma unroll
                for (int j = 0; j < kUcChunk / 2; ++j) {
                    const uint4 b = rv[j];
#pragma unroll
                    for (int k = 0; k < kUcPer; ++k) {
                        acc[k][4 * j] |= b.x & mv[k];
                        acc[k][4 * j + 1] |= b.y & mv[k];
                        acc[k][4 * j + 2] |= b.z & mv[k];
                        acc[k][4 * j + 3] |= b.w & mv[k];
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kUcPer; ++k)
#pragma unroll
                for (int j = 0; j < 2 * kUcChunk; ++j) f[k] += __popc(acc[k][j]);
        }
    }
    for (; lw0 < LW; ++lw0) {   // the rest, one word at a time
        uint64_t acc[kUcPer];
#pragma unroll
        for (int k = 0; k < kUcPer; ++k) acc[k] = sbm[lw0];
        for (int v = 1; v <= a.nodes; ++v) {
            const uint64_t b = sbm[v * LW + lw0];
#pragma unroll
            for (int k = 0; k < kUcPer; ++k) acc[k] |= b & (0ull - static_cast<uint64_t>((mask[k] >> (v - 1)) & 1u));
        }
#pragma unroll
        for (int k = 0; k < kUcPer; ++k) f[k] += __popcll(acc[k]);
    }
    // R, T and the outputs; the thread's best in ascending subset order: its first subset,
    // then any strictly larger ratio (lowest index on ties, whatever the signs)
    double ratio = -INFINITY;
    int index = 0x7fffffff;
#pragma unroll
    for (int k = 0; k < kUcPer; ++k) {
        if (cs[k] >= a.count) continue;
        int n = 0;
        double rr = 1.0;
        for (int v = 1; v <= a.nodes; ++v)
            if ((mask[k] >> (v - 1)) & 1u) {
                ++n;
                rr += a.pv[v - 1];
            }
        // no fused multiply-add: the same rounding as the plain product and sum
        const double tt = __dadd_rn(a.bcoef[n], __dmul_rn(a.beta, static_cast<double>(f[k])));
        a.F[cs[k]] = f[k];
        a.size[cs[k]] = n;
        a.R[cs[k]] = rr;
        a.T[cs[k]] = tt;
        const double q = rr / tt;
        if (index == 0x7fffffff || q > ratio) {
            ratio = q;
            index = cs[k];
        }
    }
    // the block's lowest index of the largest ratio
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const double orat = __shfl_xor_sync(0xFFFFFFFFu, ratio, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, index, off);
        if (orat > ratio || (orat == ratio && oi < index)) {
            ratio = orat;
            index = oi;
        }
    }
    __shared__ double wr[8];
    __shared__ int wi[8];
    if ((threadIdx.x & 31) == 0) {
        wr[threadIdx.x >> 5] = ratio;
        wi[threadIdx.x >> 5] = index;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (blockDim.x + 31) / 32; ++w)
            if (wr[w] > ratio || (wr[w] == ratio && wi[w] < index)) {
                ratio = wr[w];
                index = wi[w];
            }
        blk_ratio[blockIdx.x] = ratio;
        blk_index[blockIdx.x] = index;
    }
}

__global__ void __launch_bounds__(256) union_best_kernel(const double *blk_ratio, const int *blk_index, int blocks,
                                                        int32_t *best) {
    pdl_wait();
    pdl_trigger();
    double ratio = -INFINITY;
    int index = 0x7fffffff;
    for (int i = threadIdx.x; i < blocks; i += blockDim.x)
        if (blk_ratio[i] > ratio || (blk_ratio[i] == ratio && blk_index[i] < index)) {
            ratio = blk_ratio[i];
            index = blk_index[i];
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const double orat = __shfl_xor_sync(0xFFFFFFFFu, ratio, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, index, off);
        if (orat > ratio || (orat == ratio && oi < index)) {
            ratio = orat;
            index = oi;
        }
    }
    __shared__ double wr[8];
    __shared__ int wi[8];
    if ((threadIdx.x & 31) == 0) {
        wr[threadIdx.x >> 5] = ratio;
        wi[threadIdx.x >> 5] = index;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < static_cast<int>(blockDim.x + 31) / 32; ++w)
            if (wr[w] > ratio || (wr[w] == ratio && wi[w] < index)) {
                ratio = wr[w];
                index = wi[w];
            }
        *best = index == 0x7fffffff ? -1 : index;
    }
}

}  // namespace

int spec_segment(int V) {
    const int warps = kSpecCluster * kSpecWarps;
    const int per = (V + warps - 1) / warps;
    return (per + kStepElems - 1) / kStepElems * kStepElems;
}

cudaError_t launch_spec_accept(const SpecArgs &a, cudaStream_t s, bool pdl) {
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSpecCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B * kSpecCluster));
    cfg.blockDim = dim3(kSpecThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, spec_accept_kernel, a);
}

size_t union_cost_scratch_bytes(int count) {
    const size_t blocks = static_cast<size_t>((count + 255) / 256);
    return blocks * (sizeof(double) + sizeof(int));
}

cudaError_t launch_union_cost(const UnionArgs &a, void *scratch, cudaStream_t s, bool pdl) {
    const int blocks = (a.count + 255) / 256;
    double *blk_ratio = static_cast<double *>(scratch);
    int *blk_index = reinterpret_cast<int *>(blk_ratio + blocks);
    // the node-triple table when the row width is even and it fits beside the bitmaps
    UnionArgs b = a;
    const size_t lw = static_cast<size_t>(a.L) * a.W;
    const size_t bm_bytes = static_cast<size_t>(a.nodes + 1) * lw * sizeof(uint64_t);
    const size_t tab_bytes = static_cast<size_t>((a.nodes + 2) / 3) * 8 * lw * sizeof(uint64_t);
    b.tab = (lw % 2 == 0 && a.nodes > 0 && lw * sizeof(uint64_t) + tab_bytes <= kMaxUnionSmem) ? 1 : 0;
    const size_t smem = b.tab ? lw * sizeof(uint64_t) + tab_bytes : bm_bytes;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(union_cost_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxUnionSmem));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kUcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, union_cost_kernel, static_cast<const UnionArgs>(b), blk_ratio, blk_index);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, union_best_kernel, static_cast<const double *>(blk_ratio),
                              static_cast<const int *>(blk_index), blocks, a.best);
}

}  // namespace moe
