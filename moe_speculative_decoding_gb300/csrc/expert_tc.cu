// expert_tc.cu -- tensor-core (tcgen05 + TMA) kernels of the expert operation, bf16.
//
// "Speculative Decoding for Mixture-of-Experts Models" (Lan), §1: the expert operation
// is the gate, up and down projections of each token of a pass with the weights of its
// selected experts.  Per-slot form: one expert read per slot (m*n*w bytes requested).
// Deduplicating form: the pass's tokens grouped by expert, each distinct expert read once
// (w * X(n) bytes).  §2 "Effective bandwidth": the figure of merit is requested expert
// bytes over time, so the design streams weights at the memory's rate and keeps every
// other byte off the memory path.
//
// A group is one slot (per-slot form) or one distinct expert with all of its tokens
// (deduplicating form); an item is (group, 64-row tile of f).  One call is two kernels,
// chained by programmatic dependent launch, each with one CTA per SM and 6 warps (warp 0
// the TMA producer, warp 1 the tcgen05.mma issuer, warps 2-5 the epilogue, one TMEM lane
// per thread):
//
//   gate/up kernel.  A block is one 64-wide k slice of an item: 64 rows of W_gate and
//   the same 64 rows of W_up (16 KB, the M = 128 operand) plus the pass's x for that k
//   slice (16 tokens x 64, 2 KB, from L2).  All G*T*KB blocks of the call are cut into
//   equal contiguous ranges, one per CTA, so every SM streams the same number of weight
//   bytes whatever the pass size and the number of groups.  A CTA accumulates the blocks
//   of each item it touches in TMEM (bf16 in, fp32 out, weights as M, tokens as N = 16)
//   and stores the partial sums of its share of the item, [128 rows] per token, to the
//   workspace.  With at most 2*G*T CTAs every range holds at least half an item, so at
//   most three CTAs share an item.  The kernel also zeroes y when the call overwrites it.
//
//   down kernel.  A block is (item, 128-row block of d): 128 rows of W_down by the tile's
//   64 columns (16 KB); the blocks are again cut into equal ranges.  Its producer starts
//   streaming W_down as soon as the CTA is resident, while the gate/up kernel still runs:
//   neither the weights nor the routing depend on it.  After the wait, the epilogue warps
//   form h = silu(g) * u of each item from its (at most three) partial sums in a fixed
//   order, as bf16 in the swizzled layout of the MMA's B operand, one item ahead of the
//   MMAs, and add gate * (W_down h) into the fp32 output with atomics: the weighted
//   combine and the reduction over f tiles are fused there.
//
// FP8 layers (e4m3 weights and x, one fp32 scale per weight row and per token) run the same
// two kernels instantiated for kind::f8f6f4: a 128-byte row then holds 128 elements, so a
// gate/up block is a 128-wide k slice and one down block covers the item's whole 128-wide
// f span.  The gate/up epilogue applies the row and token scales to its partial sums; the
// h formers quantize h per (token, 128-wide f span) with scale amax/448, and the down
// epilogue applies that scale and the W_down row scale.
//
// Both kernels' shared memory fits one SM together (about 215 KB of 228 KB), so a down
// CTA is resident beside a gate/up CTA and its first W_down stages are in flight before
// the gate/up kernel ends.  Every wait is bounded (common.cuh); a time-out raises an abort
// flag that every role honours, records MOE_ERR_DEVICE_TIMEOUT, drains copies and MMAs in
// flight and frees TMEM before the CTA exits.
#include "common.cuh"
#include "expert_args.cuh"

#include <algorithm>
#include <mutex>

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kOB = 128;                      // d rows per down block
constexpr int kNT = 16;                       // MMA N (token columns)
constexpr uint32_t kWBytes = 16384;           // weight bytes of one block
constexpr uint32_t kXTileBytes = kNT * 128;   // x of one k slice: 16 rows x 128 B
constexpr uint32_t kGUStageBytes = kWBytes + kXTileBytes;
constexpr uint32_t kHBytes = kNT * 128;       // one h tile: 16 rows x 64 bf16
constexpr int kGUStages = 7;
constexpr int kDownStages = 5;
constexpr int kDownBufs = 8;                  // TMEM ring of down-block accumulators
constexpr int kEpiBatch = 4;                  // down blocks per epilogue round
constexpr uint32_t kGUTmemCols = 32;          // two 16-column accumulators
constexpr uint32_t kDownTmemCols = 16 * kDownBufs;
constexpr long long kDrainCycles = 400000000ll;   // about 0.2 s

// Element type of a kernel instantiation: bf16 (kind::f16) or e4m3 (kind::f8f6f4).
template <bool F8>
struct Elt {
    static constexpr int BK = F8 ? 128 : 64;   // k elements per 128-byte row of an operand tile
    static constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(128, kNT) : idesc_bf16_f32(128, kNT);
    // down blocks per unit: two 64-wide f tiles of bf16, or one 128-wide tile of e4m3
    static constexpr int UNIT = F8 ? 1 : 2;
    __device__ __forceinline__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
        if constexpr (F8) tc_mma_f8(d, a, b, IDESC, acc);
        else tc_mma_bf16(d, a, b, IDESC, acc);
    }
};
constexpr uint32_t kFull = 0xFFFFFFFFu;

// Shared memory of the gate/up kernel: stages, then barriers full[S], empty[S],
// acc_full[2], acc_empty[2], drain, then the TMEM address and the abort flag.
constexpr uint32_t kGUBars = kGUStages * kGUStageBytes;
constexpr uint32_t kGUNumBars = 2 * kGUStages + 5;
constexpr uint32_t kGUMisc = kGUBars + 8 * kGUNumBars;
constexpr uint32_t kSmemPerSM = 233472;             // shared memory of one SM (228 KB)
constexpr uint32_t kSmemReserved = 1024;            // reserved by the system per CTA
// A gate/up CTA takes more than half an SM, so two of them never share one: every SM then
// keeps room for one down CTA beside its gate/up CTA (see the note at the top).
constexpr uint32_t kGUSmemMin = (kSmemPerSM - 2 * kSmemReserved) / 2 + 16;
constexpr uint32_t kGUSmemUsed = kGUMisc + 16 + 1024;   // + alignment slack of the base
constexpr uint32_t kGUSmem = kGUSmemUsed > kGUSmemMin ? kGUSmemUsed : kGUSmemMin;
// Shared memory of the down kernel: stages, kHRing h tiles, their group records, then
// barriers full[S], empty[S], acc_full[B], acc_empty[B], h_full[R], h_empty[R], drain,
// then the misc words.
constexpr int kHRing = 4;
constexpr int kGUMaxRegs = 64;
constexpr int kDnMaxRegs = 192;
static_assert(2 * 32 * (kGUMaxRegs + kDnMaxRegs) <= 16384, "two warps of each kernel per sub-partition");
constexpr int kDnSub = 2;                     // f tiles per down item: blocks of one d block accumulate
constexpr int kDnThreads = 256;               // + warps 6-7: the h formers
constexpr uint32_t kDnH = kDownStages * kWBytes;
constexpr uint32_t kHEntry = kDnSub * kHBytes;
constexpr uint32_t kDnInfo = kDnH + kHRing * kHEntry;
constexpr uint32_t kInfoBytes = 144;          // mask, the 16 gates, the 16 h scales (FP8)
constexpr uint32_t kDnScratch = kDnInfo + kHRing * kInfoBytes;   // [2][2 warps][16] h amax (FP8)
constexpr uint32_t kDnBars = kDnScratch + 2 * 2 * kNT * 4;
constexpr uint32_t kDnNumBars = 2 * kDownStages + 2 * kDownBufs + 2 * kHRing + 1;
constexpr uint32_t kDnMisc = kDnBars + 8 * kDnNumBars;
constexpr uint32_t kDnSmem = kDnMisc + 16 + 1024;
static_assert(kGUSmem + kDnSmem + 2 * kSmemReserved <= kSmemPerSM, "a gate/up and a down CTA must share one SM");
static_assert(2 * (kGUSmem + kSmemReserved) > kSmemPerSM, "two gate/up CTAs must not fit one SM");

// Equal contiguous ranges of `blocks` work blocks over `parts` CTAs: CTA c takes
// [lo(c), lo(c + 1)).
struct Split {
    long long blocks;
    int parts;
    __device__ __forceinline__ long long lo(int c) const { return static_cast<long long>(c) * blocks / parts; }
    // the CTA whose range holds block b (blocks > 0, 0 <= b < blocks)
    __device__ __forceinline__ int part_of(long long b) const {
        return static_cast<int>(((b + 1) * parts + blocks - 1) / blocks - 1);
    }
};

// CTAs that share the gate/up blocks: at most 2*G*T, so that every range holds at least
// KB/2 blocks and an item of KB blocks meets at most kMaxSpan = 3 ranges.
__device__ __forceinline__ int gu_parts(int G, int T, int grid) {
    const long long cap = 2ll * G * T;
    return static_cast<int>(cap < 1 ? 1 : (cap < grid ? cap : grid));
}

__device__ __forceinline__ int num_groups(const ExpertArgs &a) {
    if (a.mode == kModePerSlot) return a.n * a.m;
    // the device-side count is clamped to the buffer sizes the host validated
    const int cap = a.n * a.m < a.N ? a.n * a.m : a.N;
    return max(0, min(a.num_distinct[0], cap));
}

// The part of one item inside a CTA's block range [.., hi); `inner` blocks per item.
struct Seg {
    long long b0, b1;
    int item, g, tile, e;
    bool valid;   // expert id inside [0, N): every role skips the others the same way
};

__device__ __forceinline__ Seg seg_at(const ExpertArgs &a, long long b, long long hi, int inner, int T) {
    Seg s;
    s.item = static_cast<int>(b / inner);
    s.b0 = b;
    const long long end = static_cast<long long>(s.item + 1) * inner;
    s.b1 = end < hi ? end : hi;
    s.g = s.item / T;
    s.tile = s.item - s.g * T;
    s.e = (a.mode == kModePerSlot) ? a.ids[s.g] : a.expert_list[s.g];
    s.valid = s.e >= 0 && s.e < a.N;
    return s;
}

// Tokens of group g, computed by one whole warp: the mask of pass tokens in the group,
// each token's summed gate and its slot position p (its row of the partial-sum buffer).
// The deduplicating form reads the group's slot list with one lane per slot and gathers
// it with ballots, so a group of k slots costs one round trip to memory, not k.
struct GroupInfo {
    uint32_t mask;
    float gt[kNT];
    int pos[kNT];
};

__device__ __forceinline__ void group_tokens(const ExpertArgs &a, int g, int lane, GroupInfo &gi) {
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        gi.gt[t] = 0.0f;
        gi.pos[t] = 0;
    }
    if (a.mode == kModePerSlot) {
        const int tt = g / a.m;
        const float gv = a.gates[g];
#pragma unroll
        for (int t = 0; t < kNT; ++t)
            if (t == tt) {
                gi.gt[t] = gv;
                gi.pos[t] = g;
            }
        gi.mask = 1u << tt;
        return;
    }
    const int S = a.n * a.m;   // offsets are clamped to the slot buffer
    const int p0 = max(0, a.offsets[g]), p1 = min(S, a.offsets[g + 1]);
    uint32_t mask = 0;
    for (int pb = p0; pb < p1; pb += 32) {
        const int p = pb + lane;
        int tt = -1;
        float gv = 0.0f;
        if (p < p1) {
            const int slot = a.slot_order[p];
            if (slot >= 0 && slot < S) {
                tt = slot / a.m;
                gv = a.gates[slot];
            }
        }
#pragma unroll
        for (int t = 0; t < kNT; ++t) {
            uint32_t bal = __ballot_sync(kFull, tt == t);
            if (bal == 0u) continue;
            mask |= 1u << t;
            gi.pos[t] = pb + 31 - __clz(bal);
            // a token appears once per group in a grouping of distinct top-m ids; a
            // repeated one gets the sum of its gates
            float sum = 0.0f;
            while (bal) {
                sum += __shfl_sync(kFull, gv, __ffs(bal) - 1);
                bal &= bal - 1u;
            }
            gi.gt[t] += sum;
        }
    }
    gi.mask = mask;
}

// Row `row` of the partial sums that CTA share `slot` holds for (slot position p, tile).
__device__ __forceinline__ size_t part_index(int p, int T, int tile, int slot, int row) {
    return ((static_cast<size_t>(p) * T + tile) * kMaxSpan + slot) * 128 + row;
}

// Wait (bounded) for the copies a producer issued and nobody consumed, after an abort.
__device__ __forceinline__ void drain_copies(uint32_t bar_full, uint32_t cnt, int stages) {
    const uint32_t first = cnt > static_cast<uint32_t>(stages) ? cnt - stages : 0u;
    for (uint32_t j = first; j < cnt; ++j)
        mbar_wait_drain(bar_full + 8u * (j % stages), (j / stages) & 1u, kDrainCycles);
}

// ==================================================================== gate/up kernel

template <bool F8>
__global__ void __maxnreg__(kGUMaxRegs)
expert_gu_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                 const __grid_constant__ CUtensorMap tm_x, const ExpertArgs a, float *const part,
                 const int zero_y) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw_addr);
    const uint32_t bar_full = base + kGUBars;
    const uint32_t bar_empty = bar_full + 8u * kGUStages;
    const uint32_t bar_acc_full = bar_empty + 8u * kGUStages;   // [2]
    const uint32_t bar_acc_empty = bar_acc_full + 16u;         // [2]
    const uint32_t bar_drain = bar_acc_empty + 16u;
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + kGUMisc);
    volatile int32_t *const abort_flag = reinterpret_cast<volatile int32_t *>(base_ptr + kGUMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGUStages; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8u * b, 1);
            mbar_init(bar_acc_empty + 8u * b, 4);   // the 4 epilogue warps
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tm_wg);
        tma_prefetch_map(&tm_wu);
        tma_prefetch_map(&tm_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kGUTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Every thread waits for the grids this one depends on before reading any input, and
    // only then lets the down kernel launch: that kernel reads the routing inputs before
    // its own wait, which is sound because they were complete when this point was passed.
    pdl_wait();
    pdl_trigger();

    using E = Elt<F8>;
    const int T = a.f / kFTile;
    const int KB = a.d / E::BK;
    const int G = num_groups(a);
    const Split sp{static_cast<long long>(G) * T * KB, gu_parts(G, T, gridDim.x)};
    const int c = blockIdx.x;
    const long long lo = c < sp.parts ? sp.lo(c) : 0, hi = c < sp.parts ? sp.lo(c + 1) : 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the schedule and waits; one elected lane issues the copies.
        uint32_t cnt = 0;
        bool ok = true;
        for (long long b = lo; ok && b < hi;) {
            const Seg s = seg_at(a, b, hi, KB, T);
            b = s.b1;
            if (!s.valid) continue;
            const int row = s.e * a.f + s.tile * kFTile;
            for (long long bb = s.b0; bb < s.b1; ++bb) {
                const uint32_t st = cnt % kGUStages, ph = (cnt / kGUStages) & 1u;
                if (!warp_wait(bar_empty + 8u * st, ph ^ 1u, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                const int k0 = static_cast<int>(bb - static_cast<long long>(s.item) * KB) * E::BK;
                if (elect_one()) {
                    const uint32_t dst = base + st * kGUStageBytes, fb = bar_full + 8u * st;
                    mbar_arrive_expect_tx(fb, kGUStageBytes);
                    tma_load_2d(dst, &tm_wg, fb, k0, row);
                    tma_load_2d(dst + kWBytes / 2, &tm_wu, fb, k0, row);
                    tma_load_2d(dst + kWBytes, &tm_x, fb, k0, 0);
                }
                __syncwarp();
                ++cnt;
            }
        }
        if (!ok && lane == 0) drain_copies(bar_full, cnt, kGUStages);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Warp-uniform loop; waits by every lane, MMAs and commits by one elected lane.
        uint32_t cnt = 0, seg = 0;
        bool ok = true;
        for (long long b = lo; ok && b < hi;) {
            const Seg s = seg_at(a, b, hi, KB, T);
            b = s.b1;
            if (!s.valid) continue;
            const uint32_t buf = seg & 1u, sph = (seg >> 1) & 1u;
            ++seg;
            if (!warp_wait(bar_acc_empty + 8u * buf, sph ^ 1u, abort_flag, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + 16u * buf;
            for (long long bb = s.b0; bb < s.b1; ++bb) {
                const uint32_t st = cnt % kGUStages, ph = (cnt / kGUStages) & 1u;
                if (!warp_wait(bar_full + 8u * st, ph, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = base + st * kGUStageBytes;
                const uint32_t sb = sa + kWBytes;
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)   // 32 bytes of K per instruction
                        E::mma(d_tmem, desc_kmajor_sw128(sa + 32u * k), desc_kmajor_sw128(sb + 32u * k),
                               (bb != s.b0 || k != 0) ? 1u : 0u);
                    tc_commit(bar_empty + 8u * st);
                    if (bb == s.b1 - 1) tc_commit(bar_acc_full + 8u * buf);
                }
                __syncwarp();
                ++cnt;
            }
        }
        // every MMA this warp issued completes before TMEM is released
        if (elect_one()) {
            tc_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0, kDrainCycles);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int row = q * 32 + lane;        // TMEM lane = accumulator row (gate 0-63, up 64-127)
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const int et = static_cast<int>(threadIdx.x) - 64;
        if (zero_y) {
            // this CTA's share of y = 0; the down kernel adds into it after its wait
            const long long n4 = static_cast<long long>(a.n) * a.d / 4;
            const long long z0 = c * n4 / gridDim.x, z1 = (c + 1) * n4 / gridDim.x;
            float4 *const y4 = reinterpret_cast<float4 *>(a.y);
            for (long long i = z0 + et; i < z1; i += 128) y4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        uint32_t seg = 0;
        for (long long b = lo; b < hi;) {
            const Seg s = seg_at(a, b, hi, KB, T);
            b = s.b1;
            if (!s.valid) {
                // reported once per group, by the CTA holding the group's first block
                if (warp == 2 && lane == 0 && s.tile == 0 && s.b0 == static_cast<long long>(s.item) * KB)
                    record_error(a.err, MOE_ERR_BAD_ID);
                continue;
            }
            GroupInfo gi;
            group_tokens(a, s.g, lane, gi);
            // this CTA's share of the item: 0 for the CTA holding its first block
            const int slot = c - sp.part_of(static_cast<long long>(s.item) * KB);
            const uint32_t buf = seg & 1u, sph = (seg >> 1) & 1u;
            ++seg;
            // wait outcomes are made warp-uniform so the .sync.aligned TMEM loads stay converged
            if (!warp_wait(bar_acc_full + 8u * buf, sph, abort_flag, a.err)) break;
            tc_fence_after();
            float v[16];
            tmem_ld_16(tmem + lane_off + 16u * buf, v);
            tc_fence_before();
            warp_arrive(bar_acc_empty + 8u * buf);
            if (slot < 0 || slot >= kMaxSpan) continue;   // not reachable with gu_parts' bound
            if constexpr (F8) {
                // integer-exact sums of codes back to values: weight-row scale times token scale
                const int fr = s.e * a.f + s.tile * kFTile + (row & 63);
                const float rs = row < 64 ? a.s_gate[fr] : a.s_up[fr];
#pragma unroll
                for (int t = 0; t < kNT; ++t)
                    if ((gi.mask >> t) & 1u) v[t] *= rs * a.s_x[t];
            }
#pragma unroll
            for (int t = 0; t < kNT; ++t)
                if ((gi.mask >> t) & 1u) part[part_index(gi.pos[t], T, s.tile, slot, row)] = v[t];
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kGUTmemCols);
    }
}

// ==================================================================== down kernel

// Registers: one SM sub-partition (a quarter of the 64K register file) holds up to two
// warps of each kernel, so 2 * 32 * (down registers) + 2 * 32 * (gate/up registers) must stay
// within 16384: with the gate/up kernel at 64, the down kernel gets at most 192.
template <bool F8>
__global__ void __maxnreg__(kDnMaxRegs)
expert_down_kernel(const __grid_constant__ CUtensorMap tm_wd, const ExpertArgs a, const float *const part,
                   const int gu_grid) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sh = base + kDnH;
    uint8_t *const h_ptr = base_ptr + kDnH;
    uint8_t *const info_ptr = base_ptr + kDnInfo;
    float *const scratch = reinterpret_cast<float *>(base_ptr + kDnScratch);
    const uint32_t bar_full = base + kDnBars;
    const uint32_t bar_empty = bar_full + 8u * kDownStages;
    const uint32_t bar_acc_full = bar_empty + 8u * kDownStages;    // [kDownBufs]
    const uint32_t bar_acc_empty = bar_acc_full + 8u * kDownBufs;  // [kDownBufs]
    const uint32_t bar_h_full = bar_acc_empty + 8u * kDownBufs;    // [kHRing]
    const uint32_t bar_h_empty = bar_h_full + 8u * kHRing;         // [kHRing]
    const uint32_t bar_drain = bar_h_empty + 8u * kHRing;
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + kDnMisc);
    volatile int32_t *const abort_flag = reinterpret_cast<volatile int32_t *>(base_ptr + kDnMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDownStages; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int b = 0; b < kDownBufs; ++b) {
            mbar_init(bar_acc_full + 8u * b, 1);
            mbar_init(bar_acc_empty + 8u * b, 4);       // the 4 epilogue warps
        }
        for (int b = 0; b < kHRing; ++b) {
            mbar_init(bar_h_full + 8u * b, 2);          // the 2 h-former warps
            mbar_init(bar_h_empty + 8u * b, 1 + 4);     // the MMAs' commit and the epilogue warps
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tm_wd);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kDownTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the next grid on the stream may become resident now; it waits for this one
    pdl_trigger();

    // The routing inputs (ids, or the grouping and its count) were complete before every
    // CTA of the gate/up kernel passed its wait, and this grid starts only after all of
    // them did, so they are read here before this grid's own wait.  The partial sums and
    // y are touched only after it.
    //
    // An item is (group, kDnSub consecutive f tiles); its blocks run over (d block ob,
    // sub-tile s), s innermost, so the sub-tiles of one d block accumulate in one TMEM
    // accumulator: a unit.  The last item of a group has fewer real sub-tiles when T is
    // not a multiple of kDnSub; the others are skipped by every role alike.
    using E = Elt<F8>;
    const int T = a.f / kFTile;
    const int T2 = (T + kDnSub - 1) / kDnSub;
    const int KB = a.d / E::BK;
    const int OBS = a.d / kOB;
    const int IB = OBS * E::UNIT;   // blocks per item
    const int G = num_groups(a);
    const long long nblk = static_cast<long long>(G) * T2 * IB;
    const Split sp{nblk, static_cast<int>(nblk < 1 ? 1 : (nblk < gridDim.x ? nblk : gridDim.x))};
    const int c = blockIdx.x;
    const long long lo = c < sp.parts ? sp.lo(c) : 0, hi = c < sp.parts ? sp.lo(c + 1) : 0;
    // the units of segment s: for (ob = ob_first; ob <= ob_last; ++ob) sub-tiles [s_lo, s_hi)
    struct Units {
        int r0, r1, nreal;
        __device__ __forceinline__ int ob_first() const { return r0 / E::UNIT; }
        __device__ __forceinline__ int ob_last() const { return (r1 - 1) / E::UNIT; }
        __device__ __forceinline__ int s_lo(int ob) const { return max(0, r0 - ob * E::UNIT); }
        __device__ __forceinline__ int s_hi(int ob) const { return min(nreal, min(E::UNIT, r1 - ob * E::UNIT)); }
    };
    auto units_of = [&](const Seg &sg) {
        Units u;
        const long long ib0 = static_cast<long long>(sg.item) * IB;
        u.r0 = static_cast<int>(sg.b0 - ib0);
        u.r1 = static_cast<int>(sg.b1 - ib0);
        // bf16: the item's 64-wide tiles present (the last item of a group may have one);
        // e4m3: one block spans the item's 128 columns (f is a multiple of 128)
        u.nreal = F8 ? 1 : min(kDnSub, T - sg.tile * kDnSub);
        return u;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t cnt = 0;
        bool ok = true;
        for (long long b = lo; ok && b < hi;) {
            const Seg sg = seg_at(a, b, hi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const Units u = units_of(sg);
            for (int ob = u.ob_first(); ok && ob <= u.ob_last(); ++ob) {
                for (int sub = u.s_lo(ob); sub < u.s_hi(ob); ++sub) {
                    const uint32_t st = cnt % kDownStages, ph = (cnt / kDownStages) & 1u;
                    if (!warp_wait(bar_empty + 8u * st, ph ^ 1u, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        const uint32_t fb = bar_full + 8u * st;
                        mbar_arrive_expect_tx(fb, kWBytes);
                        tma_load_2d(base + st * kWBytes, &tm_wd, fb, (sg.tile * kDnSub + sub) * kFTile,
                                    sg.e * a.d + ob * kOB);
                    }
                    __syncwarp();
                    ++cnt;
                }
            }
        }
        if (!ok && lane == 0) drain_copies(bar_full, cnt, kDownStages);
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        uint32_t cnt = 0, dcnt = 0, run = 0;
        bool ok = true;
        for (long long b = lo; ok && b < hi;) {
            const Seg sg = seg_at(a, b, hi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const Units u = units_of(sg);
            const uint32_t hb = run % kHRing, hph = (run / kHRing) & 1u;
            ++run;
            if (!warp_wait(bar_h_full + 8u * hb, hph, abort_flag, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sb = sh + hb * kHEntry;
            for (int ob = u.ob_first(); ok && ob <= u.ob_last(); ++ob) {
                const int s0 = u.s_lo(ob), s1 = u.s_hi(ob);
                if (s0 >= s1) continue;
                const uint32_t buf = dcnt % kDownBufs, dph = (dcnt / kDownBufs) & 1u;
                ++dcnt;
                if (!warp_wait(bar_acc_empty + 8u * buf, dph ^ 1u, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                for (int sub = s0; sub < s1; ++sub) {
                    const uint32_t st = cnt % kDownStages, ph = (cnt / kDownStages) & 1u;
                    if (!warp_wait(bar_full + 8u * st, ph, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + st * kWBytes;
                    const uint32_t sbs = sb + static_cast<uint32_t>(sub) * kHBytes;
                    if (elect_one()) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // 32 bytes of K per instruction
                            E::mma(tmem + 16u * buf, desc_kmajor_sw128(sa + 32u * k), desc_kmajor_sw128(sbs + 32u * k),
                                   (sub != s0 || k != 0) ? 1u : 0u);
                        tc_commit(bar_empty + 8u * st);
                        if (sub == s1 - 1) tc_commit(bar_acc_full + 8u * buf);
                    }
                    __syncwarp();
                    ++cnt;
                }
            }
            // the h entry is free again once this run's MMAs have read it
            if (elect_one()) tc_commit(bar_h_empty + 8u * hb);
            __syncwarp();
        }
        if (elect_one()) {
            tc_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0, kDrainCycles);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        // y[t, o] += gate_t * (W_down h)[o, t] with the run's gates from its group record
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        pdl_wait();   // y as the gate/up kernel left it
        uint32_t dcnt = 0, run = 0;
        bool ok = true;
        for (long long b = lo; ok && b < hi;) {
            const Seg sg = seg_at(a, b, hi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const Units u = units_of(sg);
            const uint32_t hb = run % kHRing, hph = (run / kHRing) & 1u;
            ++run;
            if (!warp_wait(bar_h_full + 8u * hb, hph, abort_flag, a.err)) break;
            const uint32_t *const rec = reinterpret_cast<const uint32_t *>(info_ptr + hb * kInfoBytes);
            const uint32_t mask = rec[0];
            float gt[kNT];
#pragma unroll
            for (int t = 0; t < kNT; ++t) gt[t] = __uint_as_float(rec[1 + t]);
            if constexpr (F8) {
#pragma unroll
                for (int t = 0; t < kNT; ++t) gt[t] *= __uint_as_float(rec[17 + t]);   // h scale of the span
            }
            warp_arrive(bar_h_empty + 8u * hb);
            // units in batches of up to kEpiBatch: their TMEM loads share one wait
            for (int ob = u.ob_first(); ok && ob <= u.ob_last();) {
                int obs[kEpiBatch];
                int nb = 0;
                uint32_t r[kEpiBatch][16];
#pragma unroll
                for (int j = 0; j < kEpiBatch; ++j) {
                    obs[j] = -1;
                    while (ob <= u.ob_last() && u.s_lo(ob) >= u.s_hi(ob)) ++ob;   // no real sub-tile
                    if (ob > u.ob_last()) break;
                    const uint32_t buf = dcnt % kDownBufs, dph = (dcnt / kDownBufs) & 1u;
                    // the first unit of a batch is waited for; later ones join only if
                    // already complete, so a batch never holds back finished accumulators
                    if (j > 0 && !__all_sync(kFull, mbar_try_wait(bar_acc_full + 8u * buf, dph))) break;
                    if (!warp_wait(bar_acc_full + 8u * buf, dph, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_ld_16_async(tmem + lane_off + 16u * buf, r[j]);
                    obs[j] = ob;
                    ++nb;
                    ++dcnt;
                    ++ob;
                }
                tmem_wait_ld();   // also before leaving on an abort: no load stays in flight
                if (!ok) break;
                tc_fence_before();
#pragma unroll
                for (int j = 0; j < kEpiBatch; ++j)
                    if (j < nb) warp_arrive(bar_acc_empty + 8u * ((dcnt - nb + j) % kDownBufs));
#pragma unroll
                for (int j = 0; j < kEpiBatch; ++j) {
                    if (j >= nb) break;
                    const int o = obs[j] * kOB + row;
                    const float ws = F8 ? a.s_down[static_cast<size_t>(sg.e) * a.d + o] : 1.0f;   // W_down row scale
#pragma unroll
                    for (int t = 0; t < kNT; ++t)
                        if ((mask >> t) & 1u)
                            atomicAdd(a.y + static_cast<size_t>(t) * a.d + o, gt[t] * ws * __uint_as_float(r[j][t]));
                }
            }
        }
    } else {
        // ------------------------------------------------------------ h formers
        // One f row i per thread, up to kHRing runs ahead of the MMAs: the run's group
        // record (from the routing inputs, before the wait), then h = silu(g) * u of each
        // real sub-tile from the gate/up kernel's partial sums (after it), summed over the
        // item's CTA shares in order.
        const int i = static_cast<int>(threadIdx.x) - 192;   // 0..63
        const Split gsp{static_cast<long long>(G) * T * KB, gu_parts(G, T, gu_grid)};
        bool waited = false;
        uint32_t hround = 0;        // e4m3: rounds of the amax exchange, alternating scratch halves
        float hscale[kNT];          // e4m3: the run's h scale per token
#pragma unroll
        for (int t = 0; t < kNT; ++t) hscale[t] = 1.0f;
        uint32_t run = 0;
        for (long long b = lo; b < hi;) {
            const Seg sg = seg_at(a, b, hi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const uint32_t hb = run % kHRing, hph = (run / kHRing) & 1u;
            ++run;
            GroupInfo gi;
            group_tokens(a, sg.g, lane, gi);
            const int nreal = min(kDnSub, T - sg.tile * kDnSub);
            if (!warp_wait(bar_h_empty + 8u * hb, hph ^ 1u, abort_flag, a.err)) break;
            if (!waited) {
                pdl_wait();   // the partial sums are complete from here on
                waited = true;
            }
            uint8_t *const hp = h_ptr + hb * kHEntry;
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                if (((gi.mask >> (8 * h8)) & 0xFFu) == 0u) continue;   // no token in this half
                // eight tokens of every real sub-tile at a time: all loads first (predicated,
                // independent), then the sums
                float pg[kDnSub][8][kMaxSpan], pu[kDnSub][8][kMaxSpan];
#pragma unroll
                for (int sub = 0; sub < kDnSub; ++sub) {
                    const int tile = sg.tile * kDnSub + sub;
                    const bool real = sub < nreal;
                    const long long first = static_cast<long long>(sg.g * T + (real ? tile : 0)) * KB;
                    const int span = min(gsp.part_of(first + KB - 1) - gsp.part_of(first) + 1, kMaxSpan);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int t = 8 * h8 + j;
                        const bool on = real && ((gi.mask >> t) & 1u);
                        const float *const pp = part + part_index(gi.pos[t], T, real ? tile : 0, 0, i);
#pragma unroll
                        for (int sl = 0; sl < kMaxSpan; ++sl) {
                            const bool ld = on && sl < span;
                            pg[sub][j][sl] = ld ? pp[sl * 128] : 0.0f;
                            pu[sub][j][sl] = ld ? pp[sl * 128 + 64] : 0.0f;
                        }
                    }
                }
                if constexpr (!F8) {
#pragma unroll
                    for (int sub = 0; sub < kDnSub; ++sub) {
                        if (sub >= nreal) break;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int t = 8 * h8 + j;
                            if (!((gi.mask >> t) & 1u)) continue;
                            const float hv = silu(pg[sub][j][0] + pg[sub][j][1] + pg[sub][j][2]) *
                                             (pu[sub][j][0] + pu[sub][j][1] + pu[sub][j][2]);
                            // 128-byte swizzle: row t of 128 bytes, 16-byte chunk (i/8) ^ (t%8)
                            const uint32_t off = static_cast<uint32_t>(sub * kHBytes + (t >> 3) * 1024 + (t & 7) * 128 +
                                                                       (((i >> 3) ^ (t & 7)) << 4) + (i & 7) * 2);
                            *reinterpret_cast<__nv_bfloat16 *>(hp + off) = __float2bfloat16_rn(hv);
                        }
                    }
                } else {
                    // e4m3 h: each token's 128 values of the span share one scale, amax / 448,
                    // reduced over the 64 threads (two warps) before any value is rounded
                    float hv[kDnSub][8];
#pragma unroll
                    for (int sub = 0; sub < kDnSub; ++sub)
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            hv[sub][j] = silu(pg[sub][j][0] + pg[sub][j][1] + pg[sub][j][2]) *
                                         (pu[sub][j][0] + pu[sub][j][1] + pu[sub][j][2]);
                    float *const sc = scratch + (hround & 1u) * (2 * kNT);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float mx = fmaxf(fabsf(hv[0][j]), fabsf(hv[1][j]));
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
                        if (lane == 0) sc[(warp - 6) * kNT + j] = mx;
                    }
                    named_barrier(1, 64);
                    ++hround;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int t = 8 * h8 + j;
                        const float amax = fmaxf(sc[j], sc[kNT + j]);
                        const float hs = amax > 0.0f ? amax / 448.0f : 1.0f;
                        hscale[t] = hs;
                        if (!((gi.mask >> t) & 1u)) continue;
#pragma unroll
                        for (int sub = 0; sub < kDnSub; ++sub) {
                            const int fl = sub * 64 + i;   // column inside the 128-wide span
                            const uint32_t off = static_cast<uint32_t>((t >> 3) * 1024 + (t & 7) * 128 +
                                                                       (((fl >> 4) ^ (t & 7)) << 4) + (fl & 15));
                            hp[off] = f32_to_e4m3(hv[sub][j] / hs);
                        }
                    }
                }
            }
            if (i == 0) {
                uint32_t *const rec = reinterpret_cast<uint32_t *>(info_ptr + hb * kInfoBytes);
                rec[0] = gi.mask;
#pragma unroll
                for (int t = 0; t < kNT; ++t) rec[1 + t] = __float_as_uint(gi.gt[t]);
                if constexpr (F8) {
#pragma unroll
                    for (int t = 0; t < kNT; ++t) rec[17 + t] = __float_as_uint(hscale[t]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(bar_h_full + 8u * hb);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kDownTmemCols);
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D tensor map over a row-major [outer, inner] matrix of 2-byte (bf16) or 1-byte (e4m3
// codes) elements, 128-byte swizzle.  Coordinates and boxes are in elements.
bool encode_2d(CUtensorMap *map, const void *ptr, bool bytes1, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (bytes1 ? 1 : 2)};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, bytes1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    bool attr_set[2] = {false, false};
};

std::mutex g_info_mu;
DeviceInfo g_info[64];

template <bool F8>
cudaError_t set_attributes() {
    // the largest shared-memory carveout, so that a gate/up and a down CTA share an SM
    cudaError_t err = cudaFuncSetAttribute(expert_gu_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGUSmem);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(expert_gu_kernel<F8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(expert_down_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDnSmem);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(expert_down_kernel<F8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
    return err;
}

template <bool F8>
cudaError_t launch_pair(const ExpertArgs &a, int sms, int max_groups, bool zero_y, float *part, cudaStream_t s,
                        bool pdl) {
    using E = Elt<F8>;
    const long long T = a.f / kFTile, OBS = a.d / kOB;
    const int gu_grid = static_cast<int>(std::min<long long>(sms, 2ll * max_groups * T));
    const long long T2 = (T + kDnSub - 1) / kDnSub;
    const int dn_grid = static_cast<int>(std::min<long long>(sms, static_cast<long long>(max_groups) * T2 * OBS * E::UNIT));

    CUtensorMap tm_wg, tm_wu, tm_wd, tm_x;
    const uint64_t d = a.d, f = a.f, N = a.N;
    if (!encode_2d(&tm_wg, a.w_gate, F8, d, N * f, E::BK, kFTile) ||
        !encode_2d(&tm_wu, a.w_up, F8, d, N * f, E::BK, kFTile) ||
        !encode_2d(&tm_wd, a.w_down, F8, f, N * d, E::BK, kOB) ||
        !encode_2d(&tm_x, a.x, F8, d, static_cast<uint64_t>(a.n), E::BK, kNT))
        return cudaErrorInvalidValue;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(gu_grid));
    cfg.dynamicSmemBytes = kGUSmem;
    cudaError_t err = cudaLaunchKernelEx(&cfg, expert_gu_kernel<F8>, tm_wg, tm_wu, tm_x, a, part, zero_y ? 1 : 0);
    if (err != cudaSuccess) return err;
    cfg.gridDim = dim3(static_cast<unsigned>(dn_grid));
    cfg.blockDim = dim3(kDnThreads);
    cfg.dynamicSmemBytes = kDnSmem;
    return cudaLaunchKernelEx(&cfg, expert_down_kernel<F8>, tm_wd, a, static_cast<const float *>(part), gu_grid);
}

}  // namespace

bool expert_tc_supports(int d, int f) { return d % kOB == 0 && f % kFTile == 0 && d >= kOB && f >= kFTile; }

cudaError_t launch_expert_tc(const ExpertArgs &a, int max_groups, bool zero_y, float *part, cudaStream_t s,
                             bool pdl) {
    const bool f8 = a.w_dtype == MOE_E4M3 && a.x_dtype == MOE_E4M3;
    const bool bf = a.w_dtype == MOE_BF16 && a.x_dtype == MOE_BF16;
    if (!expert_tc_supports(a.d, a.f) || !(f8 || bf) || a.n > kNT || max_groups < 1) return cudaErrorNotSupported;
    // e4m3: 128-element k slices and 128-wide f spans
    if (f8 && (a.d % 128 != 0 || a.f % 128 != 0 || a.s_gate == nullptr || a.s_up == nullptr ||
               a.s_down == nullptr || a.s_x == nullptr))
        return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_info_mu);
        DeviceInfo &di = g_info[dev & 63];
        if (di.sms == 0) {
            err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
            if (err != cudaSuccess) return err;
        }
        if (!di.attr_set[f8 ? 1 : 0]) {
            err = f8 ? set_attributes<true>() : set_attributes<false>();
            if (err != cudaSuccess) return err;
            di.attr_set[f8 ? 1 : 0] = true;
        }
        sms = di.sms;
    }
    return f8 ? launch_pair<true>(a, sms, max_groups, zero_y, part, s, pdl)
              : launch_pair<false>(a, sms, max_groups, zero_y, part, s, pdl);
}

}  // namespace moe
