// expert_tc.cu -- the tensor-core (tcgen05 + TMA) kernel of the expert operation.
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
// (deduplicating form).  One call is one persistent kernel, one CTA per SM, 11 warps:
// warp 0 the TMA producer, warp 1 the tcgen05.mma issuer (with down units of four blocks,
// warp 10 a second one for every other down unit), warps 2-5 the epilogue (one TMEM lane per
// thread), warps 6-9 the h formers.  Every CTA streams its share of two block lists through one
// ring of shared-memory slots, without a break between them:
//
//   gate/up blocks.  A gate/up item is (group, 64-row tile of f); its block is one k slice:
//   64 rows of W_gate and the same 64 rows of W_up (16 KB, the M = 128 operand) plus the
//   pass's x for that slice (NT tokens, from L2).  All G*T*KB blocks are cut into equal
//   contiguous ranges, one per CTA, so every SM streams the same weight bytes whatever the
//   pass size and the number of groups.  A CTA accumulates the blocks of each item it
//   touches in TMEM (weights as M, tokens as N = NT, fp32) and stores the partial sums of
//   its share of the item to the workspace; with at most 2*G*T sharing CTAs an item meets
//   at most three of them.  Each partial sum is stored as one 64-bit word together with the
//   call's ticket, so the value is its own flag.
//
//   down blocks.  A down item is (group, two consecutive f tiles); its block is (item,
//   128-row block of d, tile): 128 rows of W_down by 64 columns (16 KB).  The blocks are
//   again cut into equal ranges.  The producer moves on to them as soon as its gate/up
//   blocks are issued, so the ring fills with W_down while the last gate/up sums are
//   formed elsewhere.  The h formers wait until the item's gate/up partial sums carry the
//   call's ticket and form h = silu(g) * u from them in a fixed order, as the B operand in its
//   swizzled layout (a large group's tokens split over up to four warps, each a round of
//   dependent L2 loads fewer), and the epilogue adds gate * (W_down h) into the fp32 output with
//   atomics: the weighted combine and the reduction over f tiles are fused there.
//
// The token width NT is 16 for passes of up to 16 tokens, 32 up to 32 and 64 above (the
// deduplicating forms, where a group may hold every token of the pass): the same kernel with
// NT-column accumulators, wider token masks and each warp's token table in shared memory.
//
// FP8 layers (e4m3 weights and x, one fp32 scale per weight row and per token) use the same
// kernel instantiated for kind::f8f6f4: a 128-byte row then holds 128 elements, so a
// gate/up block is a 128-wide k slice, a down block a 128-wide f slice, and a down item
// (two blocks per unit) spans 256 f.  The gate/up epilogue applies the row and token scales
// to its partial sums; the h formers quantize h per (token, item) with scale amax/448 (one
// scale for both blocks a unit accumulates), and the down epilogue applies that scale and
// the W_down row scale.
//
// The flags need no clearing between calls: every call takes a new ticket (the workspace's
// epoch word plus one), and the last CTA to start stores it back as the epoch.  All CTAs
// of a call are resident together (grid <= SMs, one CTA per SM, launch_dependents only
// after each CTA started), and every wait, on an mbarrier or on a flag, is bounded: a
// time-out raises an abort flag that every role honours, records MOE_ERR_DEVICE_TIMEOUT,
// drains copies and MMAs in flight and frees TMEM before the CTA exits.
#include "common.cuh"
#include "expert_args.cuh"

#include <algorithm>
#include <mutex>

namespace moe {
namespace {

// warps: producer, MMA, 4 epilogue, 4 h formers, a second MMA issuer for the down phase
constexpr int kThreads = 352;
constexpr int kWarps = kThreads / 32;
constexpr int kHWarps = 4;                    // h-former warps (6 .. 9)
constexpr int kMma2Warp = 10;                 // issues every other down unit of 4-block units
constexpr int kOB = 128;                      // d rows per down block
constexpr uint32_t kWBytes = 16384;           // weight bytes of one block
constexpr long long kDrainCycles = 400000000ll;   // about 0.2 s
// the grouping of the deduplicating form from ids: expert list, offsets, slot order, the count,
// two scan scratch rows, a copy of the ids (then the per-expert counts, N <= 1024)
constexpr uint32_t kGrpWords = 3 * kMaxFusedSlots + 1 + 1 + 2 * kWarps + kMaxFusedSlots;

// Token width NT of an instantiation: the MMA N, the rows of an x or h tile and the TMEM
// columns of an accumulator.  16 serves passes of up to 16 tokens; 32 and 64 serve the
// deduplicating forms up to 32 and 64 tokens, where one group can hold every token of the
// pass.  A weight block stays 16 KB, but the x tile that rides with it and the h tiles grow
// with NT, so the wide forms keep a ring as deep as shared memory allows: a slot is held
// from its copy's issue until its MMAs complete, and the copies in flight per SM must cover
// the memory latency at the stream's rate.
//
// The h ring needs no entry per h-former warp.  Its producers are kHWarps warps that each
// form only some runs, and a warp forming run r first waits, with a parity wait, for the
// release of run r - kHRing from its entry.  That wait is exact once run r - 2 * kHRing is
// released (the entry is then at most one phase behind; it cannot be ahead, as run r is not
// formed yet).  A warp knows that from its own last wait when it took part in one of the
// kHRing runs before r; any kHWarps consecutive runs give every warp a part, so with
// kHRing >= kHWarps that always holds.  With fewer entries than warps it need not (a warp
// relying on its own waits alone could pass a whole phase early), so those forms keep a shared
// count of the runs known to be released: every warp that passes an entry's wait for run r
// raises it to r - kHRing + 1, and a warp waits for it to cover run r - 2 * kHRing before its
// parity wait for run r.  Releases complete in run order (each issuer's commit covers all its
// earlier MMAs, and the epilogue warps arrive run by run), so one seen release implies all
// earlier ones.  (Waiting for every run's entry in order, also for the runs a warp skips, is
// not enough: a skipping warp can fall behind an entry that others have released twice.)
template <int NT>
struct Cfg;
template <>
struct Cfg<16> {
    // ring slots: 8 keeps enough copies in flight for the full stream (about 130 KB per SM)
    // while every dependent round trip waits behind fewer of them (11 and 6 measured slower)
    static constexpr int kStages = 8;
    static constexpr int kDownBufs = 8;       // TMEM ring of down-block accumulators
    static constexpr int kEpiBatch = 4;       // down accumulators per epilogue round
    static constexpr int kHRing = 4;          // h entries (one per down run in flight)
    static constexpr int kGuBufs = 4;         // TMEM ring of gate/up item accumulators
    static constexpr uint32_t kTmemCols = 256;
    using Mask = uint32_t;                    // a group's tokens
};
template <>
struct Cfg<32> {
    static constexpr int kStages = 8;
    static constexpr int kDownBufs = 8;
    static constexpr int kEpiBatch = 2;       // 2 x 32 columns: the registers of 4 x 16
    static constexpr int kHRing = 4;
    static constexpr int kGuBufs = 4;
    static constexpr uint32_t kTmemCols = 512;
    using Mask = uint32_t;
};
template <>
struct Cfg<64> {
    static constexpr int kStages = 7;
    static constexpr int kDownBufs = 6;
    static constexpr int kEpiBatch = 1;
    static constexpr int kHRing = 2;
    static constexpr int kGuBufs = 2;
    static constexpr uint32_t kTmemCols = 512;
    using Mask = uint64_t;
};

// Shared memory of an instantiation (token width NT, U down blocks per TMEM accumulator, a
// unit): the ring, kHRing h entries, their run records, each
// epilogue warp's copy of the token scales (FP8) and of its run's gates, the token tables
// of the wide form (below), then barriers full[S], empty[S], gacc_full[G], gacc_empty[G],
// dacc_full[B], dacc_empty[B], h_full[R], h_empty[R], drain[2], the misc words, the ring slots'
// block records, the in-kernel grouping and the per-expert counts.
template <int NT, int U>
struct Lay : Cfg<NT> {
    using C = Cfg<NT>;
    // units of 4 blocks take h entries twice as large: the 32-token form keeps 2 of them, the
    // 64-token form one ring slot fewer
    static constexpr int kStages = (NT == 64 && U == 4) ? C::kStages - 1 : C::kStages;
    static constexpr int kHRing = (NT == 32 && U == 4) ? 2 : C::kHRing;
    static constexpr uint32_t kXTileBytes = NT * 128;   // x of one k slice: NT rows x 128 B
    static constexpr uint32_t kSlotBytes = kWBytes + kXTileBytes;   // gate/up block + x, or down block
    static constexpr uint32_t kHBytes = NT * 128;       // one h tile: NT rows x 128 B
    static constexpr uint32_t kHEntry = U * kHBytes;
    // a run record: the token mask (2 words), the NT gates, the NT h scales (FP8)
    static constexpr uint32_t kInfoBytes = ((2 + 2 * NT) * 4 + 15) & ~15u;
    static constexpr uint32_t kDnCol0 = NT * C::kGuBufs;   // gate/up accumulators first, then down
    static constexpr uint32_t kHOff = kStages * kSlotBytes;
    static constexpr uint32_t kInfoOff = kHOff + kHRing * kHEntry;
    static constexpr uint32_t kSxOff = kInfoOff + kHRing * kInfoBytes;
    static constexpr uint32_t kGwOff = kSxOff + 4 * NT * 4;
    // wide form: slot positions and summed gates of the current group of each epilogue and
    // h-former warp (the 16-token form keeps them in registers)
    static constexpr uint32_t kTabOff = kGwOff + 4 * NT * 4;
    static constexpr uint32_t kTabBytes = NT == 16 ? 0u : 8u * NT * 8u;
    static constexpr uint32_t kBarOff = kTabOff + kTabBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * C::kGuBufs + 2 * C::kDownBufs + 2 * kHRing + 2;
    static constexpr uint32_t kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr uint32_t kRecOff = kMiscOff + 16;   // the block each ring slot last received
    static constexpr uint32_t kGrpOff = kRecOff + ((4 * kStages + 15) & ~15u);
    static constexpr uint32_t kCntOff = kGrpOff + ((kGrpWords * 4 + 15) & ~15u);
    static constexpr uint32_t kSmem = kCntOff + 1024 * 4 + 1024;   // + alignment slack of the base
    static_assert(kSlotBytes % 1024 == 0 && kHOff % 1024 == 0 && kHEntry % 1024 == 0, "128-byte swizzle atoms");
    static_assert(kBarOff % 8 == 0, "mbarrier alignment");
    static_assert(kSmem <= 232448, "shared memory of one CTA");
    static_assert(4 * kThreads >= 1024 && kThreads >= kMaxFusedSlots && kHWarps >= 1 && kHWarps <= NT,
                  "grouping bins and slots, h-former warps");
    static_assert(kDnCol0 + NT * C::kDownBufs <= C::kTmemCols, "TMEM columns");
    // units alternate between the two MMA issuers: with an even count every down accumulator
    // belongs to one issuer, whose waits on it then follow each other phase by phase
    static_assert(C::kDownBufs % 2 == 0, "down accumulators per issuer");
    static_assert(NT % 16 == 0 && NT <= 64 && sizeof(typename C::Mask) * 8 >= NT, "token width");
};

// Element type of a kernel instantiation: bf16 (kind::f16) or e4m3 (kind::f8f6f4), with
// token width NT and U down blocks per accumulator.
template <bool F8, int NT, int U>
struct Elt {
    static constexpr int BK = F8 ? 128 : 64;   // k elements per 128-byte row of an operand tile
    static constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(128, NT) : idesc_bf16_f32(128, NT);
    // a down block spans TPB 64-row gate/up tiles of f (one 128-byte row of W_down: 64 bf16 or
    // 128 e4m3), a unit U blocks, a down item ITEM tiles: 128 or 256 f (bf16, U = 2 or 4), 256 f
    // (e4m3, U = 2: the span of one h scale)
    static constexpr int TPB = F8 ? 2 : 1;
    static constexpr int UNIT = U;
    static constexpr int ITEM = U * TPB;
    static constexpr int COLS = ITEM * 64 / 32;   // f columns of an item per h-former lane
    // tokens per round of the h formers' loads: the 64-bit tagged words of 2 tokens fit the
    // registers at 4 columns a lane, of 1 at 8
    static constexpr int TK = COLS > 4 ? 1 : 2;
    static_assert(!F8 || U == 2, "e4m3 items span 256 f, the h scale's block");
    __device__ __forceinline__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
        if constexpr (F8) tc_mma_f8(d, a, b, IDESC, acc);
        else tc_mma_bf16(d, a, b, IDESC, acc);
    }
};
constexpr uint32_t kFull = 0xFFFFFFFFu;

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
// it with ballots, so a group of k slots costs one round trip to memory, not k.  The
// 16-token form keeps the gates and positions in registers; the wide form in a table of
// the warp's own in shared memory (gt and pos point there).
template <int NT>
struct GroupInfo {
    typename Cfg<NT>::Mask mask;
    float *gt;
    int *pos;
};
template <>
struct GroupInfo<16> {
    uint32_t mask;
    float gt[16];
    int pos[16];
};

__device__ __forceinline__ void group_tokens(const ExpertArgs &a, int g, int lane, GroupInfo<16> &gi) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        gi.gt[t] = 0.0f;
        gi.pos[t] = 0;
    }
    if (a.mode == kModePerSlot) {
        const int tt = g / a.m;
        const float gv = a.gates[g];
#pragma unroll
        for (int t = 0; t < 16; ++t)
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
        for (int t = 0; t < 16; ++t) {
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

// The wide form: lanes holding the same token find each other with one match instead of a
// ballot per token; the highest of them keeps the token's position and the gates' sum (in
// ascending lane order, as above).  Only the mask's entries of the table are written.
template <int NT>
__device__ __forceinline__ void group_tokens(const ExpertArgs &a, int g, int lane, GroupInfo<NT> &gi) {
    using Mask = typename Cfg<NT>::Mask;
    __syncwarp();   // every lane has read the previous group's table
    if (a.mode == kModePerSlot) {
        const int tt = g / a.m;
        if (lane == 0) {
            gi.gt[tt] = a.gates[g];
            gi.pos[tt] = g;
        }
        gi.mask = static_cast<Mask>(1) << tt;
        __syncwarp();
        return;
    }
    const int S = a.n * a.m;   // offsets are clamped to the slot buffer; slot < S gives token < n <= NT
    const int p0 = max(0, a.offsets[g]), p1 = min(S, a.offsets[g + 1]);
    Mask mask = 0;
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
        const uint32_t peers = __match_any_sync(kFull, tt >= 0 ? tt : -1 - lane);
        const int rounds = static_cast<int>(__reduce_max_sync(kFull, static_cast<uint32_t>(__popc(peers))));
        float sum = 0.0f;
        uint32_t rest = peers;
        for (int r = 0; r < rounds; ++r) {
            const float v = __shfl_sync(kFull, gv, rest ? __ffs(rest) - 1 : lane);
            if (rest) {
                sum += v;
                rest &= rest - 1u;
            }
        }
        if (tt >= 0 && lane == 31 - __clz(peers)) {
            const bool again = (mask >> tt) & 1u;   // a repeated token met in an earlier round
            gi.gt[tt] = again ? gi.gt[tt] + sum : sum;
            gi.pos[tt] = p;
        }
        const uint32_t lo = __reduce_or_sync(kFull, tt >= 0 && tt < 32 ? 1u << tt : 0u);
        if constexpr (sizeof(Mask) == 8) {
            const uint32_t hi = __reduce_or_sync(kFull, tt >= 32 ? 1u << (tt - 32) : 0u);
            mask |= (static_cast<uint64_t>(hi) << 32) | lo;
        } else {
            mask |= lo;
        }
        __syncwarp();
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

// Tagged partial sums: a value's fp32 bits in the low word and the call's ticket in the high
// word, stored and loaded as one aligned 64-bit access, which is single-copy atomic.  A reader
// that finds its call's ticket in a word has the value that was stored with it: the data is its
// own flag, so no release store and no separate flag sit between a gate/up share and the h
// formers waiting for it.  Words from earlier calls carry older tickets and never match.
__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t ticket) {
    const uint64_t w = (static_cast<uint64_t>(ticket) << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t *p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ bool tag_is(uint64_t w, uint32_t ticket) { return static_cast<uint32_t>(w >> 32) == ticket; }
__device__ __forceinline__ float tagged_value(uint64_t w) { return __uint_as_float(static_cast<uint32_t>(w)); }

// The call's ticket: the epoch word plus one, never 0 (zeroed flags never match it).
__device__ __forceinline__ uint32_t call_ticket(const uint32_t *sync) {
    const uint32_t t = ld_acquire_gpu(sync) + 1u;
    return t == 0u ? 1u : t;
}

// The k-th token (ascending) of a token mask, or a value >= 64 when it has fewer.
__device__ __forceinline__ uint32_t nth_token(uint32_t mask, int k) { return __fns(mask, 0u, k + 1); }
__device__ __forceinline__ uint32_t nth_token(uint64_t mask, int k) {
    const uint32_t lo = static_cast<uint32_t>(mask);
    const int nl = __popc(lo);
    if (k < nl) return __fns(lo, 0u, k + 1);
    const uint32_t r = __fns(static_cast<uint32_t>(mask >> 32), 0u, k - nl + 1);
    return r == 0xFFFFFFFFu ? r : 32u + r;
}
__device__ __forceinline__ int mask_count(uint32_t mask) { return __popc(mask); }
__device__ __forceinline__ int mask_count(uint64_t mask) { return __popcll(mask); }
// The token mask of a run record (words 0 and 1).
template <typename Mask>
__device__ __forceinline__ Mask run_mask(const uint32_t *rec) {
    if constexpr (sizeof(Mask) == 4) return rec[0];
    else return static_cast<uint64_t>(rec[0]) | (static_cast<uint64_t>(rec[1]) << 32);
}

// The grouping of the deduplicating form (the counting sort of moe_group_slots): experts in
// ascending order with their slot offsets, slots of an expert in ascending order; ids outside
// [0, N) are left out of every group.  All threads of the CTA take part; thread s holds the id
// of slot s (S <= kMaxFusedSlots <= kThreads), loaded by the caller, and ids_s receives a copy.
// On return the expert list, offsets and count are visible to every thread, the slot order to
// warps 2 and up.
__device__ void build_grouping(const ExpertArgs &a, int my_id, int32_t *lst, int32_t *off, int32_t *ord,
                               int32_t *cnt, int32_t *g_out, int32_t *scan, int32_t *ids_s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = a.N, S = a.n * a.m;
    for (int i = tid; i < N; i += kThreads) cnt[i] = 0;
    if (tid < S) ids_s[tid] = my_id;
    __syncthreads();
    bool bad = false;
    if (tid < S) {
        if (my_id >= 0 && my_id < N) atomicAdd(&cnt[my_id], 1);
        else bad = true;
    }
    if (__syncthreads_or(bad) && tid == 0 && blockIdx.x == 0) record_error(a.err, MOE_ERR_BAD_ID);
    // thread tid owns bins [4 tid, 4 tid + 4): exclusive scans of the slot counts and of the
    // non-empty bins over the CTA
    int c[4], cs = 0, ne = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = 4 * tid + j;
        c[j] = b < N ? cnt[b] : 0;
        cs += c[j];
        ne += c[j] > 0 ? 1 : 0;
    }
    int is = cs, in = ne;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int us = __shfl_up_sync(kFull, is, o), un = __shfl_up_sync(kFull, in, o);
        if (lane >= o) {
            is += us;
            in += un;
        }
    }
    if (lane == 31) {
        scan[warp] = is;
        scan[kWarps + warp] = in;
    }
    __syncthreads();
    int es = is - cs, en = in - ne, tot_s = 0, tot_n = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) {
            es += scan[w];
            en += scan[kWarps + w];
        }
        tot_s += scan[w];
        tot_n += scan[kWarps + w];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = 4 * tid + j;
        if (c[j] > 0) {
            lst[en] = b;
            off[en] = es;
            cnt[b] = es;   // the bin's next free position
            ++en;
        }
        es += c[j];
    }
    if (tid == 0) {
        *g_out = tot_n;
        off[tot_n] = tot_s;
    }
    __syncthreads();
    // Stable scatter of the slots, 32 at a time in ascending order, by the first h-former warp.
    // Only the epilogue and the h formers read the slot order (warps 2 ..), so the producer and
    // the MMA warp go on with the expert list and the offsets.
    if (warp == 6) {
        for (int c0 = 0; c0 < S; c0 += 32) {
            const int s = c0 + lane;
            const int e = s < S ? ids_s[s] : -1;
            const bool v = e >= 0 && e < N;
            const uint32_t peers = __match_any_sync(kFull, v ? e : -2 - lane);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int base = v ? cnt[e] : 0;
            if (v) ord[base + rank] = s;
            __syncwarp();
            if (v && rank == 0) cnt[e] = base + __popc(peers);
            __syncwarp();
        }
    }
    if (warp >= 2) named_barrier(3, kThreads - 64);
}

// Bounded warp-wide wait until the shared word *p holds v: the same abort and time-limit rules
// as mbar_wait, and the outcome is warp-uniform.
__device__ __forceinline__ bool warp_wait_word(const volatile uint32_t *p, uint32_t v, volatile int32_t *abort,
                                               int32_t *err, long long limit) {
    if (__all_sync(kFull, *p == v)) return true;
    const long long t0 = clock64();
    while (true) {
        if (__all_sync(kFull, *p == v)) return true;
        const bool late = clock64() - t0 > limit;
        if (__any_sync(kFull, late || *abort != 0)) {
            if (late && (threadIdx.x & 31) == 0) {
                *abort = 1;
                record_error(err, MOE_ERR_DEVICE_TIMEOUT);
            }
            return false;
        }
    }
}

// Bounded warp-wide wait until the shared count *p is at least v (it only grows): the same
// abort and time-limit rules as mbar_wait, and the outcome is warp-uniform.
__device__ __forceinline__ bool warp_wait_at_least(const uint32_t *p, uint32_t v, volatile int32_t *abort,
                                                   int32_t *err, long long limit) {
    const volatile uint32_t *const q = p;
    if (__all_sync(kFull, *q >= v)) return true;
    const long long t0 = clock64();
    while (true) {
        if (__all_sync(kFull, *q >= v)) return true;
        const bool late = clock64() - t0 > limit;
        if (__any_sync(kFull, late || *abort != 0)) {
            if (late && (threadIdx.x & 31) == 0) {
                *abort = 1;
                record_error(err, MOE_ERR_DEVICE_TIMEOUT);
            }
            return false;
        }
    }
}

// ==================================================================== the kernel

template <bool F8, int NT, int U>
__global__ void __launch_bounds__(kThreads, 1)
expert_tc_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                 const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_x,
                 const ExpertArgs a, uint64_t *const part, const int zero_y) {
    using L = Lay<NT, U>;
    using Mask = typename L::Mask;
    constexpr int kStages = L::kStages, kDownBufs = L::kDownBufs, kEpiBatch = L::kEpiBatch;
    constexpr int kIssuers = U == 4 ? 2 : 1;   // MMA issuers of the down phase
    constexpr int kHRing = L::kHRing, kGuBufs = L::kGuBufs;
    constexpr uint32_t kSlotBytes = L::kSlotBytes, kHBytes = L::kHBytes, kHEntry = L::kHEntry;
    constexpr uint32_t kInfoBytes = L::kInfoBytes, kDnCol0 = L::kDnCol0, kTmemCols = L::kTmemCols;
    constexpr uint32_t kHOff = L::kHOff, kInfoOff = L::kInfoOff, kBarOff = L::kBarOff, kMiscOff = L::kMiscOff;
    constexpr int kRoundUnroll = NT == 16 ? 16 : 1;   // the h formers' rounds of token loads
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw_addr);
    const uint32_t sh = base + kHOff;
    uint8_t *const h_ptr = base_ptr + kHOff;
    uint8_t *const info_ptr = base_ptr + kInfoOff;
    const uint32_t bar_full = base + kBarOff;
    const uint32_t bar_empty = bar_full + 8u * kStages;
    const uint32_t bar_gacc_full = bar_empty + 8u * kStages;       // [kGuBufs]
    const uint32_t bar_gacc_empty = bar_gacc_full + 8u * kGuBufs;  // [kGuBufs]
    const uint32_t bar_dacc_full = bar_gacc_empty + 8u * kGuBufs;  // [kDownBufs]
    const uint32_t bar_dacc_empty = bar_dacc_full + 8u * kDownBufs;  // [kDownBufs]
    const uint32_t bar_h_full = bar_dacc_empty + 8u * kDownBufs;   // [kHRing]
    const uint32_t bar_h_empty = bar_h_full + 8u * kHRing;         // [kHRing]
    const uint32_t bar_drain = bar_h_empty + 8u * kHRing;
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + kMiscOff);
    volatile int32_t *const abort_flag = reinterpret_cast<volatile int32_t *>(base_ptr + kMiscOff + 4);
    // runs below this are known to be released from the h ring (forms with kHRing < kHWarps)
    uint32_t *const h_seen = reinterpret_cast<uint32_t *>(base_ptr + kMiscOff + 8);
    volatile uint32_t *const slot_rec = reinterpret_cast<volatile uint32_t *>(base_ptr + L::kRecOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long wl = a.wait_limit;   // cycles before a wait gives up

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int b = 0; b < kGuBufs; ++b) {
            mbar_init(bar_gacc_full + 8u * b, 1);
            mbar_init(bar_gacc_empty + 8u * b, 4);      // the 4 epilogue warps
        }
        for (int b = 0; b < kDownBufs; ++b) {
            mbar_init(bar_dacc_full + 8u * b, 1);
            mbar_init(bar_dacc_empty + 8u * b, 4);      // the 4 epilogue warps
        }
        for (int b = 0; b < kHRing; ++b) {
            mbar_init(bar_h_full + 8u * b, kHWarps);    // the run's leader for kHWarps - W + 1, each helper 1
            mbar_init(bar_h_empty + 8u * b, kIssuers + 4);   // the MMA issuers' commits and the epilogue warps
        }
        mbar_init(bar_drain, 1);
        mbar_init(bar_drain + 8u, 1);
        for (int s = 0; s < kStages; ++s) slot_rec[s] = ~0u;
        *h_seen = 0u;
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tm_wg);
        tma_prefetch_map(&tm_wu);
        tma_prefetch_map(&tm_wd);
        tma_prefetch_map(&tm_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Before waiting for the preceding grid: warm L2 and the address translation for the small
    // inputs every CTA reads first (ids, gates, the grouping, x).  Their values are read only
    // after the wait.
    {
        const int S = a.n * a.m, tid = static_cast<int>(threadIdx.x);
        const size_t xb = static_cast<size_t>(a.n) * a.d * (F8 ? 1 : 2);
        prefetch_l2_range(a.ids, static_cast<size_t>(S) * 4, tid, kThreads);
        prefetch_l2_range(a.gates, static_cast<size_t>(S) * 4, tid, kThreads);
        prefetch_l2_range(a.x, xb, tid, kThreads);
        if (a.mode == kModeDedup) {   // the grouping's buffer sizes, as the host validated them
            const int nd = S < a.N ? S : a.N;   // at most this many distinct experts
            prefetch_l2_range(a.expert_list, static_cast<size_t>(nd) * 4, tid, kThreads);
            prefetch_l2_range(a.offsets, static_cast<size_t>(nd + 1) * 4, tid, kThreads);
            prefetch_l2_range(a.slot_order, static_cast<size_t>(S) * 4, tid, kThreads);
        }
    }
    // Every thread waits for the grids this one depends on before reading any input.  The
    // next grid may launch once every CTA of this one has passed this point, so a CTA that
    // waits for another CTA's flag never holds an SM that CTA still needs.
    pdl_wait();
    pdl_trigger();
    // The deduplicating form from ids: thread s loads the id of slot s now, so that the load
    // is in flight together with the epoch read below.
    int my_id = -1;
    if (a.mode == kModeDedupIds && static_cast<int>(threadIdx.x) < a.n * a.m) my_id = a.ids[threadIdx.x];
    // The call's ticket, read by the warps that publish or wait for flags (2 ..).  Once all of
    // them hold it, the CTA counts itself in (below, off the path to the first copies); the
    // last CTA of the grid to do so stores the ticket as the new epoch, which no CTA of this
    // call reads any more (each one read the epoch before its count, and the acquire-release
    // count orders that read before the store).  The next call reads it after this grid is
    // complete.
    uint32_t ticket = 0;
    if (warp >= 2) {
        ticket = call_ticket(a.sync);
        named_barrier(1, kThreads - 64);
    }

    // The routing every role reads: the call's, or, for the deduplicating form from ids, the
    // grouping this CTA builds here (the same in every CTA).
    ExpertArgs ar = a;
    // A one-token pass whose m ids are distinct and in range (as top-m routing gives them) is
    // its own grouping: each slot is one distinct expert with one token, so the deduplicating
    // form reads exactly what the per-slot schedule reads and computes the same sums.  Every
    // warp checks the ids itself (the same data, so the same answer), and no grouping is built.
    bool own_grouping = false;
    if (a.mode == kModeDedupIds && a.n == 1 && a.m <= 32) {
        const bool in = lane < a.m;
        const int e = in ? a.ids[lane] : -1;
        const uint32_t active = __ballot_sync(kFull, in);
        const uint32_t peers = __match_any_sync(kFull, in ? e : -1 - lane);
        own_grouping = __all_sync(kFull, !in || (e >= 0 && e < a.N && peers == (1u << lane))) && active != 0u;
    }
    if (own_grouping) {
        ar.mode = kModePerSlot;
    } else if (a.mode == kModeDedupIds) {
        int32_t *const grp = reinterpret_cast<int32_t *>(base_ptr + L::kGrpOff);
        int32_t *const lst = grp, *const off = grp + kMaxFusedSlots, *const ord = grp + 2 * kMaxFusedSlots + 1;
        int32_t *const gcount = grp + 3 * kMaxFusedSlots + 1, *const scan = gcount + 1;
        int32_t *const ids_s = scan + 2 * kWarps;
        build_grouping(a, my_id, lst, off, ord, reinterpret_cast<int32_t *>(base_ptr + L::kCntOff), gcount, scan, ids_s);
        ar.mode = kModeDedup;
        ar.expert_list = lst;
        ar.offsets = off;
        ar.slot_order = ord;
        ar.num_distinct = gcount;
    }
    // the CTA's count, after every warp of it read the epoch (the named barrier above)
    if (warp == kWarps - 1 && lane == 0 && atom_add_acq_rel_gpu(a.sync + 1, 1u) == gridDim.x - 1) {
        a.sync[1] = 0u;
        st_release_gpu(a.sync, ticket);
    }

    using E = Elt<F8, NT, U>;
    const int T = a.f / kFTile;
    const int KB = a.d / E::BK;
    const int G = num_groups(ar);
    const int c = blockIdx.x;
    const int P = gridDim.x;
    // gate/up blocks: G*T items of KB k slices
    const Split gsp{static_cast<long long>(G) * T * KB, gu_parts(G, T, P)};
    const long long glo = c < gsp.parts ? gsp.lo(c) : 0, ghi = c < gsp.parts ? gsp.lo(c + 1) : 0;
    // down blocks: G*T2 items of IB blocks, (d block ob, sub-tile s) with s innermost, so the
    // sub-tiles of one d block accumulate in one TMEM accumulator: a unit.  The last item of
    // a group has fewer real blocks when T is not a multiple of E::ITEM; the others are
    // skipped by every role alike.
    const int T2 = (T + E::ITEM - 1) / E::ITEM;
    const int OBS = a.d / kOB;
    const int IB = OBS * E::UNIT;
    const long long nblk = static_cast<long long>(G) * T2 * IB;
    const Split dsp{nblk, static_cast<int>(nblk < 1 ? 1 : (nblk < P ? nblk : P))};
    const long long dlo = c < dsp.parts ? dsp.lo(c) : 0, dhi = c < dsp.parts ? dsp.lo(c + 1) : 0;
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
        // the item's real blocks: the last item of a group may have one (f not a multiple of
        // 128 for bf16, of 256 for e4m3)
        u.nreal = min(E::ITEM, T - sg.tile * E::ITEM) / E::TPB;
        return u;
    };

    uint32_t prod_cnt = 0;   // copies the producer issued
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the schedule and waits; one elected lane issues the copies.
        uint32_t cnt = 0;
        bool ok = true;
        for (long long b = glo; ok && b < ghi;) {
            const Seg s = seg_at(ar, b, ghi, KB, T);
            b = s.b1;
            if (!s.valid) continue;
            const int row = s.e * a.f + s.tile * kFTile;
            for (long long bb = s.b0; bb < s.b1; ++bb) {
                const uint32_t st = cnt % kStages, ph = (cnt / kStages) & 1u;
                if (!warp_wait(bar_empty + 8u * st, ph ^ 1u, abort_flag, a.err, wl)) {
                    ok = false;
                    break;
                }
                const int k0 = static_cast<int>(bb - static_cast<long long>(s.item) * KB) * E::BK;
                if (elect_one()) {
                    const uint32_t dst = base + st * kSlotBytes, fb = bar_full + 8u * st;
                    mbar_arrive_expect_tx(fb, kSlotBytes);
                    tma_load_2d(dst, &tm_wg, fb, k0, row);
                    tma_load_2d(dst + kWBytes / 2, &tm_wu, fb, k0, row);
                    tma_load_2d(dst + kWBytes, &tm_x, fb, k0, 0);
                }
                __syncwarp();
                ++cnt;
            }
        }
        for (long long b = dlo; ok && b < dhi;) {
            const Seg sg = seg_at(ar, b, dhi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const Units u = units_of(sg);
            for (int ob = u.ob_first(); ok && ob <= u.ob_last(); ++ob) {
                for (int sub = u.s_lo(ob); sub < u.s_hi(ob); ++sub) {
                    const uint32_t st = cnt % kStages, ph = (cnt / kStages) & 1u;
                    if (!warp_wait(bar_empty + 8u * st, ph ^ 1u, abort_flag, a.err, wl)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        const uint32_t fb = bar_full + 8u * st;
                        if (kIssuers == 2) slot_rec[st] = cnt;   // before the phase of block cnt can complete
                        mbar_arrive_expect_tx(fb, kWBytes);
                        tma_load_2d(base + st * kSlotBytes, &tm_wd, fb, (sg.tile * E::ITEM + sub * E::TPB) * kFTile,
                                    sg.e * a.d + ob * kOB);
                    }
                    __syncwarp();
                    ++cnt;
                }
            }
        }
        prod_cnt = cnt;
        __syncwarp();
    } else if (warp == 1 || (kIssuers == 2 && warp == kMma2Warp)) {
        // ------------------------------------------------------------ MMA issuers
        // Warp-uniform loops; waits by every lane, MMAs and commits by one elected lane.  A
        // round of waits and issue costs about as much as four MMAs of its own, so a round
        // takes the next block of the same accumulator as well when its copy has already landed
        // (a non-blocking test): eight MMAs back to back where the stream runs ahead of the
        // issuer, and no wait added where the issuer waits for the stream.  Warp 1 issues the
        // gate/up blocks.  With units of four blocks the down units alternate between warp 1 and
        // warp 10 (each into its own accumulators), so two issuers feed the down phase; with
        // units of two warp 1 issues them all (two issuers were no faster there).
        const uint32_t mw = warp == 1 ? 0u : 1u;   // this issuer's down units: dcnt % 2 == mw
        uint32_t cnt = 0, seg = 0;
        bool ok = true;
        if (mw == 1u) {
            // the down blocks follow this CTA's gate/up blocks in the ring
            for (long long b = glo; b < ghi;) {
                const Seg s = seg_at(ar, b, ghi, KB, T);
                b = s.b1;
                if (s.valid) cnt += static_cast<uint32_t>(s.b1 - s.b0);
            }
        }
        for (long long b = glo; mw == 0u && ok && b < ghi;) {
            const Seg s = seg_at(ar, b, ghi, KB, T);
            b = s.b1;
            if (!s.valid) continue;
            const uint32_t buf = seg % kGuBufs, sph = (seg / kGuBufs) & 1u;
            ++seg;
            if (!warp_wait(bar_gacc_empty + 8u * buf, sph ^ 1u, abort_flag, a.err, wl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + NT * buf;
            for (long long bb = s.b0; bb < s.b1;) {
                uint32_t st[2] = {cnt % kStages, (cnt + 1) % kStages};
                if (!warp_wait(bar_full + 8u * st[0], (cnt / kStages) & 1u, abort_flag, a.err, wl)) {
                    ok = false;
                    break;
                }
                const int nbk = (s.b1 - bb >= 2 && __all_sync(kFull, mbar_test_wait(bar_full + 8u * st[1],
                                                                                   ((cnt + 1) / kStages) & 1u)))
                                    ? 2 : 1;   // blocks of this round
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (j >= nbk) break;
                        const uint32_t sa = base + st[j] * kSlotBytes;
                        const uint32_t sb = sa + kWBytes;
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // 32 bytes of K per instruction
                            E::mma(d_tmem, desc_kmajor_sw128(sa + 32u * k), desc_kmajor_sw128(sb + 32u * k),
                                   (bb + j != s.b0 || k != 0) ? 1u : 0u);
                        tc_commit(bar_empty + 8u * st[j]);   // each slot as soon as its own MMAs are done
                    }
                    if (bb + nbk == s.b1) tc_commit(bar_gacc_full + 8u * buf);
                }
                __syncwarp();
                cnt += nbk;
                bb += nbk;
            }
        }
        uint32_t dcnt = 0, run = 0;
        for (long long b = dlo; ok && b < dhi;) {
            const Seg sg = seg_at(ar, b, dhi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const Units u = units_of(sg);
            const uint32_t hb = run % kHRing, hph = (run / kHRing) & 1u;
            ++run;
            if (!warp_wait(bar_h_full + 8u * hb, hph, abort_flag, a.err, wl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t shb = sh + hb * kHEntry;
            for (int ob = u.ob_first(); ok && ob <= u.ob_last(); ++ob) {
                const int s0 = u.s_lo(ob), s1 = u.s_hi(ob);
                if (s0 >= s1) continue;
                const uint32_t du = dcnt++;
                if (kIssuers == 2 && (du & 1u) != mw) {   // the other issuer's unit: its blocks pass by
                    cnt += static_cast<uint32_t>(s1 - s0);
                    continue;
                }
                const uint32_t buf = du % kDownBufs, dph = (du / kDownBufs) & 1u;
                if (!warp_wait(bar_dacc_empty + 8u * buf, dph ^ 1u, abort_flag, a.err, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // The unit's blocks (at most E::UNIT), in rounds as above.  Each issuer skips the
                // other's blocks, so the copy into a slot that precedes this block's may not have
                // been issued yet, and a parity wait would then take that earlier phase for this
                // block's: the wait starts once the producer has recorded this block in the slot.
                for (int sub = s0; sub < s1;) {
                    if ((kIssuers == 2 && !warp_wait_word(slot_rec + cnt % kStages, cnt, abort_flag, a.err, wl)) ||
                        !warp_wait(bar_full + 8u * (cnt % kStages), (cnt / kStages) & 1u, abort_flag, a.err, wl)) {
                        ok = false;
                        break;
                    }
                    // the unit's next blocks join the round while their copies have landed
                    int nbk = 1;
#pragma unroll
                    for (int j = 1; j < E::UNIT; ++j)
                        if (nbk == j && s1 - sub > j &&
                            __all_sync(kFull, (kIssuers == 1 || slot_rec[(cnt + j) % kStages] == cnt + j) &&
                                                  mbar_test_wait(bar_full + 8u * ((cnt + j) % kStages), ((cnt + j) / kStages) & 1u)))
                            nbk = j + 1;
                    uint32_t st[E::UNIT];
#pragma unroll
                    for (int j = 0; j < E::UNIT; ++j) st[j] = (cnt + j) % kStages;
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int j = 0; j < E::UNIT; ++j) {
                            if (j >= nbk) break;
                            const uint32_t sa = base + st[j] * kSlotBytes;
                            const uint32_t sbs = shb + static_cast<uint32_t>(sub + j) * kHBytes;
#pragma unroll
                            for (int k = 0; k < 4; ++k)   // 32 bytes of K per instruction
                                E::mma(tmem + kDnCol0 + NT * buf, desc_kmajor_sw128(sa + 32u * k),
                                       desc_kmajor_sw128(sbs + 32u * k), (sub + j != s0 || k != 0) ? 1u : 0u);
                            tc_commit(bar_empty + 8u * st[j]);
                        }
                        if (sub + nbk == s1) tc_commit(bar_dacc_full + 8u * buf);
                    }
                    __syncwarp();
                    cnt += nbk;
                    sub += nbk;
                }
            }
            // the h entry is free again once this run's MMAs have read it
            if (elect_one()) tc_commit(bar_h_empty + 8u * hb);
            __syncwarp();
        }
        // every MMA this warp issued completes before TMEM is released
        if (elect_one()) {
            tc_commit(bar_drain + 8u * mw);
            mbar_wait_drain(bar_drain + 8u * mw, 0, kDrainCycles);
        }
        __syncwarp();
    } else if (warp == kMma2Warp) {
        // no second issuer in this form
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int row = q * 32 + lane;        // TMEM lane = accumulator row
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const int et = static_cast<int>(threadIdx.x) - 64;
        bool ok = true;
        if (zero_y) {
            // this CTA's share of y = 0, published per warp; atomics wait for every share
            const long long n4 = static_cast<long long>(a.n) * a.d / 4;
            const long long z0 = c * n4 / P, z1 = (c + 1) * n4 / P;
            float4 *const y4 = reinterpret_cast<float4 *>(a.y);
            for (long long i = z0 + et; i < z1; i += 128) y4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            __syncwarp();
            if (lane == 0) st_release_gpu(a.flags + c * 4 + q, ticket);
        }
        // e4m3: this warp's copy of the token scales
        float *const sxs = reinterpret_cast<float *>(base_ptr + L::kSxOff) + q * NT;
        if constexpr (F8) {
            for (int t = lane; t < NT; t += 32) sxs[t] = t < a.n ? a.s_x[t] : 1.0f;
            __syncwarp();
        }
        GroupInfo<NT> gi;
        if constexpr (NT != 16) {
            int *const tab = reinterpret_cast<int *>(base_ptr + L::kTabOff) + (warp - 2) * 2 * NT;
            gi.pos = tab;
            gi.gt = reinterpret_cast<float *>(tab + NT);
        }
        // gate/up: the partial sums [row, t] of each item share, tagged with the ticket
        uint32_t seg = 0;
        for (long long b = glo; b < ghi;) {
            const Seg s = seg_at(ar, b, ghi, KB, T);
            b = s.b1;
            if (!s.valid) {
                // reported once per group, by the CTA holding the group's first block
                if (warp == 2 && lane == 0 && s.tile == 0 && s.b0 == static_cast<long long>(s.item) * KB)
                    record_error(a.err, MOE_ERR_BAD_ID);
                continue;
            }
            // e4m3: this row's weight scale, loaded before the accumulator wait
            float rs = 1.0f;
            if constexpr (F8) {
                const int fr = s.e * a.f + s.tile * kFTile + (row & 63);
                rs = row < 64 ? a.s_gate[fr] : a.s_up[fr];
            }
            group_tokens(ar, s.g, lane, gi);
            // this CTA's share of the item: 0 for the CTA holding its first block
            const int slot = c - gsp.part_of(static_cast<long long>(s.item) * KB);
            const uint32_t buf = seg % kGuBufs, sph = (seg / kGuBufs) & 1u;
            ++seg;
            // wait outcomes are made warp-uniform so the .sync.aligned TMEM loads stay converged
            if (!warp_wait(bar_gacc_full + 8u * buf, sph, abort_flag, a.err, wl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // 16 token columns at a time, only those holding a token of the group (the mask
            // is the same in every lane); slot is in range with gu_parts' bound
            if (slot >= 0 && slot < kMaxSpan) {
                uint32_t vr[NT / 16][16];
#pragma unroll
                for (int ch = 0; ch < NT / 16; ++ch)
                    if ((static_cast<uint32_t>(gi.mask >> (16 * ch)) & 0xFFFFu) != 0u)
                        tmem_ld_16_async(tmem + lane_off + NT * buf + 16u * ch, vr[ch]);
                tmem_wait_ld();
#pragma unroll
                for (int ch = 0; ch < NT / 16; ++ch) {
                    const uint32_t cm = static_cast<uint32_t>(gi.mask >> (16 * ch)) & 0xFFFFu;
                    if (cm == 0u) continue;
                    float v[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) v[t] = __uint_as_float(vr[ch][t]);
                    if constexpr (F8) {
                        // sums of code products back to values: weight-row scale times token scale
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            if ((cm >> t) & 1u) v[t] *= rs * sxs[16 * ch + t];
                    }
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if ((cm >> t) & 1u)
                            st_tagged(part + part_index(gi.pos[16 * ch + t], T, s.tile, slot, row), v[t], ticket);
                }
            }
            tc_fence_before();
            warp_arrive(bar_gacc_empty + 8u * buf);
        }
        // down: y[t, o] += gate_t * (W_down h)[o, t] with the run's gates from its group record
        if (ok && zero_y && dlo < dhi) {
            // every CTA's zeroing of y is visible before the first atomic (4 P <= 1024 flags)
            ok = warp_wait_tickets(a.flags, 4 * P, ticket, abort_flag, a.err, wl);
        }
        uint32_t dcnt = 0, run = 0;
        for (long long b = dlo; ok && b < dhi;) {
            const Seg sg = seg_at(ar, b, dhi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const Units u = units_of(sg);
            const uint32_t hb = run % kHRing, hph = (run / kHRing) & 1u;
            ++run;
            if (!warp_wait(bar_h_full + 8u * hb, hph, abort_flag, a.err, wl)) break;
            const uint32_t *const rec = reinterpret_cast<const uint32_t *>(info_ptr + hb * kInfoBytes);
            const Mask mask = run_mask<Mask>(rec);
            // the run's gates times the h scales of the span (written for the mask's tokens
            // only): in registers (16 tokens) or in this warp's table (wide form), copied
            // before the h entry is handed back
            float gt[16];
            float *const gw = reinterpret_cast<float *>(base_ptr + L::kGwOff) + q * NT;
            if constexpr (NT == 16) {
#pragma unroll
                for (int t = 0; t < 16; ++t) gt[t] = __uint_as_float(rec[2 + t]);
                if constexpr (F8) {
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if ((mask >> t) & 1u) gt[t] *= __uint_as_float(rec[2 + NT + t]);
                }
            } else {
                __syncwarp();   // every lane has read the previous run's gates
                for (int t = lane; t < NT; t += 32) {
                    float g = 0.0f;
                    if ((mask >> t) & 1u) {
                        g = __uint_as_float(rec[2 + t]);
                        if constexpr (F8) g *= __uint_as_float(rec[2 + NT + t]);
                    }
                    gw[t] = g;
                }
                __syncwarp();
            }
            warp_arrive(bar_h_empty + 8u * hb);
            // e4m3: the W_down row scales of the next batch's units, loaded one batch ahead
            // so that their latency hides behind the accumulator waits and the atomics
            const float *const srow = F8 ? a.s_down + static_cast<size_t>(sg.e) * a.d + row : nullptr;
            float wsn[kEpiBatch];
            auto load_scales = [&](int ob0) {
#pragma unroll
                for (int j = 0; j < kEpiBatch; ++j) wsn[j] = (F8 && ob0 + j <= u.ob_last()) ? srow[(ob0 + j) * kOB] : 1.0f;
            };
            // units in batches of up to kEpiBatch (consecutive d blocks): their TMEM loads
            // share one wait.  Token columns 16 at a time, those of the group only; the first
            // 16 are loaded as each accumulator completes.
            constexpr int kCh = NT / 16;   // 16-column chunks of an accumulator
            int ob = u.ob_first();
            while (ob <= u.ob_last() && u.s_lo(ob) >= u.s_hi(ob)) ++ob;   // no real sub-tile
            load_scales(ob);
            while (ok && ob <= u.ob_last()) {
                int nb = 0;
                uint32_t r[kEpiBatch][kCh][16];
                float wsc[kEpiBatch];
#pragma unroll
                for (int j = 0; j < kEpiBatch; ++j) {
                    wsc[j] = wsn[j];
                    if (ob > u.ob_last()) break;
                    const uint32_t buf = dcnt % kDownBufs, dph = (dcnt / kDownBufs) & 1u;
                    // the first unit of a batch is waited for; later ones join only if
                    // already complete (a non-blocking test), so a batch never holds back
                    // finished accumulators
                    if (j > 0 && !__all_sync(kFull, mbar_test_wait(bar_dacc_full + 8u * buf, dph))) break;
                    if (!warp_wait(bar_dacc_full + 8u * buf, dph, abort_flag, a.err, wl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // every chunk that holds a token of the group, all behind one wait
#pragma unroll
                    for (int ch = 0; ch < kCh; ++ch)
                        if ((static_cast<uint32_t>(mask >> (16 * ch)) & 0xFFFFu) != 0u)
                            tmem_ld_16_async(tmem + kDnCol0 + lane_off + NT * buf + 16u * ch, r[j][ch]);
                    ++nb;
                    ++dcnt;
                    ++ob;
                }
                tmem_wait_ld();   // also before leaving on an abort: no load stays in flight
                if (!ok) break;
                tc_fence_before();
#pragma unroll
                for (int j = 0; j < kEpiBatch; ++j)
                    if (j < nb) warp_arrive(bar_dacc_empty + 8u * ((dcnt - nb + j) % kDownBufs));
                if constexpr (F8) load_scales(ob);
                const int ob0 = ob - nb;
#pragma unroll
                for (int ch = 0; ch < kCh; ++ch) {
                    const uint32_t cm = static_cast<uint32_t>(mask >> (16 * ch)) & 0xFFFFu;
                    if (cm == 0u) continue;
                    float g16[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        if constexpr (NT == 16) g16[t] = gt[t];
                        else g16[t] = ((cm >> t) & 1u) ? gw[16 * ch + t] : 0.0f;
                    }
#pragma unroll
                    for (int j = 0; j < kEpiBatch; ++j) {
                        if (j >= nb) break;
                        const int o = (ob0 + j) * kOB + row;
                        const float ws = wsc[j];   // W_down row scale (1 for bf16)
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            if ((cm >> t) & 1u)
                                atomicAdd(a.y + static_cast<size_t>(16 * ch + t) * a.d + o,
                                          g16[t] * ws * __uint_as_float(r[j][ch][t]));
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ h formers
        // The kHWarps warps take every run, up to kHRing runs ahead of the MMAs.  A run of a
        // group of cnt slots is formed by W = min(kHWarps, ceil(cnt / E::TK)) of them, from the
        // run's leader on, the k-th token (ascending) by the (k % W)-th: one round of loads per
        // warp for small groups, the rounds of a large group spread over the warps.  The leaders
        // rotate by the warps each run takes (run r + 1 is led by the warp after run r's last
        // one), so consecutive runs of small groups go to different warps and are formed side
        // by side, and any kHWarps consecutive runs still give every warp a part, which keeps
        // the h ring's parity waits exact (see Cfg).  The other warps skip the
        // run: the leader arrives for them on h_full (kHWarps - W + 1 arrivals, each helper
        // one), so none waits for a ring entry it does not fill.  W comes from the group's slot
        // count, which the h formers copy to shared memory first (1 per group in the per-slot
        // form), so a skipping warp reads nothing of the group.  A lane holds E::COLS of the
        // item's columns (c = lane + 32 k: gate/up tile c / 64, row c % 64).  After the flags of
        // the item's gate/up shares, h = silu(g) * u of each token from the partial sums, summed
        // over the shares in order.
        const int hw = warp - 6;
        // slot count of each group, clamped as group_tokens clamps the offsets (G <= N <= 1024;
        // the count area of the in-kernel grouping is free once it is built)
        int32_t *const gcnt = reinterpret_cast<int32_t *>(base_ptr + L::kCntOff);
        if (ar.mode != kModePerSlot) {
            const int S = a.n * a.m;
            for (int g = hw * 32 + lane; g < G; g += kHWarps * 32)
                gcnt[g] = max(0, min(S, ar.offsets[g + 1]) - max(0, ar.offsets[g]));
            named_barrier(2, kHWarps * 32);
        }
        GroupInfo<NT> gi;
        if constexpr (NT != 16) {
            int *const tab = reinterpret_cast<int *>(base_ptr + L::kTabOff) + (warp - 2) * 2 * NT;
            gi.pos = tab;
            gi.gt = reinterpret_cast<float *>(tab + NT);
        }
        uint32_t run = 0, lead = 0;   // lead: warps taken by the earlier runs
        for (long long b = dlo; b < dhi;) {
            const Seg sg = seg_at(ar, b, dhi, IB, T2);
            b = sg.b1;
            if (!sg.valid) continue;
            const uint32_t rr = run++;
            const uint32_t hb = rr % kHRing, hph = (rr / kHRing) & 1u;
            const int cnt = ar.mode == kModePerSlot ? 1 : gcnt[sg.g];
            const int nw = min(kHWarps, max(1, (cnt + E::TK - 1) / E::TK));   // warps forming the run
            const int first = (hw - static_cast<int>(lead % kHWarps) + kHWarps) % kHWarps;   // this warp's first token
            lead += static_cast<uint32_t>(nw);
            if (first >= nw) continue;   // not a warp of this run
            group_tokens(ar, sg.g, lane, gi);
            // this warp's tokens: every nw-th of the group's, from its first
            Mask mymask = gi.mask;
            if (nw > 1) {
                mymask = 0u;
                if constexpr (NT == 16) {
                    int k = 0;
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        if ((gi.mask >> t) & 1u) {
                            if (k % nw == first) mymask |= 1u << t;
                            ++k;
                        }
                } else {
                    Mask rest = gi.mask;
                    for (int k = 0; rest != 0u; ++k) {
                        const Mask low = rest & (~rest + 1u);   // the lowest remaining token
                        if (k % nw == first) mymask |= low;
                        rest ^= low;
                    }
                }
            }
            const int mine = mask_count(mymask);
            const int ntiles = min(E::ITEM, T - sg.tile * E::ITEM);   // real gate/up tiles of the item
            const int tile0 = sg.tile * E::ITEM;
            // the CTA shares of each real tile's gate/up item: first CTA and count
            int p0[E::ITEM], span[E::ITEM];
#pragma unroll
            for (int tl = 0; tl < E::ITEM; ++tl) {
                const long long first = static_cast<long long>(sg.g * T + min(tile0 + tl, T - 1)) * KB;
                p0[tl] = gsp.part_of(first);
                span[tl] = min(gsp.part_of(first + KB - 1) - p0[tl] + 1, kMaxSpan);
            }
            // a warp arrives for a run only after its entry is free, so no arrival runs ahead;
            // with fewer entries than warps, the parity wait follows a seen release of run
            // rr - 2 kHRing (see Cfg)
            if constexpr (kHRing < kHWarps) {
                if (rr >= 2u * kHRing &&
                    !warp_wait_at_least(h_seen, rr - 2u * kHRing + 1u, abort_flag, a.err, wl))
                    break;
            }
            if (!warp_wait(bar_h_empty + 8u * hb, hph ^ 1u, abort_flag, a.err, wl)) break;
            if constexpr (kHRing < kHWarps) {
                if (lane == 0 && rr >= static_cast<uint32_t>(kHRing)) atomicMax(h_seen, rr - kHRing + 1u);
            }
            bool parts_ok = true;
            uint8_t *const hp = h_ptr + hb * kHEntry;
            uint32_t *const rec = reinterpret_cast<uint32_t *>(info_ptr + hb * kInfoBytes);
            // E::TK of this warp's tokens at a time: all loads first (predicated, independent)
#pragma unroll kRoundUnroll
            for (int k0 = 0; k0 < NT; k0 += E::TK) {
                if (k0 >= mine) break;
                uint32_t tk[E::TK];
                int pk[E::TK];
#pragma unroll
                for (int j = 0; j < E::TK; ++j) {
                    tk[j] = nth_token(mymask, k0 + j);   // >= NT past the last
                    if constexpr (NT == 16) {
                        pk[j] = 0;
#pragma unroll
                        for (int t = 0; t < 16; ++t) pk[j] = (tk[j] == static_cast<uint32_t>(t)) ? gi.pos[t] : pk[j];
                    } else {
                        pk[j] = tk[j] < static_cast<uint32_t>(NT) ? gi.pos[tk[j]] : 0;
                    }
                }
                // the tagged partial sums of these tokens: all loads first (predicated,
                // independent), then reloads of the words that do not carry this call's ticket
                // yet, until every word of the warp does (bounded like every wait); words that
                // are not needed count as present with value 0
                uint64_t wg[E::TK][E::COLS][kMaxSpan], wu[E::TK][E::COLS][kMaxSpan];
                const uint64_t absent = static_cast<uint64_t>(ticket) << 32;
#pragma unroll
                for (int j = 0; j < E::TK; ++j) {
#pragma unroll
                    for (int k = 0; k < E::COLS; ++k) {
                        const int c = lane + 32 * k, tl = c >> 6, i = c & 63;
                        const bool on = tk[j] < static_cast<uint32_t>(NT) && tl < ntiles;
                        const uint64_t *const pp = part + part_index(pk[j], T, tile0 + (on ? tl : 0), 0, i);
#pragma unroll
                        for (int sl = 0; sl < kMaxSpan; ++sl) {
                            const bool ld = on && sl < span[tl];
                            wg[j][k][sl] = ld ? ld_tagged(pp + sl * 128) : absent;
                            wu[j][k][sl] = ld ? ld_tagged(pp + sl * 128 + 64) : absent;
                        }
                    }
                }
                const long long tp0 = clock64();
                while (true) {
                    bool have = true;
#pragma unroll
                    for (int j = 0; j < E::TK; ++j)
#pragma unroll
                        for (int k = 0; k < E::COLS; ++k)
#pragma unroll
                            for (int sl = 0; sl < kMaxSpan; ++sl)
                                have = have && tag_is(wg[j][k][sl], ticket) && tag_is(wu[j][k][sl], ticket);
                    if (__all_sync(kFull, have)) break;
                    const bool late = clock64() - tp0 > wl;
                    if (__any_sync(kFull, late || *abort_flag != 0)) {
                        if (late && lane == 0) {
                            *abort_flag = 1;
                            record_error(a.err, MOE_ERR_DEVICE_TIMEOUT);
                        }
                        parts_ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < E::TK; ++j) {
#pragma unroll
                        for (int k = 0; k < E::COLS; ++k) {
                            const int c = lane + 32 * k, tl = c >> 6, i = c & 63;
                            const bool on = tk[j] < static_cast<uint32_t>(NT) && tl < ntiles;
                            const uint64_t *const pp = part + part_index(pk[j], T, tile0 + (on ? tl : 0), 0, i);
#pragma unroll
                            for (int sl = 0; sl < kMaxSpan; ++sl) {
                                if (!tag_is(wg[j][k][sl], ticket)) wg[j][k][sl] = ld_tagged(pp + sl * 128);
                                if (!tag_is(wu[j][k][sl], ticket)) wu[j][k][sl] = ld_tagged(pp + sl * 128 + 64);
                            }
                        }
                    }
                }
                if (!parts_ok) break;
#pragma unroll
                for (int j = 0; j < E::TK; ++j) {
                    const uint32_t t = tk[j];
                    if (t >= static_cast<uint32_t>(NT)) break;
                    float hv[E::COLS];
#pragma unroll
                    for (int k = 0; k < E::COLS; ++k)
                        hv[k] = silu(tagged_value(wg[j][k][0]) + tagged_value(wg[j][k][1]) + tagged_value(wg[j][k][2])) *
                                (tagged_value(wu[j][k][0]) + tagged_value(wu[j][k][1]) + tagged_value(wu[j][k][2]));
                    if constexpr (!F8) {
#pragma unroll
                        for (int k = 0; k < E::COLS; ++k) {
                            const int c = lane + 32 * k, blk = c >> 6, i = c & 63;
                            if (blk >= ntiles) continue;
                            // 128-byte swizzle: row t of 128 bytes, 16-byte chunk (i/8) ^ (t%8)
                            const uint32_t off = static_cast<uint32_t>(blk * kHBytes + (t >> 3) * 1024 + (t & 7) * 128 +
                                                                       (((i >> 3) ^ (t & 7)) << 4) + (i & 7) * 2);
                            *reinterpret_cast<__nv_bfloat16 *>(hp + off) = __float2bfloat16_rn(hv[k]);
                        }
                    } else {
                        // e4m3 h: the token's values over the item's 256 (or 128) columns share
                        // one scale, amax / 448, reduced over the warp before any is rounded
                        float mx = 0.0f;
#pragma unroll
                        for (int k = 0; k < E::COLS; ++k)
                            if (((lane + 32 * k) >> 6) < ntiles) mx = fmaxf(mx, fabsf(hv[k]));
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
                        const float hs = mx > 0.0f ? mx / 448.0f : 1.0f;
                        if (lane == 0) rec[2 + NT + t] = __float_as_uint(hs);   // the token's h scale
#pragma unroll
                        for (int k = 0; k < E::COLS; ++k) {
                            const int c = lane + 32 * k, blk = c >> 7, fl = c & 127;   // block of 128, column in it
                            if ((c >> 6) >= ntiles) continue;
                            const uint32_t off = static_cast<uint32_t>(blk * kHBytes + (t >> 3) * 1024 + (t & 7) * 128 +
                                                                       (((fl >> 4) ^ (t & 7)) << 4) + (fl & 15));
                            hp[off] = f32_to_e4m3(hv[k] / hs);
                        }
                    }
                }
            }
            if (!parts_ok) break;
            // the run's record (mask and gates) by the warp of its first token; the epilogue
            // reads the h scales of the mask's tokens only
            if (first == 0) {
                if (lane == 0) {
                    rec[0] = static_cast<uint32_t>(gi.mask);
                    rec[1] = static_cast<uint32_t>(static_cast<uint64_t>(gi.mask) >> 32);
                }
                if constexpr (NT == 16) {
                    if (lane == 0) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) rec[2 + t] = __float_as_uint(gi.gt[t]);
                    }
                } else {
                    for (int t = lane; t < NT; t += 32)
                        if ((gi.mask >> t) & 1u) rec[2 + t] = __float_as_uint(gi.gt[t]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive_cnt(bar_h_full + 8u * hb, first == 0 ? static_cast<uint32_t>(kHWarps - nw + 1) : 1u);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    // After an abort, copies that no MMA consumed may still be landing: every role has left
    // its loop (the abort flag is final here), and the CTA waits (bounded) for them to land
    // before it exits.
    if (warp == 0 && lane == 0 && *abort_flag != 0) drain_copies(bar_full, prod_cnt, kStages);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
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
    bool attr_set[7] = {false, false, false, false, false, false, false};   // per kernel form
};

std::mutex g_info_mu;
DeviceInfo g_info[64];

template <bool F8, int NT, int U>
cudaError_t set_attributes() {
    return cudaFuncSetAttribute(expert_tc_kernel<F8, NT, U>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Lay<NT, U>::kSmem);
}

template <bool F8, int NT, int U>
cudaError_t launch(const ExpertArgs &a, int sms, int max_groups, bool zero_y, uint64_t *part, cudaStream_t s, bool pdl) {
    using E = Elt<F8, NT, U>;
    const long long T = a.f / kFTile, OBS = a.d / kOB;
    const long long T2 = (T + E::ITEM - 1) / E::ITEM;
    // CTAs with work: up to 2*G*T gate/up shares, and at most one per down block
    const long long work = std::max<long long>(2ll * max_groups * T, static_cast<long long>(max_groups) * T2 * OBS * E::UNIT);
    const int grid = static_cast<int>(std::min<long long>(std::min(sms, kMaxGrid), work));

    CUtensorMap tm_wg, tm_wu, tm_wd, tm_x;
    const uint64_t d = a.d, f = a.f, N = a.N;
    // x: boxes of NT rows; the rows past the pass's n are filled with zeros
    if (!encode_2d(&tm_wg, a.w_gate, F8, d, N * f, E::BK, kFTile) ||
        !encode_2d(&tm_wu, a.w_up, F8, d, N * f, E::BK, kFTile) ||
        !encode_2d(&tm_wd, a.w_down, F8, f, N * d, E::BK, kOB) ||
        !encode_2d(&tm_x, a.x, F8, d, static_cast<uint64_t>(a.n), E::BK, NT))
        return cudaErrorInvalidValue;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay<NT, U>::kSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, expert_tc_kernel<F8, NT, U>, tm_wg, tm_wu, tm_wd, tm_x, a, part, zero_y ? 1 : 0);
}

}  // namespace

bool expert_tc_supports(int d, int f) { return d % kOB == 0 && f % kFTile == 0 && d >= kOB && f >= kFTile; }

cudaError_t launch_expert_tc(const ExpertArgs &a, int max_groups, bool zero_y, uint64_t *part, cudaStream_t s,
                             bool pdl) {
    const bool f8 = a.w_dtype == MOE_E4M3 && a.x_dtype == MOE_E4M3;
    const bool bf = a.w_dtype == MOE_BF16 && a.x_dtype == MOE_BF16;
    if (!expert_tc_supports(a.d, a.f) || !(f8 || bf) || a.n < 1 || a.n > kMaxPassTokens || max_groups < 1)
        return cudaErrorNotSupported;
    if (a.sync == nullptr || a.flags == nullptr) return cudaErrorInvalidValue;
    // e4m3: 128-element k slices; h spans of 256 f (the last may be 128)
    if (f8 && (a.d % 128 != 0 || a.f % 128 != 0 || a.s_gate == nullptr || a.s_up == nullptr ||
               a.s_down == nullptr || a.s_x == nullptr))
        return cudaErrorNotSupported;
    // the token width: the narrowest instantiation that holds the pass; the unit: 4 down blocks
    // per accumulator (half the combine's reductions per y element) for bf16 per-slot launches,
    // deduplicating passes of 1-2 and of 12 or more tokens and the wide forms, 2 for bf16
    // deduplicating passes of 3-11 tokens (their h formers take two tokens a round at 2-tile
    // items, which measured faster there) and for every e4m3 form
    const int width = a.n <= 16 ? 0 : (a.n <= 32 ? 1 : 2);
    const bool u4 = !f8 && (a.mode == kModePerSlot || a.n <= 2 || a.n >= 12 || width > 0);
    const int form = f8 ? 4 + width : (width == 0 ? (u4 ? 1 : 0) : 1 + width);
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
        if (!di.attr_set[form]) {
            switch (form) {
                case 0: err = set_attributes<false, 16, 2>(); break;
                case 1: err = set_attributes<false, 16, 4>(); break;
                case 2: err = set_attributes<false, 32, 4>(); break;
                case 3: err = set_attributes<false, 64, 4>(); break;
                case 4: err = set_attributes<true, 16, 2>(); break;
                case 5: err = set_attributes<true, 32, 2>(); break;
                default: err = set_attributes<true, 64, 2>(); break;
            }
            if (err != cudaSuccess) return err;
            di.attr_set[form] = true;
        }
        sms = di.sms;
    }
    switch (form) {
        case 0: return launch<false, 16, 2>(a, sms, max_groups, zero_y, part, s, pdl);
        case 1: return launch<false, 16, 4>(a, sms, max_groups, zero_y, part, s, pdl);
        case 2: return launch<false, 32, 4>(a, sms, max_groups, zero_y, part, s, pdl);
        case 3: return launch<false, 64, 4>(a, sms, max_groups, zero_y, part, s, pdl);
        case 4: return launch<true, 16, 2>(a, sms, max_groups, zero_y, part, s, pdl);
        case 5: return launch<true, 32, 2>(a, sms, max_groups, zero_y, part, s, pdl);
        default: return launch<true, 64, 2>(a, sms, max_groups, zero_y, part, s, pdl);
    }
}

}  // namespace moe
