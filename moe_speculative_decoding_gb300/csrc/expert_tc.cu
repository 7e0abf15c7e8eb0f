// expert_tc.cu -- tensor-core (tcgen05 + TMA) kernel of the expert operation, bf16.
//
// "Speculative Decoding for Mixture-of-Experts Models" (Lan), §1: the expert operation
// is the gate, up and down projections of each token of a pass with the weights of its
// selected experts.  Per-slot form: one expert read per slot (m*n*w bytes requested).
// Deduplicating form: the pass's tokens grouped by expert, each distinct expert read once
// (w * X(n) bytes).  §2 "Effective bandwidth": the kernel's figure of merit is requested
// expert bytes over time, so the design streams weights and keeps everything else off
// the memory path.
//
// Design (one persistent CTA per SM, 6 warps):
//   * A work item is (group, 64-row tile of f).  A group is one slot (per-slot form) or
//     one distinct expert with all of its tokens (deduplicating form).  Each item streams
//     three weight blocks exactly once: W_gate[e][i0:i0+64, :], W_up[e][i0:i0+64, :] and
//     the columns W_down[e][:, i0:i0+64].
//   * Warp 0 (one lane) is the TMA producer: 16 KB stages through a ring of mbarriers,
//     128-byte-swizzled boxes.  A gate/up stage holds 64 rows of W_gate and the same 64
//     rows of W_up for one 64-wide k block (M = 128 rows); a down stage holds 128 rows
//     of W_down by the tile's 64 columns.
//   * Warp 1 (one lane) issues tcgen05.mma (bf16 in, fp32 accumulate in TMEM) with the
//     weights as the M operand and the pass's tokens as N = 16 (the narrow dimension):
//     G|U[128 x 16] = [W_gate; W_up] x^T over d, then Y[128 x 16] = W_down[rows, tile] h^T
//     for each 128-row block of d.  The whole pass x (n <= 16 rows, padded with zeros)
//     stays in shared memory for the CTA's lifetime.
//   * Warps 2-5 (128 threads, one TMEM lane each) read the gate/up accumulators,
//     form h = silu(g) * u for the tile (bf16, written to shared memory as the next
//     MMA's B operand), then read each down block and add gate * y into the fp32 output
//     with coalesced atomics: the weighted combine and the f-split reduction are fused.
//   * The MMA warp runs one item ahead on gate/up: the order of stages (and of the
//     producer's loads) is gu(0), gu(1), down(0), gu(2), down(1), ... so the tensor pipe
//     and the copy engine stay busy while the epilogue turns item j's accumulators into h.
//     The gate/up accumulators and h are double-buffered by item parity; the down blocks
//     go through a ring of kDownBufs TMEM accumulators so the MMA warp rarely waits for
//     the epilogue.
//   * Every wait is bounded (common.cuh); a time-out raises an abort flag that every role
//     honours, records MOE_ERR_DEVICE_TIMEOUT, drains copies and MMAs in flight and frees
//     TMEM before the CTA exits.
#include "common.cuh"
#include "expert_args.cuh"

#include <mutex>

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kBK = 64;                     // k elements per 128-byte row
constexpr int kOB = 128;                    // d rows per down block
constexpr int kNT = 16;                     // MMA N (token columns)
constexpr uint32_t kStageBytes = 16384;
constexpr uint32_t kXTileBytes = kNT * 128;   // one k block of x: 16 rows x 128 B
constexpr uint32_t kHBytes = kNT * 128;       // one h tile (16 rows x 64 bf16)
constexpr uint32_t kUXBytes = 64 * kNT * 4;
constexpr int kDownBufs = 8;                // TMEM ring of down-block accumulators
constexpr uint32_t kColGU = 0;              // [0,16) and [16,32): gate/up, by item parity
constexpr uint32_t kColDown = 32;           // [32, 32 + 16 * kDownBufs)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kNT);
constexpr int kMaxStages = 9;
constexpr long long kDrainCycles = 400000000ll;   // about 0.2 s

struct SmemLayout {
    uint32_t x, stages, h, ux, bars, misc, total;
};

// barrier slots after the 2*stages ring barriers
enum {
    kBarGU0 = 0,
    kBarGU1,
    kBarUX,
    kBarH,
    kBarDrain,
    kBarDFull0,
    kBarDEmpty0 = kBarDFull0 + kDownBufs,
    kNumMiscBars = kBarDEmpty0 + kDownBufs
};

__host__ __device__ inline SmemLayout smem_layout(int d, int stages) {
    SmemLayout L;
    L.x = 0;
    L.stages = L.x + static_cast<uint32_t>(d / kBK) * kXTileBytes;
    L.h = L.stages + static_cast<uint32_t>(stages) * kStageBytes;
    L.ux = L.h + 2 * kHBytes;
    L.bars = L.ux + kUXBytes;
    L.misc = L.bars + static_cast<uint32_t>(2 * stages + kNumMiscBars) * 8;
    L.total = L.misc + 16;
    return L;
}

struct Item {
    int e;       // expert
    int g;       // group
    int i0;      // first row of the f tile
};

// Work item it of this call.  Returns false for an item whose expert id is outside
// [0, N): every role skips those the same way.
__device__ __forceinline__ bool item_of(const ExpertArgs &a, int it, int tiles, Item &r) {
    r.g = it / tiles;
    r.i0 = (it - r.g * tiles) * kFTile;
    r.e = (a.mode == kModePerSlot) ? a.ids[r.g] : a.expert_list[r.g];
    return r.e >= 0 && r.e < a.N;
}

// The next valid item of this CTA at or after it (static round robin), or -1.
__device__ __forceinline__ int next_item(const ExpertArgs &a, int it, int items, int tiles, Item &r,
                                         bool report) {
    for (; it < items; it += gridDim.x) {
        if (item_of(a, it, tiles, r)) return it;
        if (report && r.i0 == 0) record_error(a.err, MOE_ERR_BAD_ID);
    }
    return -1;
}

__global__ void __launch_bounds__(kThreads, 1)
expert_tc_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                 const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_x,
                 const ExpertArgs a, const int stages) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw_addr);
    const SmemLayout L = smem_layout(a.d, stages);

    const uint32_t sx = base + L.x;
    const uint32_t sstage = base + L.stages;
    const uint32_t sh = base + L.h;
    float *const ux = reinterpret_cast<float *>(base_ptr + L.ux);
    uint8_t *const h_ptr = base_ptr + L.h;
    const uint32_t bar_full = base + L.bars;                 // [stages]
    const uint32_t bar_empty = bar_full + 8u * stages;       // [stages]
    const uint32_t bar_misc = bar_empty + 8u * stages;       // [kNumMiscBars]
    auto bar = [&](int k) { return bar_misc + 8u * static_cast<uint32_t>(k); };
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + L.misc);
    volatile int32_t *const abort_flag = reinterpret_cast<volatile int32_t *>(base_ptr + L.misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---------------------------------------------------------------- setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        mbar_init(bar(kBarGU0), 1);
        mbar_init(bar(kBarGU1), 1);
        mbar_init(bar(kBarUX), 64);
        mbar_init(bar(kBarH), 64);
        mbar_init(bar(kBarDrain), 1);
        for (int b = 0; b < kDownBufs; ++b) {
            mbar_init(bar(kBarDFull0 + b), 1);
            mbar_init(bar(kBarDEmpty0 + b), 128);
        }
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

    // inputs written by earlier kernels are read only after this point
    pdl_wait();
    pdl_trigger();

    const int tiles = a.f / kFTile;
    // the device-side count is clamped to the buffer sizes the host validated
    const int cap = a.n * a.m < a.N ? a.n * a.m : a.N;
    const int groups = (a.mode == kModePerSlot) ? a.n * a.m : max(0, min(a.num_distinct[0], cap));
    const int items = groups * tiles;
    const int KB = a.d / kBK;
    const int OBS = a.d / kOB;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the schedule and waits; one elected lane issues the copies.
        uint32_t cnt = 0;
        bool ok = true;
        auto acquire = [&](uint32_t &dst, uint32_t &fb, bool &leader, uint32_t extra) -> bool {
            const uint32_t s = cnt % stages, ph = (cnt / stages) & 1u;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_empty + 8u * s, ph ^ 1u, abort_flag, a.err))) return false;
            dst = sstage + s * kStageBytes;
            fb = bar_full + 8u * s;
            leader = elect_one();
            if (leader) mbar_arrive_expect_tx(fb, kStageBytes + extra);
            ++cnt;
            return true;
        };
        // The first gate/up item also brings the pass's x, one 2 KB k block per stage, so
        // the first weights arrive without waiting behind the whole of x.
        bool x_pending = true;
        auto load_gu = [&](const Item &im) -> bool {
            const int row = im.e * a.f + im.i0;
            for (int kb = 0; kb < KB; ++kb) {
                uint32_t dst, fb;
                bool leader;
                if (!acquire(dst, fb, leader, x_pending ? kXTileBytes : 0u)) return false;
                if (leader) {
                    tma_load_2d(dst, &tm_wg, fb, kb * kBK, row);
                    tma_load_2d(dst + kStageBytes / 2, &tm_wu, fb, kb * kBK, row);
                    if (x_pending) tma_load_2d(sx + kb * kXTileBytes, &tm_x, fb, kb * kBK, 0);
                }
                __syncwarp();
            }
            x_pending = false;
            return true;
        };
        auto load_down = [&](const Item &im) -> bool {
            for (int ob = 0; ob < OBS; ++ob) {
                uint32_t dst, fb;
                bool leader;
                if (!acquire(dst, fb, leader, 0u)) return false;
                if (leader) tma_load_2d(dst, &tm_wd, fb, im.i0, im.e * a.d + ob * kOB);
                __syncwarp();
            }
            return true;
        };
        Item cur, nxt;
        int it = next_item(a, blockIdx.x, items, tiles, cur, false);
        if (it >= 0) ok = load_gu(cur);
        while (ok && it >= 0) {
            const int it2 = next_item(a, it + gridDim.x, items, tiles, nxt, false);
            if (it2 >= 0) ok = load_gu(nxt);
            if (ok) ok = load_down(cur);
            it = it2;
            cur = nxt;
        }
        if (!ok && lane == 0) {
            // wait (bounded) for the copies this warp issued and nobody consumed
            const uint32_t first = cnt > static_cast<uint32_t>(stages) ? cnt - stages : 0u;
            for (uint32_t j = first; j < cnt; ++j)
                mbar_wait_drain(bar_full + 8u * (j % stages), (j / stages) & 1u, kDrainCycles);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Warp-uniform loop; waits by every lane, MMAs and commits by one elected lane.
        uint32_t cnt = 0, dcnt = 0, nitem = 0;
        bool ok = true;
        auto mma_gu = [&](uint32_t gbuf) -> bool {
            for (int kb = 0; kb < KB; ++kb, ++cnt) {
                const uint32_t s = cnt % stages, ph = (cnt / stages) & 1u;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_full + 8u * s, ph, abort_flag, a.err))) return false;
                tc_fence_after();
                const uint32_t sa = sstage + s * kStageBytes;
                const uint32_t sb = sx + kb * kXTileBytes;
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_bf16(tmem + kColGU + 16u * gbuf, desc_kmajor_sw128(sa + 32u * k),
                                    desc_kmajor_sw128(sb + 32u * k), kIdesc, (kb | k) != 0 ? 1u : 0u);
                    tc_commit(bar_empty + 8u * s);
                    if (kb == KB - 1) tc_commit(bar(kBarGU0 + gbuf));
                }
                __syncwarp();
            }
            return true;
        };
        auto mma_down = [&](uint32_t hbuf) -> bool {
            for (int ob = 0; ob < OBS; ++ob, ++cnt, ++dcnt) {
                const uint32_t s = cnt % stages, ph = (cnt / stages) & 1u;
                const uint32_t buf = dcnt % kDownBufs, dph = (dcnt / kDownBufs) & 1u;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar_full + 8u * s, ph, abort_flag, a.err))) return false;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarDEmpty0 + buf), dph ^ 1u, abort_flag, a.err)))
                    return false;
                tc_fence_after();
                const uint32_t sa = sstage + s * kStageBytes;
                const uint32_t sb = sh + hbuf * kHBytes;
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_bf16(tmem + kColDown + 16u * buf, desc_kmajor_sw128(sa + 32u * k),
                                    desc_kmajor_sw128(sb + 32u * k), kIdesc, k != 0 ? 1u : 0u);
                    tc_commit(bar_empty + 8u * s);
                    tc_commit(bar(kBarDFull0 + buf));
                }
                __syncwarp();
            }
            return true;
        };
        Item cur, nxt;
        int it = next_item(a, blockIdx.x, items, tiles, cur, false);
        if (ok && it >= 0) ok = mma_gu(0);
        while (ok && it >= 0) {
            const int it2 = next_item(a, it + gridDim.x, items, tiles, nxt, false);
            if (it2 >= 0) ok = mma_gu((nitem + 1) & 1u);
            if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarH), nitem & 1u, abort_flag, a.err));
            if (ok) {
                tc_fence_after();
                ok = mma_down(nitem & 1u);
            }
            ++nitem;
            it = it2;
        }
        // every MMA this warp issued completes before TMEM is released
        if (elect_one()) {
            tc_commit(bar(kBarDrain));
            mbar_wait_drain(bar(kBarDrain), 0, kDrainCycles);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int row = q * 32 + lane;        // TMEM lane = accumulator row
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const bool reporter = (warp == 2 && lane == 0);
        uint32_t dcnt = 0, nitem = 0;
        bool ok = true;
        Item cur;
        for (int it = next_item(a, blockIdx.x, items, tiles, cur, reporter); ok && it >= 0;
             it = next_item(a, it + gridDim.x, items, tiles, cur, reporter), ++nitem) {
            // gate of each pass token in this group (0 if absent)
            float gt[kNT];
#pragma unroll
            for (int t = 0; t < kNT; ++t) gt[t] = 0.0f;
            uint32_t mask = 0;
            if (a.mode == kModePerSlot) {
                const int tt = cur.g / a.m;
                const float gv = a.gates[cur.g];
#pragma unroll
                for (int t = 0; t < kNT; ++t)
                    if (t == tt) gt[t] = gv;
                mask = 1u << tt;
            } else {
                const int S = a.n * a.m;   // offsets are clamped to the slot buffer
                const int p0 = max(0, a.offsets[cur.g]), p1 = min(S, a.offsets[cur.g + 1]);
                for (int p = p0; p < p1; ++p) {
                    const int slot = a.slot_order[p];
                    const int tt = slot / a.m;
                    if (slot < 0 || tt >= a.n) continue;
                    const float gv = a.gates[slot];
#pragma unroll
                    for (int t = 0; t < kNT; ++t)
                        if (t == tt) gt[t] += gv;
                    mask |= 1u << tt;
                }
            }

            // gate/up accumulators -> h (bf16, swizzled B operand of the down MMA).
            // Wait outcomes are made warp-uniform so the .sync.aligned TMEM loads stay
            // converged.
            const uint32_t gbuf = nitem & 1u;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarGU0 + gbuf), (nitem >> 1) & 1u, abort_flag, a.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[16];
            tmem_ld_16(tmem + lane_off + kColGU + 16u * gbuf, v);
            if (q >= 2) {
                const int r = row - 64;
#pragma unroll
                for (int c = 0; c < kNT; ++c)
                    if ((mask >> c) & 1u) ux[c * 64 + r] = v[c];
                tc_fence_before();
                mbar_arrive(bar(kBarUX));
            } else {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarUX), nitem & 1u, abort_flag, a.err))) {
                    ok = false;
                    break;
                }
                const int i = row;   // 0..63
                uint8_t *const hb = h_ptr + gbuf * kHBytes;
#pragma unroll
                for (int c = 0; c < kNT; ++c) {
                    // columns of tokens outside the group are never read back: skip them
                    if (!((mask >> c) & 1u)) continue;
                    const float hv = silu(v[c]) * ux[c * 64 + i];
                    const uint32_t off = static_cast<uint32_t>((c >> 3) * 1024 + (c & 7) * 128 +
                                                               ((((i >> 3) ^ (c & 7))) << 4) + (i & 7) * 2);
                    *reinterpret_cast<__nv_bfloat16 *>(hb + off) = __float2bfloat16_rn(hv);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(kBarH));
            }

            // down blocks: y[t, o] += gate_t * Y[o, t]
            for (int ob = 0; ob < OBS; ++ob, ++dcnt) {
                const uint32_t buf = dcnt % kDownBufs, dph = (dcnt / kDownBufs) & 1u;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarDFull0 + buf), dph, abort_flag, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_ld_16(tmem + lane_off + kColDown + 16u * buf, v);
                tc_fence_before();
                mbar_arrive(bar(kBarDEmpty0 + buf));
                const int o = ob * kOB + row;
#pragma unroll
                for (int t = 0; t < kNT; ++t)
                    if ((mask >> t) & 1u) atomicAdd(a.y + static_cast<size_t>(t) * a.d + o, gt[t] * v[t]);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
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

// 2-D bf16 tensor map over a row-major [outer, inner] matrix, 128-byte swizzle.
bool encode_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
    bool attr_set = false;
};

DeviceInfo &device_info(int dev) {
    static DeviceInfo info[64];
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &di = info[dev & 63];
    if (di.sms == 0) {
        cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return di;
}

int pick_stages(int d, int smem_optin) {
    for (int st = kMaxStages; st >= 2; --st)
        if (static_cast<int>(smem_layout(d, st).total) + 1024 <= smem_optin) return st;
    return 0;
}

}  // namespace

bool expert_tc_supports(int d, int f) {
    // x for 16 tokens and at least two stages must fit in shared memory
    return d % kOB == 0 && f % kFTile == 0 && d >= kOB && d <= 4096 && f >= kFTile;
}

cudaError_t launch_expert_tc(const ExpertArgs &a, int max_groups, cudaStream_t s, bool pdl) {
    if (!expert_tc_supports(a.d, a.f) || a.w_dtype != MOE_BF16 || a.x_dtype != MOE_BF16 || a.n > kNT)
        return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    DeviceInfo &di = device_info(dev);
    const int stages = pick_stages(a.d, di.smem_optin);
    if (stages < 2) return cudaErrorNotSupported;
    const uint32_t smem = smem_layout(a.d, stages).total + 1024;
    {
        static std::mutex mu;
        std::lock_guard<std::mutex> lock(mu);
        if (!di.attr_set) {
            err = cudaFuncSetAttribute(expert_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       di.smem_optin);
            if (err != cudaSuccess) return err;
            di.attr_set = true;
        }
    }
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_x;
    const uint64_t d = a.d, f = a.f, N = a.N;
    if (!encode_2d(&tm_wg, a.w_gate, d, N * f, kBK, kFTile) || !encode_2d(&tm_wu, a.w_up, d, N * f, kBK, kFTile) ||
        !encode_2d(&tm_wd, a.w_down, f, N * d, kBK, kOB) ||
        !encode_2d(&tm_x, a.x, d, static_cast<uint64_t>(a.n), kBK, kNT))
        return cudaErrorInvalidValue;

    const int items_max = max_groups * (a.f / kFTile);
    const int grid = items_max < di.sms ? items_max : di.sms;
    if (grid <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, expert_tc_kernel, tm_wg, tm_wu, tm_wd, tm_x, a, stages);
}

}  // namespace moe
