// common.cuh -- shared device helpers of libmoeverify (sm_103a).
//
// Inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), tcgen05 (MMA, TMEM),
// programmatic dependent launch and the bounded waits every pipeline uses.
#pragma once

#include <cuda.h>          // CUtensorMap (type only; no driver symbol is linked)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_verify.h"

namespace moe {

// ------------------------------------------------------------------ workspace
// Device workspace layout.  Word 0 is the device error word (first error wins).
struct DeviceWorkspace {
    int32_t error;
    uint32_t sync[2];   // tensor-core path: the epoch of its flags, and a CTA exit count
    int32_t reserved[61];
};
constexpr size_t kWorkspaceBytes = sizeof(DeviceWorkspace);   // 256

__device__ __forceinline__ void record_error(int32_t *err, int32_t code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

// Time limit of every spin-wait on an mbarrier, in SM clock cycles (about 2 s at the
// 2.07 GHz maximum clock; longer at lower clocks).
constexpr long long kWaitLimitCycles = 4000000000ll;

// ------------------------------------------------------------------ basics
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


// Programmatic dependent launch: wait for the grids this one depends on (no-op when
// the launch carried no programmatic dependency), and allow dependents to launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Warm L2 (and the address translation) for the 128-byte lines of [p, p + bytes), thread
// `tid` of `nthreads` taking every nthreads-th line.  A prefetch reads no value: loads that
// follow it see whatever was written last.
__device__ __forceinline__ void prefetch_l2_range(const void *p, size_t bytes, int tid, int nthreads) {
    if (p == nullptr) return;
    const char *c = static_cast<const char *>(p);
    for (size_t off = static_cast<size_t>(tid) * 128; off < bytes; off += static_cast<size_t>(nthreads) * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

// One lane of the (fully active) warp returns true.  Issuing tensor-core and TMA
// instructions from an elected lane inside warp-uniform code keeps their operands in
// uniform registers; a lone divergent lane issuing them is several times slower.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(pred));
    return pred != 0;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// `count` arrivals at once (count >= 1, at most the pending count of the phase).
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity (try_wait may suspend the thread
// for a while; this never does).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Gives up when *abort becomes
// non-zero (another role gave up) or after `limit` cycles (kWaitLimitCycles unless the call
// asked for a shorter limit); on a time-out it raises the abort flag and records
// MOE_ERR_DEVICE_TIMEOUT.  Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int32_t *abort,
                                          int32_t *err, long long limit = kWaitLimitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            record_error(err, MOE_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// Warp-wide forms for warp-uniform code.  Every lane polls and acquires for itself (one
// polling lane with a broadcast measured slower on GB300), and the outcome is made uniform
// so that .sync.aligned instructions after it stay converged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int32_t *abort, int32_t *err,
                                          long long limit = kWaitLimitCycles) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort, err, limit));
}
// One arrival for the whole warp, after every lane's earlier work (barrier counts are in warps).
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
__device__ __forceinline__ void warp_arrive_cnt(uint32_t bar, uint32_t count) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_cnt(bar, count);
}

// gpu-scope release store and acquire load of a 32-bit flag in global memory: a flag
// written with st_release_gpu after a CTA's stores makes them visible to every thread that
// reads the flag's value with ld_acquire_gpu.
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Relaxed gpu-scope load (several may be in flight at once); followed by fence_acq_rel_gpu once
// a value written with st_release_gpu was seen, it orders later accesses after that store.
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// gpu-scope atomic add with acquire and release semantics; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Warp-wide bounded wait until the flag of every lane holds `ticket` (lanes with p == nullptr
// have none).  The same abort and time-limit rules as mbar_wait; the outcome is warp-uniform,
// and every lane's later loads are ordered after the flags it waited for.
__device__ __forceinline__ bool warp_wait_ticket(const uint32_t *p, uint32_t ticket, volatile int32_t *abort,
                                                 int32_t *err, long long limit = kWaitLimitCycles) {
    bool ok = p == nullptr || ld_acquire_gpu(p) == ticket;
    const long long t0 = clock64();
    while (!__all_sync(0xFFFFFFFFu, ok)) {
        if (!ok) ok = ld_acquire_gpu(p) == ticket;
        const bool late = clock64() - t0 > limit;
        if (__any_sync(0xFFFFFFFFu, late || *abort != 0)) {
            if (late) {
                *abort = 1;
                record_error(err, MOE_ERR_DEVICE_TIMEOUT);
            }
            return false;
        }
    }
    __syncwarp();
    return true;
}

// Warp-wide bounded wait until every flag of flags[0, count) holds `ticket` (count <= 32 * 32):
// lane l watches flags l + 32 r, all of its loads in flight together, so the wait costs one
// round trip to memory when the flags are already set, not one per 32 flags.  The same abort
// and time-limit rules as mbar_wait; every lane's later accesses are ordered after the flags.
__device__ __forceinline__ bool warp_wait_tickets(const uint32_t *flags, int count, uint32_t ticket,
                                                  volatile int32_t *abort, int32_t *err,
                                                  long long limit = kWaitLimitCycles) {
    const int lane = static_cast<int>(threadIdx.x & 31);
    uint32_t missing = 0;   // bit r: flag lane + 32 r not seen yet
    for (int r = 0; r < 32; ++r)
        if (lane + 32 * r < count) missing |= 1u << r;
    const long long t0 = clock64();
    while (true) {
        uint32_t v[32];
#pragma unroll
        for (int r = 0; r < 32; ++r)
            if ((missing >> r) & 1u) v[r] = ld_relaxed_gpu(flags + lane + 32 * r);   // all in flight together
#pragma unroll
        for (int r = 0; r < 32; ++r)
            if (((missing >> r) & 1u) && v[r] == ticket) missing &= ~(1u << r);
        if (__all_sync(0xFFFFFFFFu, missing == 0u)) break;
        const bool late = clock64() - t0 > limit;
        if (__any_sync(0xFFFFFFFFu, late || *abort != 0)) {
            if (late) {
                *abort = 1;
                record_error(err, MOE_ERR_DEVICE_TIMEOUT);
            }
            return false;
        }
    }
    fence_acq_rel_gpu();   // the flags seen (relaxed) now order this lane's later accesses
    __syncwarp();
    return true;
}

// Bounded wait that ignores the abort flag (used to drain copies in flight on abort).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, long long limit_cycles) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit_cycles) return false;
    }
    return true;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on bar as
// transaction bytes.  c0 is the inner (contiguous) coordinate, c1 the outer one.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy
// (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulators, one thread issues.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with e4m3 A and B (kind::f8f6f4, fp32 accumulators; K = 32 per instruction).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on bar when every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane into
// raw registers; the values may be used only after tmem_wait_ld().  Several loads in flight
// share one wait.
__device__ __forceinline__ void tmem_ld_16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the 128-byte
// swizzle (rows of 128 bytes, 8-row atoms of 1024 bytes, atoms 1024 bytes apart), the
// layout a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes.  saddr: the tile start plus
// the byte offset of the K slice inside the 128-byte row.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);   // start address
    d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version (tcgen05)
    d |= static_cast<uint64_t>(2u) << 61;                 // swizzle mode: 128-byte
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                                  // D: fp32
           | (1u << 7)                                // A: bf16
           | (1u << 10)                               // B: bf16
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Instruction descriptor of kind::f8f6f4 with e4m3 A and B (format code 0), fp32 D, both
// K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                                  // D: fp32
           | (0u << 7)                                // A: e4m3
           | (0u << 10)                               // B: e4m3
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Round to the nearest e4m3 value, ties to even, saturating at +-448 (cvt.rn.satfinite).
__device__ __forceinline__ uint8_t f32_to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return static_cast<uint8_t>(r & 0xFFu);
}

// Named barrier over `count` threads (a multiple of 32) of the CTA; id 0 is __syncthreads'.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ numerics
// silu(z) = z * sigmoid(z) with the fast exponential and division: about 1e-6 relative,
// far below the bf16 rounding that the tensor-core path applies to h next.  For z very
// negative the denominator overflows and the quotient is 0, the limit of silu.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

}  // namespace moe
