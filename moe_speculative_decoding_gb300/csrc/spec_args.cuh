// spec_args.cuh -- arguments of the verify-side kernels (spec.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace moe {

constexpr int kMaxSpecK = 31;            // drafts per sequence (one warp walks them, K + 1 lanes)
constexpr int kMaxSpecV = 262144;        // vocabulary: 64 warps x 32 steps x 128; W sums fit 64 bits
constexpr size_t kMaxUnionSmem = 200 * 1024;   // bitmaps of a pool, in shared memory

// One round of speculative sampling for B sequences: draft [B, K], q [B, K, V], p [B, K+1, V],
// r [B, K], u [B]; out n_acc [B], token [B].  seg: vocabulary elements per warp (spec_segment).
struct SpecArgs {
    const int32_t *draft;
    const float *q;
    const float *p;
    const float *r;
    const float *u;
    int32_t *n_acc;
    int32_t *token;
    int B, K, V, greedy, seg;
    int vec;   // V % 4 == 0 and p, q 16-byte aligned: float4 loads
};

// Union cost of `count` candidate subtrees over a pool of `nodes` draft nodes (+ the root).
struct UnionArgs {
    const uint64_t *bitmaps;   // [nodes+1][L][W]
    const uint32_t *subsets;   // [count]
    const double *pv;          // [nodes]
    const double *bcoef;       // [nodes+1]
    double beta;
    int32_t *F, *size;
    double *R, *T;
    int32_t *best;
    int nodes, L, W, count;
    int tab;                   // set by launch_union_cost: the kernel uses the node-triple table
};

int spec_segment(int V);
cudaError_t launch_spec_accept(const SpecArgs &a, cudaStream_t s, bool pdl);
size_t union_cost_scratch_bytes(int count);
cudaError_t launch_union_cost(const UnionArgs &a, void *scratch, cudaStream_t s, bool pdl);

}  // namespace moe
