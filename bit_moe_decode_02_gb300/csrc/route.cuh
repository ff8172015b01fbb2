// route.cuh -- the router shared by the decode kernels: per token, the top-k
// of E logits and a softmax over the k selected ("Sovereign gpt-oss-20B
// (MXFP4) on Apple Silicon", section 3: top-4 routing; GPU top-k on the
// serving path, "Amortizing the per-token host-sync setup tax ...", section 3).
#pragma once
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {
namespace rt {

// One warp: top-k of E logits (largest first; ties to the lower index; NaN
// as -inf), then softmax over the k selected.  Lane 0 writes sel[0..k) and
// the weights wt[0..k).
__device__ __forceinline__ void warp_topk(const float* __restrict__ lg, int E, int k, int* sel, float* wt)
{
    const int lane = threadIdx.x & 31;
    float v[kMaxExperts / 32];
    uint32_t avail = 0;
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
        const int e = lane + 32 * j;
        if (32 * j < E)   // all loads issued before any use
            v[j] = __ldcg(lg + (e < E ? e : E - 1));
    }
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
        const int e = lane + 32 * j;
        float t = v[j];
        if (e < E) {
            if (t != t)
                t = -INFINITY;
            avail |= 1u << j;
        } else {
            t = -INFINITY;
        }
        v[j] = t;
    }
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) {
            const int e = lane + 32 * j;
            if (((avail >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < be))) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane)
            avail &= ~(1u << (be >> 5));
        if (lane == 0) {
            sel[s] = be;
            wt[s] = bv;
        }
    }
    __syncwarp();
    const float lmax = wt[0];
    const float l = lane < k ? wt[lane] : -INFINITY;
    const float e = lane < k ? expf(l - lmax) : 0.0f;
    float sum = e;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, off);
    __syncwarp();
    if (lane < k)
        wt[lane] = e / sum;
}

}  // namespace rt
}  // namespace moe
