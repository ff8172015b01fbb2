// route.cuh -- the router shared by the decode kernels: per token, the top-k
// of E logits and a softmax over the k selected ("Sovereign gpt-oss-20B
// (MXFP4) on Apple Silicon", section 3: top-4 routing; GPU top-k on the
// serving path, "Amortizing the per-token host-sync setup tax ...", section 3).
#pragma once
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {
namespace rt {

constexpr int kTopkRegs = kMaxExperts / 32;   // logits held per lane

// One warp: logit e of a token to lane e % 32, register e / 32 (NaN as -inf,
// absent experts as -inf), for E <= 32 * NR.  All loads are issued before any
// use, so a warp can hold several tokens' loads in flight.
template <int NR = kTopkRegs>
__device__ __forceinline__ void topk_load(const float* __restrict__ lg, int E, float (&v)[NR])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int e = lane + 32 * j;
        if (32 * j < E)
            v[j] = __ldcg(lg + (e < E ? e : E - 1));
    }
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int e = lane + 32 * j;
        const float t = v[j];
        v[j] = e < E && t == t ? t : -INFINITY;
    }
}

// One warp: top-k of the loaded logits (largest first; ties to the lower
// index), then softmax over the k selected.  Lane 0 writes sel[0..k) and the
// weights wt[0..k).
template <int NR = kTopkRegs>
__device__ __forceinline__ void topk_select(float (&v)[NR], int E, int k, int* sel, float* wt)
{
    const int lane = threadIdx.x & 31;
    uint32_t avail = 0;
#pragma unroll
    for (int j = 0; j < NR; ++j)
        if (lane + 32 * j < E)
            avail |= 1u << j;
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NR; ++j) {
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

// One warp, one token: load, then select.
template <int NR = kTopkRegs>
__device__ __forceinline__ void warp_topk_n(const float* __restrict__ lg, int E, int k, int* sel, float* wt)
{
    float v[NR];
    topk_load<NR>(lg, E, v);
    topk_select<NR>(v, E, k, sel, wt);
}
__device__ __forceinline__ void warp_topk(const float* __restrict__ lg, int E, int k, int* sel, float* wt)
{
    warp_topk_n<kTopkRegs>(lg, E, k, sel, wt);
}
// The same, with the register count taken from E (one copy of the code runs).
__device__ __forceinline__ void warp_topk_fit(const float* __restrict__ lg, int E, int k, int* sel, float* wt)
{
    if (E <= 32)
        warp_topk_n<1>(lg, E, k, sel, wt);
    else if (E <= 64)
        warp_topk_n<2>(lg, E, k, sel, wt);
    else if (E <= 128)
        warp_topk_n<4>(lg, E, k, sel, wt);
    else
        warp_topk_n<8>(lg, E, k, sel, wt);
}

}  // namespace rt
}  // namespace moe
