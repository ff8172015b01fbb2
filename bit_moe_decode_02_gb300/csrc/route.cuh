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
// index), then softmax over the k selected.  Lanes s < k write sel[s] and the
// weight wt[s].  Each round is two warp reductions: the maximum of an
// order-preserving integer key of the logits (redux.sync), then the lowest
// expert index among the lanes holding it.  -0 is taken as +0 first, so equal
// logits stay ties exactly as under a float comparison.  The softmax takes the
// k selected logits from registers: exp(l - l_max) summed by a fixed
// butterfly, so the result does not depend on timing.
__device__ __forceinline__ uint32_t order_key(float v)
{
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

template <int NR = kTopkRegs>
__device__ __forceinline__ void topk_select(float (&v)[NR], int E, int k, int* sel, float* wt)
{
    const int lane = threadIdx.x & 31;
    uint32_t key[NR];
    uint32_t avail = 0;
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        key[j] = order_key(v[j]);
        if (lane + 32 * j < E)
            avail |= 1u << j;
    }
    float myv = -INFINITY, vmax = -INFINITY;
    int mye = 0;
    for (int s = 0; s < k; ++s) {
        // this lane's best available key, ties to the lower register (lower index)
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int j = NR - 1; j >= 0; --j)
            if (((avail >> j) & 1u) && key[j] >= bk) {
                bk = key[j];
                bj = j;
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t be = __reduce_min_sync(0xffffffffu, (bk == mk && avail) ? (uint32_t)(lane + 32 * bj)
                                                                               : 0xffffffffu);
        if ((int)(be & 31u) == lane)
            avail &= ~(1u << (be >> 5));
        const float bv = key_value(mk);
        if (s == 0)
            vmax = bv;
        if (lane == s) {
            myv = bv;
            mye = (int)be;
        }
    }
    const float e = lane < k ? expf(myv - vmax) : 0.0f;
    float sum = e;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        sel[lane] = mye;
        wt[lane] = e / sum;
    }
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
