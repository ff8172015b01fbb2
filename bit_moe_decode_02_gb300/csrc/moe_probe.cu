// moe_probe.cu -- the HBM streaming floor of a decode layer's weight bytes on
// this GPU: the same copy engine and stage sizes the decode kernels use, and
// nothing else.  n regions (one per layer) are read in sequence with a grid
// barrier between them, as dependent decode layers are; every CTA streams its
// share of a region into a shared-memory ring with bulk copies (4 stages of
// 32 KB in flight) and consumes nothing.  Measurement only: no forward path
// calls it.
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kProbeStage = 32768;
constexpr int kProbeDepth = 4;

__global__ void __launch_bounds__(32, 1)
    stream_read_kernel(const uint8_t* base, long long region_stride, long long bytes, int nregions,
                       unsigned long long* cnt, int spin_limit, int* status)
{
    extern __shared__ __align__(128) uint8_t pbuf[];
    __shared__ __align__(8) uint64_t bar[kProbeDepth];
    const int lane = threadIdx.x, G = gridDim.x, b = blockIdx.x;
    if (lane == 0) {
        for (int i = 0; i < kProbeDepth; ++i)
            mbar_init(&bar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    // this CTA's share of a region: [b0, b1), 16-byte aligned
    const long long per = ((bytes + G - 1) / G + 15) / 16 * 16;
    const long long b0 = (long long)b * per < bytes ? (long long)b * per : bytes;
    const long long b1 = b0 + per < bytes ? b0 + per : bytes;
    const long long nst = (b1 - b0 + kProbeStage - 1) / kProbeStage;
    uint32_t used = 0;   // stages issued so far on this CTA (the ring's phases follow it)
    unsigned long long tgt = 0;
    for (int r = 0; r < nregions; ++r) {
        if (lane == 0) {
            const uint8_t* src = base + (long long)r * region_stride + b0;
            auto issue = [&](long long s) {
                const uint32_t slot = (used + (uint32_t)s) % kProbeDepth;
                const long long off = s * kProbeStage;
                const uint32_t n = (uint32_t)((b1 - b0) - off < kProbeStage ? (b1 - b0) - off : kProbeStage);
                mbar_expect_tx(&bar[slot], n);
                bulk_copy(pbuf + slot * kProbeStage, src + off, n, &bar[slot]);
            };
            for (long long s = 0; s < nst && s < kProbeDepth; ++s)
                issue(s);
            for (long long s = 0; s < nst; ++s) {
                const uint32_t k = used + (uint32_t)s;
                if (!mbar_wait(&bar[k % kProbeDepth], (k / kProbeDepth) & 1, status))
                    break;
                if (s + kProbeDepth < nst)
                    issue(s + kProbeDepth);
            }
            used += (uint32_t)nst;
            // the next region starts after every CTA has this one (a dependent layer)
            const unsigned long long old = atom_add_release_u64(cnt, 1ull);
            tgt = r == 0 ? count_target(old, G) : tgt + (unsigned long long)G;
            wait_count(cnt, tgt, spin_limit, status);
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_stream_read(const uint8_t* base, long long region_stride, long long bytes, int nregions,
                               unsigned long long* cnt, int spin_limit, int* status, int grid, cudaStream_t s)
{
    const size_t smem = (size_t)kProbeStage * kProbeDepth;
    cudaError_t e = cudaFuncSetAttribute(stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    stream_read_kernel<<<grid, 32, smem, s>>>(base, region_stride, bytes, nregions, cnt, spin_limit, status);
    return cudaGetLastError();
}

}  // namespace moe
