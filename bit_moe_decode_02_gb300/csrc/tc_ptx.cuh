// tc_ptx.cuh -- device helpers shared by the tensor-core kernels (the batched
// grouped GEMM and the tensor-core decode layer): mbarriers, bulk copies,
// tcgen05 (tensor memory, block-scaled MMA), bf16 conversions and the OCP MX
// quantiser.  Included by .cu files only.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"

namespace moe {
namespace tc {

__device__ __forceinline__ uint32_t su32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(su32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking test of one phase of an mbarrier (try_wait may suspend the
// thread for a while before it reports an incomplete phase).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(su32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait on one phase of an mbarrier; on give-up record a timeout and
// return false (the caller carries on: every loop of these kernels is bounded).
// Not inlined: the kernels wait at many places, and one copy keeps the code
// small enough for the instruction caches.
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status)
{
#pragma unroll 1
    for (int i = 0; i < (1 << 22); ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
    return false;
}

// Bulk copy global -> shared completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(su32(dst)), "l"(src), "r"(bytes), "r"(su32(bar)) : "memory");
}

// L2 policy for data read once per call (streamed weights): evict first, so
// it does not push out what is reused (activations, partial sums, code).
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void bulk_copy_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(su32(dst)), "l"(src), "r"(bytes), "r"(su32(bar)), "l"(pol) : "memory");
}

// Shared-memory matrix descriptor, no swizzle, K-major canonical layout:
// 8-row x 16-byte core matrices, `lbo` bytes between core matrices along K,
// `sbo` bytes between 8-row groups; bits 46..48 = 0b001 (tcgen05 descriptor).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 128 bits of shared memory (rows 16 bytes apart) into tensor
// memory columns col..col+3, replicated to all four lane quarters.
__device__ __forceinline__ void tc_cp_sf(uint32_t tcol, uint32_t saddr)
{
    const uint64_t d = smem_desc(saddr, 16, 128);
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tcol), "l"(d) : "memory");
}

// D[128 x N] (+)= A[128 x 64] * B[N x 64]^T with E8M0 block scales.
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accum)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
                 "[%0], %1, %2, %3, [%5], [%6], p;\n\t}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb) : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(su32(bar)) : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The SwiGLU form h = gc sigmoid(alpha gc) (uc + beta), gc = min(g, limit),
// uc = clamp(u, -limit, limit) (a NaN passes through).  alpha = 1, limit =
// +inf, beta = 0 is the plain silu(g) u, and gives its bits: -(1 g) = -g,
// u + 0 = u.
__device__ __forceinline__ float swiglu(float g, float u, float alpha, float limit, float beta)
{
    if (g > limit)
        g = limit;
    if (u > limit)
        u = limit;
    if (u < -limit)
        u = -limit;
    return g / (1.0f + expf(-(alpha * g))) * (u + beta);
}

// Grid-wide signalling through global counters and flags (gpu scope).
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long atom_add_release_u64(unsigned long long* p, unsigned long long v)
{
    unsigned long long old;
    asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
// The counters only grow: every CTA adds 1 per call, so a call's count is
// complete at the next multiple of G above what this CTA's own add saw.
__device__ __forceinline__ unsigned long long count_target(unsigned long long old, int G)
{
    return (old / (unsigned long long)G + 1ull) * (unsigned long long)G;
}
// Add without waiting for the old value (the arrival at a grid barrier whose
// target is already known), with release semantics.
__device__ __forceinline__ void red_add_release_u64(unsigned long long* p, unsigned long long v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Wait (one thread) until a grid counter reaches `tgt`; gives up after `limit`
// polls and records a timeout.
__device__ __forceinline__ void wait_count(const unsigned long long* cnt, unsigned long long tgt, int limit, int* status)
{
    int spins = 0;
#pragma unroll 1
    while (ld_acquire_u64(cnt) < tgt) {
        if (++spins > limit) {
            atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
            break;
        }
    }
}

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f2bf16_rne(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x40);   // quiet NaN
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// ------------------------------------------------------------ MX quantiser

// Two fp32 values -> one byte of E2M1 codes (lo in the low nibble), round to
// nearest even, saturating at +-6.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// One block of 32 values -> 16 code bytes (4 words, element 2j in the low
// nibble of byte j) and the E8M0 scale byte.  The scale byte is the exponent
// field of amax minus 2, floored at 0: X = floor(log2 amax) - 2 clamped to
// -127 (amax < 2^-124, including 0 and subnormals, gives byte 0); amax = 0
// gives +0 codes.  v * 2^-X is exact in fp32 down to results far below the
// smallest E2M1 step, so every rounding decision is the exact one.
__device__ __forceinline__ uint32_t mx_block(const float (&v)[32], uint32_t (&code)[4])
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        amax = fmaxf(amax, fabsf(v[i]));
    const int ef = (int)((__float_as_uint(amax) >> 23) & 0xff);
    const uint32_t sbyte = ef > 2 ? (uint32_t)(ef - 2) : 0u;
    const float inv = __uint_as_float((254u - sbyte) << 23);    // 2^(127 - sbyte) = 2^-X
    const bool zero = amax == 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int i = 8 * w + 2 * b;
            word |= e2m1x2(v[i] * inv, v[i + 1] * inv) << (8 * b);
        }
        code[w] = zero ? 0u : word;
    }
    return sbyte;
}

// Fence ordering this thread's earlier generic-proxy shared-memory writes
// before later async-proxy (tensor core, bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// E2M1 code byte (two codes) -> the two values as fp32 (exact).
__device__ __forceinline__ float2 e2m1x2_to_f32(uint32_t byte)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h2) : "r"(byte));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

}  // namespace tc
}  // namespace moe
