// moe_decode.cu -- sm_103a kernels of the 4-bit routed-expert decode layer.
//
// One layer is one persistent launch (one CTA per SM, all co-resident):
//
//   prologue  every CTA routes the M tokens itself (top-k of the router
//             logits, softmax over the selected) and lists the distinct
//             selected experts ("units"); thread 0 starts bulk copies
//             (cp.async.bulk, TMA engine) of the CTA's first weight slabs into
//             a shared-memory ring; the warps turn their K-slice of x into
//             MMA B fragments.
//   gate_up   items (unit, 16 gate rows + the matching 16 up rows), dealt
//             round-robin over the CTAs; the 12 warps split K, decode E2M1 /
//             int4 codes in registers into f16 A fragments and run
//             m16n8k16 MMAs (tokens on the N side, so M = 1..4 costs the same),
//             apply the block scales in fp32, sum the warps' partials in
//             shared memory and write h = silu(gate) * up (fp32).  Each item
//             bumps its unit's completion counter.
//   down      items (unit, 16 output rows); the slabs were already streamed
//             into the ring behind the gate_up items; before its first item of
//             a unit a CTA waits (bounded) until every CTA has finished that
//             unit's gate_up items, then multiplies against h split into f16
//             hi + lo parts (so h keeps ~22 bits: it is never rounded to 16),
//             adds the bias, and the last CTA to finish a 16-row output slab
//             forms out = bf16(r + sum_s w_s * y_s) in routing-slot order.
//
// The pages' kernel for this step ("Sovereign gpt-oss-20B (MXFP4) on Apple
// Silicon", sections 3-4: 16-byte coalesced loads with on-chip dequant, several
// SIMD groups sharing a row with a cross-group fp32 sum; one command buffer
// per decode) is prior art.  On GB300 a CUDA-core decode-and-FMA loop costs
// about five instructions per weight, which is more issue time than the HBM
// stream takes; decoding straight into MMA fragments brings that near one.
//
// Numerics: E2M1 -> f16 by the hardware cvt (exact); int4 -> f16 as
// (1024 + q) - 1032 (exact); x enters as f16 after an exact power-of-two
// rescale per (warp, token) (bf16 fits f16's 11-bit significand); products
// and the in-MMA sums are fp32; each E8M0 / fp16 block scale multiplies the
// fp32 sum of its block once.  No flush to zero (the denormal hazard noted on
// the TinyTitan tracker, D108).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "../../include/moe.h"
#include "moe_internal.h"
#include "route.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arm `bar` for `bytes` and start a bulk copy global -> shared completing on it.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for a phase of an mbarrier; on give-up record a timeout.
__device__ __forceinline__ void mbar_wait(uint64_t* bar, uint32_t parity, int* status)
{
    for (int i = 0; i < (1 << 22); ++i)
        if (mbar_try_wait(bar, parity))
            return;
    atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
}

// Barrier among `nthreads` threads (a multiple of 32) of the CTA, id 1..15.
__device__ __forceinline__ void named_barrier(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Order this thread's earlier generic-proxy global accesses before later
// bulk-copy (async proxy) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, const float (&c)[4])
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// d = a * b (+ d unless `restart`): the first MMA of a scale block starts from 0.
__device__ __forceinline__ void mma_step(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         bool restart)
{
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    if (restart)
        mma16816(d, a, b0, b1, zero);
    else
        mma16816(d, a, b0, b1, d);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f)
{
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ __half2 as_half2(uint32_t u)
{
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return h;
}

// ---------------------------------------------------------------- decoding

// One code word of a slab -> the four f16x2 A registers of one m16n8k16 MMA.
//   MXFP4: byte i holds the two E2M1 codes of register i (low nibble first).
//   int4 : register i holds nibbles i and i+4 (code - 8).
template <int FMT>
__device__ __forceinline__ void decode_a(uint32_t w, uint32_t (&a)[4])
{
    if constexpr (FMT == FMT_MXFP4) {
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
            "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
            "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
            "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
            : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
            : "r"(w));
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t t = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;   // fp16 1024 + q
            a[i] = h2_bits(__hsub2(as_half2(t), as_half2(0x64086408u)));    // - 1032 = q - 8
        }
    }
}

// E8M0 byte -> fp32 2^(s-127): exact for every byte (0 -> 2^-127, 255 -> NaN).
__device__ __forceinline__ float e8m0_exact(uint32_t s)
{
    const uint32_t bits = s == 0 ? 0x00400000u : (s == 255 ? 0x7fc00000u : (s << 23));
    return __uint_as_float(bits);
}
// Same for bytes 1..254 only.
__device__ __forceinline__ float e8m0_fast(uint32_t word, int byte)
{
    return __uint_as_float(((word >> (8 * byte)) & 0xffu) << 23);
}

// Scales of rows g (sg) and g+8 (sh) for block b (0/1: K 0..31 / 32..63 of
// the segment), kept as the raw entry and decoded at use.  With one scale per
// segment both blocks read the same pair.
template <int FMT, int SB>
struct SegScales {
    uint32_t w0, w1;
    __device__ __forceinline__ void load(const uint8_t* entry)
    {
        if constexpr (SB == 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(entry);
            w0 = v.x;
            w1 = v.y;
        } else {
            w0 = *reinterpret_cast<const uint32_t*>(entry);
            w1 = 0u;
        }
    }
    __device__ __forceinline__ float sg(int b, bool exact) const
    {
        if constexpr (FMT == FMT_MXFP4)
            return exact ? e8m0_exact((w0 >> (16 * b)) & 0xffu) : e8m0_fast(w0, 2 * b);
        else if constexpr (SB == 4)
            return __low2float(as_half2(w0));
        else
            return __low2float(as_half2(b ? w1 : w0));
    }
    __device__ __forceinline__ float sh(int b, bool exact) const
    {
        if constexpr (FMT == FMT_MXFP4)
            return exact ? e8m0_exact((w0 >> (16 * b + 8)) & 0xffu) : e8m0_fast(w0, 2 * b + 1);
        else if constexpr (SB == 4)
            return __high2float(as_half2(w0));
        else
            return __high2float(as_half2(b ? w1 : w0));
    }
};

// This warp's partial products for one item: rows g / g+8 and columns
// 2t / 2t+1 of the m16n8 tiles, summed over this warp's segments of K.
//   gu_item_mma: acc0 = gate slab, acc1 = up slab, both against the x
//                fragments kept in shared memory (xf: [seg][j][lane] uint2).
//   dn_item_mma: acc0 = the slab against h = hi + lo (fragments in registers).
// The segment's code words and scales are read first; the two MMA chains of
// each step (gate / up, or hi / lo) are independent.
template <int FMT, int SB>
__device__ __forceinline__ void gu_item_mma(const uint8_t* slab0, const uint8_t* slab1, int codes_bytes,
                                            int nseg, const uint2* xf, bool exact, float (&acc0)[4],
                                            float (&acc1)[4])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2;
    constexpr bool one_scale = (FMT == FMT_INT4 && SB == 4);
#pragma unroll
    for (int si = 0; si < kMaxSegPerWarp; ++si) {
        const int q = warp + kComputeWarps * si;
        if (q < nseg) {
            const uint4 c0 = lds128(slab0 + ((size_t)q * 32 + lane) * 16);
            const uint4 c1 = lds128(slab1 + ((size_t)q * 32 + lane) * 16);
            SegScales<FMT, SB> s0, s1;
            s0.load(slab0 + codes_bytes + ((size_t)q * 8 + g) * SB);
            s1.load(slab1 + codes_bytes + ((size_t)q * 8 + g) * SB);
            uint2 bxv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                bxv[j] = xf[(si * 4 + j) * 32 + lane];
            const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w};
            const uint32_t w1[4] = {c1.x, c1.y, c1.z, c1.w};
            float d0[4], d1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool first = one_scale ? (j == 0) : ((j & 1) == 0);
                uint32_t a0[4], a1[4];
                decode_a<FMT>(w0[j], a0);
                decode_a<FMT>(w1[j], a1);
                mma_step(d0, a0, bxv[j].x, bxv[j].y, first);
                mma_step(d1, a1, bxv[j].x, bxv[j].y, first);
                const bool last = one_scale ? (j == 3) : ((j & 1) == 1);
                if (last) {
                    const int blk = one_scale ? 0 : (j >> 1);
                    const float g0 = s0.sg(blk, exact), h0 = s0.sh(blk, exact);
                    const float g1 = s1.sg(blk, exact), h1 = s1.sh(blk, exact);
                    acc0[0] = fmaf(d0[0], g0, acc0[0]);
                    acc0[1] = fmaf(d0[1], g0, acc0[1]);
                    acc0[2] = fmaf(d0[2], h0, acc0[2]);
                    acc0[3] = fmaf(d0[3], h0, acc0[3]);
                    acc1[0] = fmaf(d1[0], g1, acc1[0]);
                    acc1[1] = fmaf(d1[1], g1, acc1[1]);
                    acc1[2] = fmaf(d1[2], h1, acc1[2]);
                    acc1[3] = fmaf(d1[3], h1, acc1[3]);
                }
            }
        }
    }
}

template <int FMT, int SB>
__device__ __forceinline__ void dn_item_mma(const uint8_t* slab, int codes_bytes, int nseg,
                                            const uint32_t (&bh)[kMaxSegPerWarp][4][2],
                                            const uint32_t (&bl)[kMaxSegPerWarp][4][2], bool exact,
                                            float (&acc)[4])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2;
    constexpr bool one_scale = (FMT == FMT_INT4 && SB == 4);
#pragma unroll
    for (int si = 0; si < kMaxSegPerWarp; ++si) {
        const int q = warp + kComputeWarps * si;
        if (q < nseg) {
            const uint4 c0 = lds128(slab + ((size_t)q * 32 + lane) * 16);
            SegScales<FMT, SB> s0;
            s0.load(slab + codes_bytes + ((size_t)q * 8 + g) * SB);
            const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w};
            float d0[4], d1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool first = one_scale ? (j == 0) : ((j & 1) == 0);
                uint32_t a0[4];
                decode_a<FMT>(w0[j], a0);
                mma_step(d0, a0, bh[si][j][0], bh[si][j][1], first);
                mma_step(d1, a0, bl[si][j][0], bl[si][j][1], first);
                const bool last = one_scale ? (j == 3) : ((j & 1) == 1);
                if (last) {
                    const int blk = one_scale ? 0 : (j >> 1);
                    const float g0 = s0.sg(blk, exact), h0 = s0.sh(blk, exact);
                    acc[0] = fmaf(d0[0] + d1[0], g0, acc[0]);
                    acc[1] = fmaf(d0[1] + d1[1], g0, acc[1]);
                    acc[2] = fmaf(d0[2] + d1[2], h0, acc[2]);
                    acc[3] = fmaf(d0[3] + d1[3], h0, acc[3]);
                }
            }
        }
    }
}

// Exponent p with amax * 2^-p in [2^14, 2^15) (p = 0 for 0, inf or NaN).
__device__ __forceinline__ int prescale_exp(float amax)
{
    const uint32_t e = (__float_as_uint(amax) >> 23) & 0xffu;
    if (e == 0 || e == 255)
        return 0;
    int p = (int)e - 127 - 14;
    return p < -126 ? -126 : (p > 126 ? 126 : p);
}
__device__ __forceinline__ float exp2i(int p) { return __uint_as_float((uint32_t)(p + 127) << 23); }

// ---------------------------------------------------------------- routing

using rt::warp_topk;

struct RouteSmem {
    int sel[kMaxTokens][kMaxTopK];
    float wt[kMaxTokens][kMaxTopK];
    int nu;                                         // distinct experts
    int unit_expert[kMaxUnits];                     // ascending expert index
    signed char unit_slot[kMaxUnits][kMaxTokens];   // slot of the unit in token m's list, or -1
    unsigned char unit_of[kMaxExperts];
};

// All threads: route the M tokens into shared memory and list the units
// (distinct selected experts in ascending order, with each token's slot).
__device__ void route_block(const float* __restrict__ logits, int M, int E, int k, RouteSmem& rs)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < M)
        warp_topk(logits + (size_t)warp * E, E, k, rs.sel[warp], rs.wt[warp]);
    __syncthreads();
    if (warp == 0) {
        // lane w < 8 owns experts 32w .. 32w+31 of the selection bitmap
        uint32_t bits = 0;
        if (lane < kMaxExperts / 32)
            for (int m = 0; m < M; ++m)
                for (int s = 0; s < k; ++s) {
                    const int e = rs.sel[m][s];
                    if ((e >> 5) == lane)
                        bits |= 1u << (e & 31);
                }
        const int cnt = __popc(bits);
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off)
                incl += v;
        }
        int u = incl - cnt;
        while (bits) {
            const int e = lane * 32 + __ffs(bits) - 1;
            bits &= bits - 1;
            rs.unit_of[e] = (unsigned char)u;
            rs.unit_expert[u] = e;
            ++u;
        }
        const int nu = __shfl_sync(0xffffffffu, incl, 31);
        for (int x = lane; x < nu * kMaxTokens; x += 32)
            rs.unit_slot[x / kMaxTokens][x % kMaxTokens] = -1;
        __syncwarp();
        for (int x = lane; x < M * k; x += 32) {
            const int m = x / k, s = x % k;
            rs.unit_slot[rs.unit_of[rs.sel[m][s]]][m] = (signed char)s;
        }
        if (lane == 0)
            rs.nu = nu;
    }
    __syncthreads();
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Number of items i < total with i % G == b.
__device__ __forceinline__ int my_count(int b, int total, int G) { return total > b ? (total - b + G - 1) / G : 0; }

// ================================================================ layer kernel
//
// Warp roles: warps 0..11 compute (MMA), warp 12 produces (bulk copies of the
// layer input and of the weight slabs into the ring), warp 13 signals (the
// gpu-scope fences and counter updates that publish h and the down partials,
// batched over every item that has finished; the last-arriver combine; bulk
// copies of each unit's h into a double-buffered staging area once every CTA
// has finished that unit's gate_up items).  All hand-offs inside the CTA are
// mbarriers, so the compute warps never wait on a gpu-scope fence.
//
// Schedule of a CTA: its gate_up items (dealt round-robin over the CTAs, in
// unit order), then its down items (likewise).  The down slabs stream into the
// ring behind the last gate_up items, and a unit's h is staged as soon as that
// unit is complete, so the down phase starts without a bubble.
//
// Ring entries of a CTA: entry 0 is the layer input (x, or the residual to be
// normalised); gate_up item i uses entries 1 + 2i (gate) and 2 + 2i (up);
// down item j uses entry 1 + 2 n_gu + j.  Entry e lives in slot e % NS.

constexpr int kEpiDepth = 8;       // items in flight between the compute and the signalling warps

// Item `it` of CTA b: gate_up item it (< n_gu) or down item it - n_gu;
// returns its global index q and whether it is a down item.
__device__ __forceinline__ int item_q(int it, int n_gu, int b, int G, bool& down)
{
    down = it >= n_gu;
    return b + G * (down ? it - n_gu : it);
}
__device__ __forceinline__ int item_entry(int it, int n_gu) { return it < n_gu ? 1 + 2 * it : 1 + n_gu + it; }

template <int FMT, int SB>
__global__ void __launch_bounds__(kThreads, 1) layer_kernel(const LayerParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kMaxSlots];
    __shared__ __align__(8) uint64_t empty[kMaxSlots];
    __shared__ __align__(8) uint64_t hx_full[2];
    __shared__ __align__(8) uint64_t hx_empty[2];
    __shared__ __align__(8) uint64_t epi[kEpiDepth];
    __shared__ __align__(8) uint64_t sig_done[kEpiDepth];
    __shared__ RouteSmem rs;
    __shared__ float nrm[kComputeWarps][kMaxTokens];
    __shared__ float hmax_s[2][kMaxTokens];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int G = gridDim.x, b = blockIdx.x;
    const int NS = p.nslots;
    uint8_t* ring = smem;
    float* hbuf = reinterpret_cast<float*>(smem + (size_t)NS * p.slot_bytes);   // [2][mmax][I]
    float* red = hbuf + 2 * (size_t)p.mmax * p.I;   // [2][kComputeWarps][32 rows][kMaxTokens]
    uint2* xfrag = reinterpret_cast<uint2*>(red + 2 * kComputeWarps * 32 * kMaxTokens);   // [warp][seg][j][lane]
    auto red_at = [&](int bb, int w, int row, int col) -> float& {
        return red[((bb * kComputeWarps + w) * 32 + row) * kMaxTokens + col];
    };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kComputeWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&hx_full[i], 1);
            mbar_init(&hx_empty[i], kComputeWarps);
        }
        for (int i = 0; i < kEpiDepth; ++i) {
            mbar_init(&epi[i], 64);
            mbar_init(&sig_done[i], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();   // the previous kernel (prior layer, or the writer of x / logits) is complete
    if (tid == 0)   // ring entry 0: the layer input rows, which do not depend on the routing
        bulk_load(ring, p.x ? (const void*)p.x : (const void*)p.resid, (uint32_t)(p.M * p.H * 2), &full[0]);
    route_block(p.logits, p.M, p.E, p.k, rs);   // last block-wide barrier of the kernel
    pdl_launch_dependents();

    const int nu = rs.nu, M = p.M;
    const int gpu = p.I / kSlabRows, dpu = p.H / kSlabRows;   // items per unit
    const int nseg_h = p.H / 64, nseg_i = p.I / 64;
    const int n_gu = my_count(b, nu * gpu, G), n_dn = my_count(b, nu * dpu, G);
    const int nitems = n_gu + n_dn;
    if (b == 0 && tid == 0 && p.nu_out)
        *p.nu_out = nu;

    // ============================================================ producer
    if (warp == kComputeWarps) {
        if (lane == 0) {
            for (int it = 0; it < nitems; ++it) {
                bool down;
                const int q = item_q(it, n_gu, b, G, down);
                for (int part = 0; part < (down ? 1 : 2); ++part) {
                    const int ent = item_entry(it, n_gu) + part;
                    const int slot = ent % NS;
                    if (ent >= NS) {
                        mbar_wait(&empty[slot], (uint32_t)(((ent / NS) - 1) & 1), p.status);
                        fence_proxy_async();
                    }
                    const uint8_t* src;
                    int bytes;
                    if (!down) {
                        const int u = q / gpu, pp = q % gpu;
                        src = p.gu + (size_t)rs.unit_expert[u] * p.gu_expert_bytes +
                              (size_t)(part ? gpu + pp : pp) * p.gu_slab_bytes;
                        bytes = p.gu_slab_bytes;
                    } else {
                        const int u = q / dpu, sl = q % dpu;
                        src = p.dn + (size_t)rs.unit_expert[u] * p.dn_expert_bytes + (size_t)sl * p.dn_slab_bytes;
                        bytes = p.dn_slab_bytes;
                    }
                    bulk_load(ring + (size_t)slot * p.slot_bytes, src, (uint32_t)bytes, &full[slot]);
                }
            }
        }
        return;
    }

    // ============================================================ signaller
    if (warp == kComputeWarps + 1) {
        int staged = 0;          // units of the down items staged so far
        int scan = 0;            // next item to look at for the next unit to stage
        int last_u = -1;
        int ev = 0;
        while (ev < nitems) {
            bool got = false;
            for (int it = 0; it < (1 << 22) && !got; ++it) {
                // stage h of the next down unit once it is complete and its buffer is free
                int stage_u = -1;
                if (lane == 0) {
                    while (scan < n_dn && (b + G * scan) / dpu == last_u)
                        ++scan;
                    if (scan < n_dn) {
                        const int u = (b + G * scan) / dpu;
                        const int bb = staged & 1;
                        const bool buf_free = staged < 2 ||
                            mbar_try_wait(&hx_empty[bb], (uint32_t)(((staged >> 1) - 1) & 1));
                        if (buf_free && ld_acquire(p.done + u) >= (unsigned)gpu)
                            stage_u = u;
                    }
                }
                stage_u = __shfl_sync(0xffffffffu, stage_u, 0);
                if (stage_u >= 0) {
                    const int bb = staged & 1;
                    if (lane == 0) {
                        fence_proxy_async_global();
                        uint32_t bytes = 0;
                        for (int m = 0; m < M; ++m) {
                            hmax_s[bb][m] = __uint_as_float(__ldcg(p.hmax + stage_u * kMaxTokens + m));
                            if (rs.unit_slot[stage_u][m] >= 0)
                                bytes += (uint32_t)p.I * 4u;
                        }
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                                     ::"r"(smem_u32(&hx_full[bb])), "r"(bytes) : "memory");
                        for (int m = 0; m < M; ++m) {
                            const int slot = rs.unit_slot[stage_u][m];
                            if (slot >= 0)
                                asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes"
                                             " [%0], [%1], %2, [%3];"
                                             ::"r"(smem_u32(hbuf + ((size_t)bb * p.mmax + m) * p.I)),
                                               "l"(p.h + ((size_t)m * p.kmax + slot) * p.I),
                                               "r"((uint32_t)p.I * 4u), "r"(smem_u32(&hx_full[bb]))
                                             : "memory");
                        }
                        last_u = stage_u;
                    }
                    ++staged;
                }
                got = __shfl_sync(0xffffffffu,
                                  mbar_try_wait(&epi[ev % kEpiDepth], (uint32_t)((ev / kEpiDepth) & 1)) ? 1 : 0,
                                  0) != 0;
                if (!got && stage_u < 0)
                    __nanosleep(64);
            }
            if (!got && lane == 0)
                atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
            // every further item whose epilogue is already done joins this batch
            int end = ev + 1;
            if (lane == 0)
                while (end < nitems && end < ev + kEpiDepth &&
                       mbar_try_wait(&epi[end % kEpiDepth], (uint32_t)((end / kEpiDepth) & 1)))
                    ++end;
            end = __shfl_sync(0xffffffffu, end, 0);
            if (lane == 0)
                __threadfence();   // the batch's h / ypart stores (acquired through epi) first
            for (; ev < end; ++ev) {
                bool down;
                const int q = item_q(ev, n_gu, b, G, down);
                if (!down) {
                    if (lane == 0)
                        atomicAdd(p.done + q / gpu, 1u);
                } else {
                    const int sl = q % dpu;
                    int last = 0;
                    if (lane == 0) {
                        last = atomicAdd(p.slab_cnt + sl, 1u) == (unsigned)nu - 1u;
                        if (last)
                            __threadfence();
                    }
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (last) {
                        // every unit's rows of this slab are in ypart: combine in slot order
                        for (int x = lane; x < kSlabRows * M; x += 32) {
                            const int r = x % kSlabRows, m = x / kSlabRows;
                            const int jj = sl * kSlabRows + r;
                            float acc = 0.f;
                            for (int k2 = 0; k2 < p.k; ++k2)
                                acc = fmaf(rs.wt[m][k2], __ldcg(p.ypart + ((size_t)m * p.kmax + k2) * p.H + jj), acc);
                            uint16_t* o = p.resid + (size_t)m * p.H + jj;
                            const float v = bf16_to_f32(__ldcg(o)) + acc;
                            *o = f32_to_bf16_rn(v);
                            if (p.out_f32)
                                p.out_f32[(size_t)m * p.H + jj] = v;
                        }
                        __syncwarp();
                        if (lane == 0)
                            p.slab_cnt[sl] = 0u;
                    }
                }
                if (lane == 0)
                    mbar_arrive(&sig_done[ev % kEpiDepth]);
                __syncwarp();
            }
        }
        if (lane == 0) {
            __threadfence();
            const unsigned old = atomicAdd(p.exit_cnt, 1u);
            if (old == (unsigned)G - 1u) {
                // every CTA is past its waits: reset the counters for the next call
                for (int u = 0; u < nu; ++u) {
                    p.done[u] = 0u;
                    for (int m = 0; m < kMaxTokens; ++m)
                        p.hmax[u * kMaxTokens + m] = 0u;
                }
                *p.exit_cnt = 0u;
                __threadfence();
            }
        }
        return;
    }

    // ============================================================ compute warps
    constexpr int kComputeThreads = kComputeWarps * 32;
    // ---- x fragments from ring entry 0 ([M][H] bf16)
    mbar_wait(&full[0], 0u, p.status);
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(ring);
    float inv = 1.0f;
    if (!p.x) {
        // weightless RMSNorm of the residual: x = bf16(r / sqrt(mean(r^2) + 1e-6))
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m) {
            float a = 0.0f;
            if (m < M)
                for (int i = tid; i < p.H / 2; i += kComputeThreads) {
                    const uint32_t w = reinterpret_cast<const uint32_t*>(xs + (size_t)m * p.H)[i];
                    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
                    a = fmaf(lo, lo, a);
                    a = fmaf(hi, hi, a);
                }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                a += __shfl_xor_sync(0xffffffffu, a, off);
            if (lane == 0)
                nrm[warp][m] = a;
        }
        named_barrier(1, kComputeThreads);
        if (g < M) {
            float tot = 0.0f;
            for (int w = 0; w < kComputeWarps; ++w)
                tot += nrm[w][g];
            inv = 1.0f / sqrtf(tot / (float)p.H + 1e-6f);
        }
    }
    uint32_t bx[kMaxSegPerWarp][4][2];
    float px[kMaxTokens];   // 2^p that undoes the prescale of token m's x fragment in this warp
    uint2* xf = xfrag + (size_t)warp * kMaxSegPerWarp * 4 * 32;
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(xs) + (size_t)(g < M ? g : 0) * (p.H / 2);
        float amax = 0.0f;
#pragma unroll
        for (int si = 0; si < kMaxSegPerWarp; ++si) {
            const int q = warp + kComputeWarps * si;
            const bool ok = q < nseg_h && g < M;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t w = ok ? src[(64 * q + 16 * j + 2 * t) / 2 + 4 * hf] : 0u;
                    if (!p.x) {
                        const float lo = __uint_as_float(w << 16) * inv;
                        const float hi = __uint_as_float(w & 0xffff0000u) * inv;
                        w = (uint32_t)f32_to_bf16_rn(lo) | ((uint32_t)f32_to_bf16_rn(hi) << 16);
                    }
                    bx[si][j][hf] = w;
                    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w << 16)),
                                             fabsf(__uint_as_float(w & 0xffff0000u))));
                }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[0]);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int pe = prescale_exp(amax);
        const float sdown = exp2i(-pe);
#pragma unroll
        for (int si = 0; si < kMaxSegPerWarp; ++si)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t hv[2];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const uint32_t w = bx[si][j][hf];
                    hv[hf] = h2_bits(__floats2half2_rn(__uint_as_float(w << 16) * sdown,
                                                       __uint_as_float(w & 0xffff0000u) * sdown));
                }
                xf[(si * 4 + j) * 32 + lane] = make_uint2(hv[0], hv[1]);
            }
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m)
            px[m] = exp2i(__shfl_sync(0xffffffffu, pe, 4 * m));
    }

    // ---- items in schedule order
    const int gu_codes = 8 * p.H, dn_codes = 8 * p.I;
    uint32_t bh[kMaxSegPerWarp][4][2], bl[kMaxSegPerWarp][4][2];
    float ph[kMaxTokens];
    int cur_u = -1, uj = -1;
    for (int it = 0; it < nitems; ++it) {
        bool down;
        const int q = item_q(it, n_gu, b, G, down);
        const int ent = item_entry(it, n_gu);
        const int bb = it & 1;
        const int ew = 2 * (it % (kComputeWarps / 2));     // this item's epilogue warps: ew, ew + 1
        const bool epi_warp = warp == ew || warp == ew + 1;
        const int et = tid - ew * 32;                      // 0..63 within the epilogue pair
        if (!down) {
            // ---------------- gate_up item: gate slab and up slab of (unit, 16 rows)
            const int u = q / gpu, pp = q % gpu;
            const int e = rs.unit_expert[u];
            const bool exact = p.special[2 * e] != 0;
            const int s0 = ent % NS, s1 = (ent + 1) % NS;
            mbar_wait(&full[s0], (uint32_t)((ent / NS) & 1), p.status);
            mbar_wait(&full[s1], (uint32_t)(((ent + 1) / NS) & 1), p.status);
            float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
            gu_item_mma<FMT, SB>(ring + (size_t)s0 * p.slot_bytes, ring + (size_t)s1 * p.slot_bytes,
                                 gu_codes, nseg_h, xf, exact, ag, au);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s0]);
                mbar_arrive(&empty[s1]);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col = 2 * t + c;
                if (col < kMaxTokens) {
                    red_at(bb, warp, g, col) = ag[c] * px[col];
                    red_at(bb, warp, g + 8, col) = ag[2 + c] * px[col];
                    red_at(bb, warp, 16 + g, col) = au[c] * px[col];
                    red_at(bb, warp, 16 + g + 8, col) = au[2 + c] * px[col];
                }
            }
            named_barrier(1, kComputeThreads);
            if (epi_warp) {
                if (it >= kEpiDepth)
                    mbar_wait(&sig_done[it % kEpiDepth], (uint32_t)(((it / kEpiDepth) - 1) & 1), p.status);
                const int r = et >> 2, m = et & 3;
                const int slot = m < M ? rs.unit_slot[u][m] : -1;
                uint32_t habs = 0u;
                if (slot >= 0) {
                    float gs = 0.f, us = 0.f;
                    for (int w = 0; w < kComputeWarps; ++w) {
                        gs += red_at(bb, w, r, m);
                        us += red_at(bb, w, 16 + r, m);
                    }
                    const int irow = pp * kSlabRows + r;
                    if (p.gu_bias) {
                        gs += bf16_to_f32(p.gu_bias[(size_t)e * 2 * p.I + irow]);
                        us += bf16_to_f32(p.gu_bias[(size_t)e * 2 * p.I + p.I + irow]);
                    }
                    const float hv = silu(gs) * us;
                    p.h[((size_t)m * p.kmax + slot) * p.I + irow] = hv;
                    habs = __float_as_uint(fabsf(hv));
                }
                // largest |h| of the item per token, for the down stage's prescale
#pragma unroll
                for (int off = 4; off < 32; off <<= 1)
                    habs = max(habs, __shfl_xor_sync(0xffffffffu, habs, off));
                if (lane < 4 && slot >= 0)
                    atomicMax(p.hmax + u * kMaxTokens + m, habs);
                mbar_arrive(&epi[it % kEpiDepth]);
            }
        } else {
            // ---------------- down item: 16 output rows of one unit
            const int u = q / dpu, sl = q % dpu;
            const int e = rs.unit_expert[u];
            if (u != cur_u) {
                cur_u = u;
                ++uj;
                const int hb = uj & 1;
                mbar_wait(&hx_full[hb], (uint32_t)((uj >> 1) & 1), p.status);
                const int slot = g < M ? rs.unit_slot[u][g] : -1;
                const float* hrow = hbuf + ((size_t)hb * p.mmax + (g < M ? g : 0)) * p.I;
                const float amax = slot >= 0 ? hmax_s[hb][g] : 0.0f;
                const int pe = prescale_exp(amax);
                const float sdown = exp2i(-pe);
#pragma unroll
                for (int si = 0; si < kMaxSegPerWarp; ++si) {
                    const int qq = warp + kComputeWarps * si;
                    const bool ok = qq < nseg_i && slot >= 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            float2 v = make_float2(0.f, 0.f);
                            if (ok)
                                v = *reinterpret_cast<const float2*>(hrow + 64 * qq + 16 * j + 2 * t + 8 * hf);
                            const float a0 = v.x * sdown, a1 = v.y * sdown;
                            const __half2 hi = __floats2half2_rn(a0, a1);
                            const float2 hif = __half22float2(hi);
                            bh[si][j][hf] = h2_bits(hi);
                            bl[si][j][hf] = h2_bits(__floats2half2_rn(a0 - hif.x, a1 - hif.y));
                        }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&hx_empty[hb]);
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m)
                    ph[m] = exp2i(__shfl_sync(0xffffffffu, pe, 4 * m));
            }
            const bool exact = p.special[2 * e + 1] != 0;
            const int s0 = ent % NS;
            mbar_wait(&full[s0], (uint32_t)((ent / NS) & 1), p.status);
            float ay[4] = {0.f, 0.f, 0.f, 0.f};
            dn_item_mma<FMT, SB>(ring + (size_t)s0 * p.slot_bytes, dn_codes, nseg_i, bh, bl, exact, ay);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s0]);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int col = 2 * t + c;
                if (col < kMaxTokens) {
                    red_at(bb, warp, g, col) = ay[c] * ph[col];
                    red_at(bb, warp, g + 8, col) = ay[2 + c] * ph[col];
                }
            }
            named_barrier(1, kComputeThreads);
            if (epi_warp) {
                if (it >= kEpiDepth)
                    mbar_wait(&sig_done[it % kEpiDepth], (uint32_t)(((it / kEpiDepth) - 1) & 1), p.status);
                const int r = et >> 2, m = et & 3;
                const int slot = m < M ? rs.unit_slot[u][m] : -1;
                if (slot >= 0) {
                    float y = 0.f;
                    for (int w = 0; w < kComputeWarps; ++w)
                        y += red_at(bb, w, r, m);
                    if (p.dn_bias)
                        y += bf16_to_f32(p.dn_bias[(size_t)e * p.H + sl * kSlabRows + r]);
                    p.ypart[((size_t)m * p.kmax + slot) * p.H + sl * kSlabRows + r] = y;
                }
                mbar_arrive(&epi[it % kEpiDepth]);
            }
        }
    }
}

// ================================================================ load-time repack

template <int FMT, int SB>
__global__ void repack_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                              int E, int N, int K, int group, uint8_t* __restrict__ out,
                              long long expert_bytes, int slab_bytes, uint32_t* special, int proj)
{
    const int nseg = K / 64, nslab = N / kSlabRows;
    const long long words = (long long)E * nslab * nseg * 32 * 4;
    const long long entries = (long long)E * nslab * nseg * 8;
    const size_t row_b = (size_t)K / 2;
    const int nsc = FMT == FMT_MXFP4 ? K / 32 : K / group;   // scales per row
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < words + entries;
         idx += (long long)gridDim.x * blockDim.x) {
        if (idx < words) {
            long long r = idx;
            const int j = (int)(r % 4); r /= 4;
            const int lane = (int)(r % 32); r /= 32;
            const int q = (int)(r % nseg); r /= nseg;
            const int slab = (int)(r % nslab);
            const int e = (int)(r / nslab);
            const int g = lane >> 2, t = lane & 3;
            const uint8_t* r0 = codes + ((size_t)e * N + (size_t)slab * kSlabRows + g) * row_b;
            const uint8_t* r1 = r0 + 8 * row_b;
            const int k0 = 64 * q + 16 * j;
            uint32_t word;
            if constexpr (FMT == FMT_MXFP4) {
                const int bi = k0 / 2 + t;
                word = (uint32_t)r0[bi] | ((uint32_t)r1[bi] << 8) | ((uint32_t)r0[bi + 4] << 16) |
                       ((uint32_t)r1[bi + 4] << 24);
            } else {
                auto nib = [&](const uint8_t* row, int k) -> uint32_t {
                    return (row[k >> 1] >> (4 * (k & 1))) & 0xfu;
                };
                const int c = k0 + 2 * t;
                word = nib(r0, c) | (nib(r1, c) << 4) | (nib(r0, c + 8) << 8) | (nib(r1, c + 8) << 12) |
                       (nib(r0, c + 1) << 16) | (nib(r1, c + 1) << 20) | (nib(r0, c + 9) << 24) |
                       (nib(r1, c + 9) << 28);
            }
            *reinterpret_cast<uint32_t*>(out + (size_t)e * expert_bytes + (size_t)slab * slab_bytes +
                                         ((size_t)q * 32 + lane) * 16 + 4 * j) = word;
        } else {
            long long r = idx - words;
            const int g = (int)(r % 8); r /= 8;
            const int q = (int)(r % nseg); r /= nseg;
            const int slab = (int)(r % nslab);
            const int e = (int)(r / nslab);
            const size_t row0 = (size_t)e * N + (size_t)slab * kSlabRows + g, row1 = row0 + 8;
            uint8_t* dst = out + (size_t)e * expert_bytes + (size_t)slab * slab_bytes + 8 * (size_t)K +
                           ((size_t)q * 8 + g) * SB;
            if constexpr (FMT == FMT_MXFP4) {
                const uint8_t s0 = scales[row0 * nsc + 2 * q], s1 = scales[row1 * nsc + 2 * q];
                const uint8_t s2 = scales[row0 * nsc + 2 * q + 1], s3 = scales[row1 * nsc + 2 * q + 1];
                dst[0] = s0; dst[1] = s1; dst[2] = s2; dst[3] = s3;
                const bool sp = s0 == 0 || s0 == 255 || s1 == 0 || s1 == 255 || s2 == 0 || s2 == 255 ||
                                s3 == 0 || s3 == 255;
                if (sp)
                    atomicOr(special + 2 * e + proj, 1u);
            } else {
                const uint16_t* s16 = reinterpret_cast<const uint16_t*>(scales);
                uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
                if constexpr (SB == 4) {
                    const int gi = (64 * q) / group;
                    d16[0] = s16[row0 * nsc + gi];
                    d16[1] = s16[row1 * nsc + gi];
                } else {
                    d16[0] = s16[row0 * nsc + 2 * q];
                    d16[1] = s16[row1 * nsc + 2 * q];
                    d16[2] = s16[row0 * nsc + 2 * q + 1];
                    d16[3] = s16[row1 * nsc + 2 * q + 1];
                }
            }
        }
    }
}

// ================================================================ debug kernels

// Element (n, k) of one projection read back from its slabs with the same
// decode as the layer kernel, times its scale, in fp32.
template <int FMT, int SB>
__global__ void dequant_kernel(const uint8_t* __restrict__ slabs, int N, int K, int slab_bytes,
                               float* __restrict__ out)
{
    const long long total = (long long)N * K;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx / K), k = (int)(idx % K);
        const int slab = n / kSlabRows, r = n % kSlabRows, gg = r & 7, hi = r >> 3;
        const int q = k / 64, k64 = k % 64, j = k64 / 16, kk = k64 % 16;
        const int t = (kk & 7) >> 1, second = kk >= 8, lane = 4 * gg + t;
        const uint8_t* base = slabs + (size_t)slab * slab_bytes;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(base + ((size_t)q * 32 + lane) * 16 + 4 * j);
        uint32_t a[4];
        decode_a<FMT>(w, a);
        const float2 f = __half22float2(as_half2(a[2 * second + hi]));
        const float v = (kk & 1) ? f.y : f.x;
        const uint8_t* ent = base + 8 * (size_t)K + ((size_t)q * 8 + gg) * SB;
        const int blk = k64 / 32;
        float s;
        if constexpr (FMT == FMT_MXFP4) {
            s = e8m0_exact(ent[hi + 2 * blk]);
        } else if constexpr (SB == 4) {
            s = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(ent)[hi]));
        } else {
            s = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(ent)[hi + 2 * blk]));
        }
        out[idx] = v * s;
    }
}

__global__ void route_kernel(const float* __restrict__ logits, int M, int E, int k, int* idx, float* w)
{
    const int tok = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (tok < M)
        warp_topk(logits + (size_t)tok * E, E, k, idx + (size_t)tok * k, w + (size_t)tok * k);
}

template <int FMT, int SB>
cudaError_t launch_layer_t(const LayerParams& p, int grid, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = layer_smem_bytes(p);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, layer_kernel<FMT, SB>, p);
}

template <int FMT, int SB>
cudaError_t prepare_t(size_t smem, int* blocks)
{
    cudaError_t e = cudaFuncSetAttribute(layer_kernel<FMT, SB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, layer_kernel<FMT, SB>, kThreads, smem);
}

}  // namespace

size_t layer_smem_bytes(const LayerParams& p)
{
    return (size_t)p.nslots * p.slot_bytes + 2 * (size_t)p.mmax * p.I * sizeof(float) + kRedBytes +
           kXfragBytes;
}

cudaError_t prepare_layer_kernel(int fmt, int group, size_t smem, int* blocks_per_sm)
{
    if (fmt != FMT_INT4)
        return cudaErrorInvalidValue;
    if (scale_entry_bytes(fmt, group) == 8)
        return prepare_t<FMT_INT4, 8>(smem, blocks_per_sm);
    return prepare_t<FMT_INT4, 4>(smem, blocks_per_sm);
}

cudaError_t launch_layer(const LayerParams& p, int fmt, int grid, cudaStream_t stream)
{
    if (fmt != FMT_INT4)
        return cudaErrorInvalidValue;
    if (scale_entry_bytes(fmt, p.group) == 8)
        return launch_layer_t<FMT_INT4, 8>(p, grid, stream);
    return launch_layer_t<FMT_INT4, 4>(p, grid, stream);
}

cudaError_t launch_repack(int fmt, int group, const uint8_t* codes, const uint8_t* scales, int E,
                          int N, int K, uint8_t* out, long long expert_bytes, int slab_bytes,
                          uint32_t* special, int proj, cudaStream_t stream)
{
    const long long work = (long long)E * (N / kSlabRows) * (K / 64) * (128 + 8);
    const int blocks = (int)((work + 255) / 256 < 65536 ? (work + 255) / 256 : 65536);
    if (fmt != FMT_INT4)
        return cudaErrorInvalidValue;
    if (scale_entry_bytes(fmt, group) == 8)
        repack_kernel<FMT_INT4, 8><<<blocks, 256, 0, stream>>>(codes, scales, E, N, K, group, out,
                                                               expert_bytes, slab_bytes, special, proj);
    else
        repack_kernel<FMT_INT4, 4><<<blocks, 256, 0, stream>>>(codes, scales, E, N, K, group, out,
                                                               expert_bytes, slab_bytes, special, proj);
    return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, int group, const uint8_t* slabs, int N, int K, int slab_bytes,
                           float* out, cudaStream_t stream)
{
    const long long total = (long long)N * K;
    const int blocks = (int)((total + 255) / 256 < 8192 ? (total + 255) / 256 : 8192);
    if (fmt != FMT_INT4)
        return cudaErrorInvalidValue;
    if (scale_entry_bytes(fmt, group) == 8)
        dequant_kernel<FMT_INT4, 8><<<blocks, 256, 0, stream>>>(slabs, N, K, slab_bytes, out);
    else
        dequant_kernel<FMT_INT4, 4><<<blocks, 256, 0, stream>>>(slabs, N, K, slab_bytes, out);
    return cudaGetLastError();
}

cudaError_t launch_route(const float* logits, int M, int E, int k, int* idx, float* w,
                         cudaStream_t stream)
{
    const int warps = 8;
    route_kernel<<<(M + warps - 1) / warps, warps * 32, 0, stream>>>(logits, M, E, k, idx, w);
    return cudaGetLastError();
}

}  // namespace moe
