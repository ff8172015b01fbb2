// moe_batched.cu -- the routed-expert block for batches of more than four
// tokens, as per-expert grouped GEMMs on the 5th-generation tensor cores.
//
// "Sovereign gpt-oss-20B (MXFP4) on Apple Silicon", section 5 (threats to
// validity) names grouped-expert GEMM batching as the lever left untried; this
// file builds it for the same layer the decode kernel computes (router top-k,
// softmax over the selected, gate_up, SwiGLU, down, weighted sum into the
// residual).  Both MMA operands are FP4: x and h are quantised to MXFP4 per
// 32 consecutive elements along K by the OCP MX v1.0 rule (shared exponent
// floor(log2 amax) - 2, E2M1 round-to-nearest-even with saturation at +-6,
// amax = 0 -> scale byte 0 and +0 codes), and tcgen05.mma kind::mxf4 applies
// the E8M0 scales of both sides per 32 along K with fp32 accumulation in
// tensor memory.
//
// Kernels, in stream order:
//   route_kernel (moe_decode.cu)  top-k + softmax per token
//   plan_kernel                   per-expert stable permutation, token tiles
//   quant_x_kernel                MX(x) into the token tiles
//   gemm_kernel<true>             gate and up tiles, + bias, SwiGLU -> h (fp32)
//   quant_h_kernel                MX(h) into the token tiles
//   gemm_kernel<false>            down tiles, + bias -> y (fp32, slot order)
//   combine_kernel                out = bf16(r + sum_s w_s y_s)
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {
namespace {

// ---------------------------------------------------------------- PTX helpers

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

// Bounded wait on one phase of an mbarrier; on give-up record a timeout and
// return false (the caller carries on: every loop of these kernels is bounded).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status)
{
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

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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

// Byte offset of (row r, k-step s, half kc) of an activation tile with npad
// rows, and of (row r, K-block kb) in the tile's scale chunks.
__device__ __forceinline__ long long act_code_off(int npad, int r, int kb)
{
    return (long long)(kb >> 1) * npad * 32 + (r >> 3) * 256 + (kb & 1) * 128 + (r & 7) * 16;
}
__device__ __forceinline__ int act_sf_off(int r, int kb)
{
    return (kb >> 2) * kSfChunk + (r & 31) * 16 + (r >> 5) * 4 + (kb & 3);
}

// ------------------------------------------------------------------- plan

// One CTA of 1024 threads.  Entries q = m*k + s (token m, choice s) are ranked
// within their expert in q order (a stable counting sort), experts get
// consecutive slot ranges in expert order, and each expert's slots are cut
// into token tiles of at most kTokTile.
__global__ void __launch_bounds__(1024) plan_kernel(BatchParams p)
{
    __shared__ int cnt[32][kMaxExperts];
    __shared__ int base[kMaxExperts];
    __shared__ int off[kMaxExperts];
    __shared__ int toff[kMaxExperts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Mk = p.M * p.k, E = p.E;
    for (int e = tid; e < kMaxExperts; e += 1024)
        base[e] = 0;
    const unsigned lt = (1u << lane) - 1u;
    for (int c = 0; c < Mk; c += 1024) {
        for (int i = tid; i < 32 * kMaxExperts; i += 1024)
            (&cnt[0][0])[i] = 0;
        __syncthreads();
        const int q = c + tid;
        const bool valid = q < Mk;
        int e = valid ? p.idx[q] : -1;
        if (valid && (e < 0 || e >= E)) {   // cannot happen after route_kernel; keep indices in range
            atomicExch(p.status, MOE_ERR_DEVICE_FAULT);
            e = 0;
        }
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rw = __popc(same & lt);
        if (valid && (__ffs(same) - 1) == lane)
            cnt[warp][e] = __popc(same);
        __syncthreads();
        if (tid < E) {
            int run = base[tid];
            for (int w = 0; w < 32; ++w) {
                const int t = cnt[w][tid];
                cnt[w][tid] = run;
                run += t;
            }
            base[tid] = run;
        }
        __syncthreads();
        if (valid)
            p.erow[q] = cnt[warp][e] + rw;   // rank within the expert, rewritten below
        __syncthreads();
    }
    if (tid == 0) {
        int so = 0, to = 0, nu = 0;
        long long bo = 0;
        for (int e = 0; e < E; ++e) {
            const int n = base[e];
            nu += n > 0;
            off[e] = so;
            toff[e] = to;
            for (int j = 0; j * kTokTile < n; ++j) {
                TokTile t;
                t.e = e;
                t.p0 = so + j * kTokTile;
                t.n = n - j * kTokTile < kTokTile ? n - j * kTokTile : kTokTile;
                t.npad = (t.n + 15) & ~15;
                t.boff = bo;
                bo += t.npad * 32;
                if (to < p.max_tiles)
                    p.tiles[to] = t;
                ++to;
            }
            so += n;
        }
        if (to > p.max_tiles) {
            atomicExch(p.status, MOE_ERR_DEVICE_FAULT);
            to = p.max_tiles;
        }
        *p.ntiles = to;
        if (p.nu_out)
            *p.nu_out = nu;
    }
    __syncthreads();
    for (int q = tid; q < Mk; q += 1024) {
        int e = p.idx[q];
        e = e < 0 || e >= E ? 0 : e;
        const int r = p.erow[q];
        p.slot[q] = off[e] + r;
        p.etile[q] = toff[e] + r / kTokTile;
        p.erow[q] = r % kTokTile;
    }
}

// ----------------------------------------------------------- quantisation

// One thread per (token m, K-block kb): MX(x[m][32kb..]) written to the tile
// row of each of the token's k choices.
__global__ void quant_x_kernel(BatchParams p)
{
    const int nkb = p.H / 32;
    const long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (g >= (long long)p.M * nkb)
        return;
    const int m = (int)(g / nkb), kb = (int)(g % nkb);
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)m * p.H + 32 * kb);
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 u = __ldg(src + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
            v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
    }
    uint32_t code[4];
    const uint32_t sb = mx_block(v, code);
    const int ntiles = *p.ntiles;
    const int C = ceil_div(p.H, 128);
    for (int s = 0; s < p.k; ++s) {
        const int q = m * p.k + s;
        const int t = p.etile[q], r = p.erow[q];
        if (t >= ntiles)
            continue;
        const TokTile tt = p.tiles[t];
        *reinterpret_cast<uint4*>(p.xq + tt.boff * (p.H / 64) + act_code_off(tt.npad, r, kb)) =
            make_uint4(code[0], code[1], code[2], code[3]);
        p.xsf[(size_t)t * C * kSfChunk + act_sf_off(r, kb)] = (uint8_t)sb;
    }
}

// One thread per (entry q, K-block kb of I): MX(h[slot][32kb..]).
__global__ void quant_h_kernel(BatchParams p)
{
    const int nkb = p.I / 32;
    const long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (g >= (long long)p.M * p.k * nkb)
        return;
    const int q = (int)(g / nkb), kb = (int)(g % nkb);
    const int t = p.etile[q], r = p.erow[q];
    if (t >= *p.ntiles)
        return;
    const float4* src = reinterpret_cast<const float4*>(p.h + (size_t)p.slot[q] * p.I + 32 * kb);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 f = src[i];
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
    }
    uint32_t code[4];
    const uint32_t sb = mx_block(v, code);
    const TokTile tt = p.tiles[t];
    *reinterpret_cast<uint4*>(p.hq + tt.boff * (p.I / 64) + act_code_off(tt.npad, r, kb)) =
        make_uint4(code[0], code[1], code[2], code[3]);
    p.hsf[(size_t)t * ceil_div(p.I, 128) * kSfChunk + act_sf_off(r, kb)] = (uint8_t)sb;
}

// Debug: natural-order MX quantisation of a flat vector, one thread per block.
__global__ void mx_quantize_kernel(const float* __restrict__ in, long long nblk, uint8_t* codes,
                                   uint8_t* scales)
{
    const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (b >= nblk)
        return;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = in[32 * b + i];
    uint32_t code[4];
    scales[b] = (uint8_t)mx_block(v, code);
    *reinterpret_cast<uint4*>(codes + 16 * b) = make_uint4(code[0], code[1], code[2], code[3]);
}

// Debug: the h codes of the last call back in entry order [M*k][I/2], [M*k][I/32].
__global__ void untile_h_kernel(BatchParams p, uint8_t* codes, uint8_t* scales)
{
    const int nkb = p.I / 32;
    const long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (g >= (long long)p.M * p.k * nkb)
        return;
    const int q = (int)(g / nkb), kb = (int)(g % nkb);
    const int t = p.etile[q], r = p.erow[q];
    if (t >= *p.ntiles)
        return;
    const TokTile tt = p.tiles[t];
    *reinterpret_cast<uint4*>(codes + (size_t)q * (p.I / 2) + 16 * kb) =
        *reinterpret_cast<const uint4*>(p.hq + tt.boff * (p.I / 64) + act_code_off(tt.npad, r, kb));
    scales[(size_t)q * nkb + kb] = p.hsf[(size_t)t * ceil_div(p.I, 128) * kSfChunk + act_sf_off(r, kb)];
}

// ------------------------------------------------------------ grouped GEMM

struct GemmParams {
    const uint8_t* w;       // tile-layout weights; expert e at + e * w_expert
    long long w_expert;
    long long proj2;        // offset of the second (up) projection, DUAL only
    int rows, K;            // output rows of one projection, reduction length
    const uint8_t* bq;      // activation codes (tile order)
    const uint8_t* bsf;     // activation scale chunks
    const TokTile* tiles;
    const int* ntiles;
    const uint16_t* bias;   // [E][bias_stride] bf16 or nullptr; DUAL: up bias at + rows
    int bias_stride;
    float* out;             // [slots][rows]
    int* status;
};

constexpr int kStageSteps = 4;                          // k-steps (64 of K) per pipeline stage
constexpr int kAStage = kStageSteps * kRowTile * 32;    // 16 KB of weight codes
constexpr int kBStage = kStageSteps * kTokTile * 32;    // activation codes
constexpr int kSfCol = 448;                             // first tensor-memory column of the scale sets

template <bool DUAL>
struct GemmCfg {
    static constexpr int kSfBytes = (DUAL ? 3 : 2) * 2 * kSfChunk;
    static constexpr int kStage = (DUAL ? 2 : 1) * kAStage + kBStage + kSfBytes;
    static constexpr int kStages = DUAL ? 4 : 6;
    static constexpr int kSmem = kStages * kStage;
    static constexpr int kAccCols = (DUAL ? 2 : 1) * kTokTile;   // per accumulator buffer
    static constexpr int kSfSet = (DUAL ? 3 : 2) * 8;             // tensor-memory columns per scale set
};

// Persistent: one CTA per SM walks items w = blockIdx.x + i * gridDim.x, item
// w = (token tile w / T, row tile w % T).  Warp 0 feeds a ring of shared-memory
// stages with bulk copies; warp 1 owns tensor memory and issues the MMAs from
// one thread; warps 2..5 (one per lane quarter) drain the accumulators, which
// are double-buffered so the next item's MMAs overlap this item's epilogue.
template <bool DUAL>
__global__ void __launch_bounds__(192, 1) gemm_kernel(GemmParams p)
{
    using C = GemmCfg<DUAL>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[C::kStages], empty[C::kStages], accf[2], acce[2];
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;"
                     ::"r"(su32(&tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    const int T = ceil_div(p.rows, kRowTile);
    const int KS = p.K / 64, NSTG = ceil_div(KS, kStageSteps), CH = ceil_div(p.K, 128);
    const int items = *p.ntiles * T;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t ctr = 0;
            for (int w = blockIdx.x; w < items; w += gridDim.x) {
                const int tt = w / T, t = w % T;
                const TokTile tile = p.tiles[tt];
                const int R = p.rows - t * kRowTile < kRowTile ? p.rows - t * kRowTile : kRowTile;
                const uint8_t* a0 = p.w + tile.e * p.w_expert + (long long)t * kRowTile * (p.K / 2);
                const uint8_t* s0 = p.w + tile.e * p.w_expert + (long long)p.rows * (p.K / 2) +
                                    (long long)t * CH * kSfChunk;
                const uint8_t* b0 = p.bq + tile.boff * KS;
                const uint8_t* sb0 = p.bsf + (long long)tt * CH * kSfChunk;
                for (int j = 0; j < NSTG; ++j, ++ctr) {
                    const int slot = ctr % C::kStages;
                    const uint32_t use = ctr / C::kStages;
                    if (use > 0)
                        mbar_wait(&empty[slot], (use - 1) & 1, p.status);
                    const int steps = KS - j * kStageSteps < kStageSteps ? KS - j * kStageSteps : kStageSteps;
                    const int chunks = (steps + 1) >> 1;
                    const uint32_t abytes = steps * R * 32, bbytes = steps * tile.npad * 32;
                    const uint32_t sfbytes = chunks * kSfChunk;
                    uint8_t* st = smem + slot * C::kStage;
                    uint8_t* sA0 = st;
                    uint8_t* sA1 = st + kAStage;
                    uint8_t* sB = st + (DUAL ? 2 : 1) * kAStage;
                    uint8_t* sSF = sB + kBStage;
                    mbar_expect_tx(&full[slot], (DUAL ? 2 : 1) * (abytes + sfbytes) + bbytes + sfbytes);
                    const long long aoff = (long long)j * kStageSteps * R * 32;
                    const long long soff = (long long)j * 2 * kSfChunk;
                    bulk_copy(sA0, a0 + aoff, abytes, &full[slot]);
                    bulk_copy(sSF, s0 + soff, sfbytes, &full[slot]);
                    if (DUAL) {
                        bulk_copy(sA1, a0 + p.proj2 + aoff, abytes, &full[slot]);
                        bulk_copy(sSF + 2 * kSfChunk, s0 + p.proj2 + soff, sfbytes, &full[slot]);
                    }
                    bulk_copy(sB, b0 + (long long)j * kStageSteps * tile.npad * 32, bbytes, &full[slot]);
                    bulk_copy(sSF + (DUAL ? 4 : 2) * kSfChunk, sb0 + soff, sfbytes, &full[slot]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t ctr = 0, it = 0;
            for (int w = blockIdx.x; w < items; w += gridDim.x, ++it) {
                const int tt = w / T, t = w % T;
                const TokTile tile = p.tiles[tt];
                const int R = p.rows - t * kRowTile < kRowTile ? p.rows - t * kRowTile : kRowTile;
                const uint32_t buf = it & 1;
                if (it >= 2)
                    mbar_wait(&acce[buf], ((it >> 1) - 1) & 1, p.status);
                tc_fence_after();
                const uint32_t d0 = tmem + buf * C::kAccCols;
                const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(tile.npad >> 3) << 17) |
                                       (1u << 23) | ((uint32_t)(kRowTile >> 4) << 24);
                for (int j = 0; j < NSTG; ++j, ++ctr) {
                    const int slot = ctr % C::kStages;
                    mbar_wait(&full[slot], (ctr / C::kStages) & 1, p.status);
                    tc_fence_after();
                    const int steps = KS - j * kStageSteps < kStageSteps ? KS - j * kStageSteps : kStageSteps;
                    const int chunks = (steps + 1) >> 1;
                    const uint32_t st = su32(smem + slot * C::kStage);
                    const uint32_t sA0 = st, sA1 = st + kAStage;
                    const uint32_t sB = st + (DUAL ? 2 : 1) * kAStage;
                    const uint32_t sSF = sB + kBStage;
                    const uint32_t sf = tmem + kSfCol + (ctr & 1) * C::kSfSet;
                    const uint32_t sfa0 = sf, sfa1 = sf + 8, sfb = sf + (DUAL ? 16 : 8);
                    for (int c = 0; c < chunks; ++c) {
                        tc_cp_sf(sfa0 + 4 * c, sSF + c * kSfChunk);
                        if (DUAL)
                            tc_cp_sf(sfa1 + 4 * c, sSF + (2 + c) * kSfChunk);
                        tc_cp_sf(sfb + 4 * c, sSF + ((DUAL ? 4 : 2) + c) * kSfChunk);
                    }
                    for (int i = 0; i < steps; ++i) {
                        const uint32_t id = (uint32_t)(2 * (i & 1));
                        const uint32_t desc = idesc | (id << 4) | (id << 29);
                        const uint64_t bd = smem_desc(sB + i * tile.npad * 32, 128, 256);
                        const uint32_t acc = (j | i) != 0;
                        tc_mma_mxf4(d0, smem_desc(sA0 + i * R * 32, 128, 256), bd, desc,
                                    sfa0 + 4 * (i >> 1), sfb + 4 * (i >> 1), acc);
                        if (DUAL)
                            tc_mma_mxf4(d0 + kTokTile, smem_desc(sA1 + i * R * 32, 128, 256), bd, desc,
                                        sfa1 + 4 * (i >> 1), sfb + 4 * (i >> 1), acc);
                    }
                    tc_commit(&empty[slot]);
                }
                tc_commit(&accf[buf]);
            }
        }
    } else {
        const int q = warp & 3;   // lane quarter this warp may access
        uint32_t it = 0;
        for (int w = blockIdx.x; w < items; w += gridDim.x, ++it) {
            const int tt = w / T, t = w % T;
            const TokTile tile = p.tiles[tt];
            const uint32_t buf = it & 1;
            mbar_wait(&accf[buf], (it >> 1) & 1, p.status);
            tc_fence_after();
            const int row = t * kRowTile + 32 * q + lane;
            const bool valid = row < p.rows;
            float b0 = 0.0f, b1 = 0.0f;
            if (p.bias && valid) {
                const uint16_t* bb = p.bias + (size_t)tile.e * p.bias_stride;
                b0 = bf16f(bb[row]);
                if (DUAL)
                    b1 = bf16f(bb[p.rows + row]);
            }
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * C::kAccCols;
            float* out = p.out + (size_t)tile.p0 * p.rows + row;
            for (int c0 = 0; c0 < tile.n; c0 += 16) {
                float g[16], u[16];
                tc_ld16(taddr + c0, g);
                if (DUAL)
                    tc_ld16(taddr + kTokTile + c0, u);
                tc_wait_ld();
                if (valid) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        if (c0 + jj < tile.n) {
                            float v;
                            if (DUAL) {
                                const float gg = g[jj] + b0;
                                v = gg / (1.0f + expf(-gg)) * (u[jj] + b1);
                            } else {
                                v = g[jj] + b0;
                            }
                            out[(size_t)(c0 + jj) * p.rows] = v;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acce[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
    }
}

// out[m][j] = bf16(r[m][j] + sum_s w[m][s] * y[slot(m, s)][j]), s in order;
// one thread per 8 consecutive j.
__global__ void combine_kernel(BatchParams p)
{
    const int n8 = p.H / 8;
    const long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (g >= (long long)p.M * n8)
        return;
    const int m = (int)(g / n8), j0 = 8 * (int)(g % n8);
    uint4* rp = reinterpret_cast<uint4*>(p.resid + (size_t)m * p.H + j0);
    const uint4 rv = *rp;
    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
    float acc[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __uint_as_float(rw[i] << 16);
        acc[2 * i + 1] = __uint_as_float(rw[i] & 0xffff0000u);
    }
    float sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int s = 0; s < p.k; ++s) {
        const int q = m * p.k + s;
        const float wq = p.wt[q];
        const float4* yp = reinterpret_cast<const float4*>(p.y + (size_t)p.slot[q] * p.H + j0);
        const float4 a = yp[0], b = yp[1];
        sum[0] += wq * a.x; sum[1] += wq * a.y; sum[2] += wq * a.z; sum[3] += wq * a.w;
        sum[4] += wq * b.x; sum[5] += wq * b.y; sum[6] += wq * b.z; sum[7] += wq * b.w;
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = (uint32_t)f2bf16_rne(acc[2 * i] + sum[2 * i]) |
               ((uint32_t)f2bf16_rne(acc[2 * i + 1] + sum[2 * i + 1]) << 16);
    *rp = make_uint4(o[0], o[1], o[2], o[3]);
}

// --------------------------------------------------------------- repacking

// Caller layout -> tile layout, one projection (rows row0 .. row0+N-1 of each
// expert's [src_rows][K/2] code matrix).  Work item g < E*N*K/32 moves one
// 16-byte run of codes; g beyond that writes one scale byte.
__global__ void repack_tiles_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                    int E, int src_rows, int row0, int N, int K, uint8_t* out,
                                    long long expert_bytes)
{
    const int c16 = K / 32;                       // 16-byte runs per row
    const int T = ceil_div(N, kRowTile), CH = ceil_div(K, 128);
    const long long ncode = (long long)E * N * c16;
    const long long nsf = (long long)E * T * CH * kSfChunk;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < ncode + nsf;
         g += (long long)gridDim.x * blockDim.x) {
        if (g < ncode) {
            const int e = (int)(g / ((long long)N * c16));
            const long long rem = g % ((long long)N * c16);
            const int n = (int)(rem / c16), c = (int)(rem % c16);
            const int t = n / kRowTile, r = n % kRowTile;
            const int R = N - t * kRowTile < kRowTile ? N - t * kRowTile : kRowTile;
            const uint4 v = *reinterpret_cast<const uint4*>(
                codes + ((size_t)e * src_rows + row0 + n) * (K / 2) + 16 * c);
            const long long dst = (long long)e * expert_bytes + (long long)t * kRowTile * (K / 2) +
                                  (long long)(c >> 1) * R * 32 + (r >> 3) * 256 + (c & 1) * 128 + (r & 7) * 16;
            *reinterpret_cast<uint4*>(out + dst) = v;
        } else {
            const long long h = g - ncode;
            const int e = (int)(h / ((long long)T * CH * kSfChunk));
            const long long rem = h % ((long long)T * CH * kSfChunk);
            const int t = (int)(rem / (CH * kSfChunk)), ch = (int)(rem / kSfChunk % CH);
            const int b = (int)(rem % kSfChunk);
            const int i = b >> 4, j = (b >> 2) & 3, kb = b & 3;
            const int n = t * kRowTile + 32 * j + i, blk = 4 * ch + kb;
            uint8_t v = 0;
            if (n < N && blk < K / 32)
                v = scales[((size_t)e * src_rows + row0 + n) * (K / 32) + blk];
            out[(long long)e * expert_bytes + (long long)N * (K / 2) + rem] = v;
        }
    }
}

template <bool DUAL>
cudaError_t launch_gemm(const GemmParams& g, int grid, cudaStream_t s)
{
    gemm_kernel<DUAL><<<grid, 192, GemmCfg<DUAL>::kSmem, s>>>(g);
    return cudaGetLastError();
}

unsigned blocks_for(long long n, int threads)
{
    return (unsigned)((n + threads - 1) / threads);
}

}  // namespace

cudaError_t prepare_batched_kernels()
{
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GemmCfg<true>::kSmem);
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg<false>::kSmem);
}

cudaError_t launch_batched(const BatchParams& p, int grid, cudaStream_t s, int* launches)
{
    cudaError_t e;
    *launches = 0;
    if ((e = launch_route(p.logits, p.M, p.E, p.k, p.idx, p.wt, s)) != cudaSuccess)
        return e;
    plan_kernel<<<1, 1024, 0, s>>>(p);
    quant_x_kernel<<<blocks_for((long long)p.M * (p.H / 32), 256), 256, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    GemmParams g{};
    g.w = p.gu;
    g.w_expert = p.gu_expert;
    g.proj2 = tile_proj_bytes(p.I, p.H);
    g.rows = p.I;
    g.K = p.H;
    g.bq = p.xq;
    g.bsf = p.xsf;
    g.tiles = p.tiles;
    g.ntiles = p.ntiles;
    g.bias = p.gu_bias;
    g.bias_stride = 2 * p.I;
    g.out = p.h;
    g.status = p.status;
    if ((e = launch_gemm<true>(g, grid, s)) != cudaSuccess)
        return e;
    quant_h_kernel<<<blocks_for((long long)p.M * p.k * (p.I / 32), 256), 256, 0, s>>>(p);
    g.w = p.dn;
    g.w_expert = p.dn_expert;
    g.proj2 = 0;
    g.rows = p.H;
    g.K = p.I;
    g.bq = p.hq;
    g.bsf = p.hsf;
    g.bias = p.dn_bias;
    g.bias_stride = p.H;
    g.out = p.y;
    if ((e = launch_gemm<false>(g, grid, s)) != cudaSuccess)
        return e;
    combine_kernel<<<blocks_for((long long)p.M * (p.H / 8), 256), 256, 0, s>>>(p);
    *launches = 7;
    return cudaGetLastError();
}

cudaError_t launch_repack_tiles(const uint8_t* codes, const uint8_t* scales, int E, int src_rows,
                                int row0, int N, int K, uint8_t* out, long long expert_bytes,
                                cudaStream_t stream)
{
    const long long work = (long long)E * N * (K / 32) +
                           (long long)E * ceil_div(N, kRowTile) * ceil_div(K, 128) * kSfChunk;
    const long long blocks = (work + 255) / 256 < 65536 ? (work + 255) / 256 : 65536;
    repack_tiles_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, E, src_rows, row0, N, K, out,
                                                              expert_bytes);
    return cudaGetLastError();
}

cudaError_t launch_mx_quantize(const float* in, long long n, uint8_t* codes, uint8_t* scales,
                               cudaStream_t stream)
{
    const long long nblk = n / 32;
    if (nblk > 0)
        mx_quantize_kernel<<<blocks_for(nblk, 128), 128, 0, stream>>>(in, nblk, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_untile_h(const BatchParams& p, uint8_t* codes, uint8_t* scales, cudaStream_t stream)
{
    const long long n = (long long)p.M * p.k * (p.I / 32);
    untile_h_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(p, codes, scales);
    return cudaGetLastError();
}

}  // namespace moe
