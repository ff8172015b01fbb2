// moe_batched_f16.cu -- the batched layer's bf16 numerics (M > 4, selected with
// moe_set_batched_numerics): tcgen05.mma kind::f16 on the MXFP4 weights
// dequantised to bf16 in shared memory, against activations that are not
// quantised -- x as given (bf16), h as a pair of bf16 values hi + lo (hi =
// bf16(h), lo = bf16(h - hi), ~16 significant bits).  The kind::mxf4 path
// quantises x and h to MXFP4 because that instruction wants FP4 on both sides;
// this variant trades that activation rounding for a dequantisation of every
// weight on the CUDA cores.
//
// It reuses the batched path's routing, plan (per-expert token tiles of up to
// 96 tokens) and combine; only the activation packing and the two GEMMs
// differ.  Each GEMM is persistent (one CTA per SM walking (token tile, row
// tile) items, as gemm_kernel does), with four roles:
//   warp 0      streams the weights, one k-step a stage (the 128-row tile's
//               E2M1 codes, 4 KB, and its 128-column scale chunk), 10 stages
//               in flight;
//   warp 14     streams the activation blocks (a ring of their own: they are
//               mostly L2 hits, re-read by every row tile);
//   warps 6..13 dequantise the codes into a bf16 copy of the k-step (half a
//               row per thread, each element e2m1 * 2^(s - 127) exactly, then
//               RNE to bf16 -- exact: a 2-bit significand, and bf16 has
//               fp32's exponent range);
//   warp 1      issues 4 MMAs of K = 16 per k-step (M = 128, N = the token
//               tile, or twice it for the down GEMM's hi and lo rows) into
//               double-buffered tensor-memory accumulators;
//   warps 2..5  drain the accumulators (one lane quarter each): gate_up
//               applies SwiGLU and writes h as hi/lo bf16 rows of the down
//               GEMM's activation tile; down adds the hi and lo columns and
//               writes fp32 rows y for the combine.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kTileA16 = kRowTile * 32;           // one k-step of a 128-row tile of E2M1 codes: 4 KB
constexpr int kF16RawA = kTileA16 + kSfChunk;     // ... and its 128-column scale chunk
constexpr int kASlots = 10;                       // weight ring: k-steps in flight (the HBM stream)
constexpr int kBSlots = 5;                        // activation ring (mostly L2 hits)
constexpr int kF16B = 2 * kTokTile * 128;         // an activation block: up to 2 x 96 rows x 64 bf16
constexpr int kA16 = kRowTile * 64 * 2;           // a dequantised k-step: 128 rows x 64 bf16
constexpr int kF16Smem = kASlots * kF16RawA + kBSlots * kF16B + 2 * kA16;
constexpr int kConvWarps = 8;                     // converter warps: two threads a tile row
constexpr int kThreadsF16 = 480;                  // 2 producers, MMA, 4 epilogue and 8 converter warps
constexpr int kAccF16 = 2 * kTokTile;             // accumulator columns per buffer (down: hi + lo)
static_assert(2 * kAccF16 <= 512, "tensor memory: two accumulator buffers");
static_assert(kF16RawA % 128 == 0 && kF16B % 128 == 0, "shared-memory alignment of the operands");
static_assert(kF16Smem <= 227 * 1024, "shared memory");

struct F16Params {
    const uint8_t* w;       // tile-layout weights; expert e at + e * w_expert
    long long w_expert;
    int kmajor;             // k-step-major tile order (down)
    int rows, K;            // DUAL: rows of h (the projection has 2 * rows); else output rows
    const uint8_t* act;     // bf16 activation tiles (x, or h as hi/lo rows)
    const TokTile* tiles;
    const int* ntiles;
    const uint16_t* bias;   // [E][bias_stride] bf16 or nullptr; DUAL: gate | up
    int bias_stride;
    float* out;             // single: y [slots][rows] fp32
    uint8_t* h16;           // DUAL: h as hi/lo rows of the down GEMM's activation tiles
    int* status;
    float sw_alpha, sw_limit, sw_beta;   // DUAL: the SwiGLU form
};

// Byte offset of element (row r, column k) of a bf16 activation tile whose
// k-step blocks hold nb rows: block k / 64 of nb x 64 bf16 in the canonical
// no-swizzle K-major order (8 rows x 8 elements per core matrix, core
// matrices 128 bytes apart along K and 1024 bytes apart along the rows).
__device__ __forceinline__ long long act16_off(int nb, int r, int k)
{
    return (long long)(k >> 6) * nb * 128 + (r >> 3) * 1024 + ((k & 63) >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// Tile base of the bf16 activations: token tile rows start at boff / 32 in the
// padded row space; x rows hold K bf16, h rows twice I (hi and lo rows).
__device__ __forceinline__ long long act16_base(const TokTile& t, int K, int per_row)
{
    return (t.boff / 32) * (long long)K * 2 * per_row;
}

// One (token, 8-element group): x[m][8 g .. 8 g + 7] to the tile row of each of
// the token's k choices.
__global__ void pack_x16_kernel(const uint16_t* __restrict__ x, int M, int H, int k, const int* __restrict__ etile,
                                const int* __restrict__ erow, const TokTile* __restrict__ tiles,
                                const int* __restrict__ ntiles, uint8_t* __restrict__ x16)
{
    const long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const int ng = H / 8;
    if (g >= (long long)M * ng)
        return;
    const int m = (int)(g / ng), c = 8 * (int)(g % ng);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)m * H + c));
    const int nt = *ntiles;
    for (int s = 0; s < k; ++s) {
        const int q = m * k + s;
        const int t = etile[q], r = erow[q];
        if (t >= nt)
            continue;
        const TokTile tt = tiles[t];
        *reinterpret_cast<uint4*>(x16 + act16_base(tt, H, 1) + act16_off(tt.npad, r, c)) = v;
    }
}

// Half a row of a k-step (half hf: elements 32 hf .. 32 hf + 31 = bytes 16 hf
// .. 16 hf + 15, element 2b in the low nibble of byte b) times its block scale
// -> 32 bf16 in the canonical layout (e2m1 * 2^(s-127) in fp32 is exact, and
// so is its RNE conversion to bf16).
__device__ __forceinline__ void dequant_half_row(const uint8_t* raw, const uint8_t* chunk, int r, int hf, int kpair,
                                                 uint8_t* a16)
{
    const uint4 cw = *reinterpret_cast<const uint4*>(raw + (r >> 3) * 256 + hf * 128 + (r & 7) * 16);
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
    const uint32_t sb = chunk[(r & 31) * 16 + (r >> 5) * 4 + 2 * kpair + hf];
    const float s = __uint_as_float(sb == 0u ? 0x00400000u : (sb == 255u ? 0x7fc00000u : sb << 23));
#pragma unroll
    for (int kg = 0; kg < 4; ++kg) {   // elements 8 kg .. 8 kg + 7 of the half: word kg
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = e2m1x2_to_f32(w[kg] >> (8 * j));
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[j]) : "f"(f.y * s), "f"(f.x * s));
        }
        *reinterpret_cast<uint4*>(a16 + (r >> 3) * 1024 + (4 * hf + kg) * 128 + (r & 7) * 16) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Issue, one lane each, the stages [c, c + n) of a ring of `slots` stages
// whose slots are free: lane 0 waits for stage c's slot, the others only test
// theirs (a slot is tested against its previous use, at most one phase
// behind), and the ready prefix goes out.  Returns the number issued.
template <typename Issue>
__device__ __forceinline__ int issue_batch(uint64_t* empty, int slots, uint32_t c, int n, int lane, int* status,
                                           Issue&& issue)
{
    if (lane == 0 && c >= (uint32_t)slots)
        mbar_wait(&empty[c % slots], ((c / slots) - 1) & 1, status);
    __syncwarp();
    const uint32_t k = c + (uint32_t)lane;
    bool ready = lane < slots && lane < n;
    if (ready && lane > 0 && k >= (uint32_t)slots)
        ready = mbar_test_wait(&empty[k % slots], ((k / slots) - 1) & 1);
    const int nb = __ffs(~__ballot_sync(0xffffffffu, ready)) - 1;
    if (lane < nb)
        issue(k, k % slots);
    __syncwarp();
    return nb;
}

template <bool DUAL>
__global__ void __launch_bounds__(kThreadsF16, 1) gemm16_kernel(F16Params p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ float xbuf[DUAL ? 2 * 2 * 2 * 32 * 8 : 1];
    __shared__ __align__(8) uint64_t fullA[kASlots], emptyA[kASlots], fullB[kBSlots], emptyB[kBSlots];
    __shared__ __align__(8) uint64_t a16f[2], a16e[2], accf[2], acce[2];
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ringA = smem;
    uint8_t* ringB = smem + kASlots * kF16RawA;
    uint8_t* a16 = ringB + kBSlots * kF16B;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kASlots; ++i) {
            mbar_init(&fullA[i], 1);
            mbar_init(&emptyA[i], kConvWarps);
        }
        for (int i = 0; i < kBSlots; ++i) {
            mbar_init(&fullB[i], 1);
            mbar_init(&emptyB[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a16f[i], kConvWarps);
            mbar_init(&a16e[i], 1);
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    const int T = DUAL ? p.rows / 64 : ceil_div(p.rows, kRowTile);
    const int KS = p.K / 64;
    const int prow = DUAL ? 2 * p.rows : p.rows;
    const int items = *p.ntiles * T;
    // this CTA's items are w = blockIdx.x + i gridDim.x; its k-steps run c = i KS + s
    const int nitems = blockIdx.x < items ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t total = (uint32_t)nitems * (uint32_t)KS;

    if (warp == 0) {
        // ================================================================ weight producer
        for (uint32_t c = 0; c < total;) {
            c += issue_batch(emptyA, kASlots, c, (int)(total - c), lane, p.status, [&](uint32_t k, uint32_t slot) {
                const int w = blockIdx.x + (int)(k / KS) * gridDim.x, s = (int)(k % KS);
                const int t = w % T;
                const TokTile tile = p.tiles[w / T];
                const int R = prow - t * kRowTile < kRowTile ? prow - t * kRowTile : kRowTile;
                const uint8_t* we = p.w + tile.e * p.w_expert;
                uint8_t* st = ringA + slot * kF16RawA;
                mbar_expect_tx(&fullA[slot], (uint32_t)R * 32 + kSfChunk);
                bulk_copy(st, we + tile_block_off(prow, p.K, t, s, p.kmajor), (uint32_t)R * 32, &fullA[slot]);
                bulk_copy(st + kTileA16, we + tile_sf_off(prow, p.K, t, s >> 1, p.kmajor), kSfChunk, &fullA[slot]);
            });
        }
    } else if (warp == 6 + kConvWarps) {
        // ================================================================ activation producer
        for (uint32_t c = 0; c < total;) {
            c += issue_batch(emptyB, kBSlots, c, (int)(total - c), lane, p.status, [&](uint32_t k, uint32_t slot) {
                const int w = blockIdx.x + (int)(k / KS) * gridDim.x, s = (int)(k % KS);
                const TokTile tile = p.tiles[w / T];
                const int nb = DUAL ? tile.npad : 2 * tile.npad;
                const uint8_t* ab = p.act + act16_base(tile, p.K, DUAL ? 1 : 2);
                mbar_expect_tx(&fullB[slot], (uint32_t)nb * 128);
                bulk_copy(ringB + slot * kF16B, ab + (long long)s * nb * 128, (uint32_t)nb * 128, &fullB[slot]);
            });
        }
    } else if (warp >= 6) {
        // ================================================================ converters (warps 6..13)
        const int r = (threadIdx.x - 192) & 127, hf = (threadIdx.x - 192) >> 7;   // row, half of it
        for (uint32_t c = 0; c < total; ++c) {
            const int w = blockIdx.x + (int)(c / KS) * gridDim.x, s = (int)(c % KS);
            const int t = w % T;
            const int R = prow - t * kRowTile < kRowTile ? prow - t * kRowTile : kRowTile;
            const uint32_t slot = c % kASlots, a = c & 1;
            mbar_wait(&fullA[slot], (c / kASlots) & 1, p.status);
            if (c >= 2)
                mbar_wait(&a16e[a], ((c >> 1) - 1) & 1, p.status);
            const uint8_t* st = ringA + slot * kF16RawA;
            if (r < R)   // rows past a partial tile feed MMA rows nobody reads
                dequant_half_row(st, st + kTileA16, r, hf, s & 1, a16 + a * kA16);
            fence_proxy_async_smem();   // generic writes -> the MMA's reads
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&a16f[a]);
                mbar_arrive(&emptyA[slot]);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            uint32_t c = 0, it = 0;
            for (int w = blockIdx.x; w < items; w += gridDim.x, ++it) {
                const TokTile tile = p.tiles[w / T];
                const int nb = DUAL ? tile.npad : 2 * tile.npad;
                const uint32_t buf = it & 1;
                if (it >= 2)
                    mbar_wait(&acce[buf], ((it >> 1) - 1) & 1, p.status);
                tc_fence_after();
                const uint32_t d = tmem + buf * kAccF16;
                // kind::f16: f32 accumulate (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1),
                // both K-major, N / 8 at bit 17, M / 16 at bit 24
                const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(nb >> 3) << 17) |
                                       ((uint32_t)(kRowTile >> 4) << 24);
                for (int s = 0; s < KS; ++s, ++c) {
                    const uint32_t slot = c % kBSlots, a = c & 1;
                    mbar_wait(&fullB[slot], (c / kBSlots) & 1, p.status);
                    mbar_wait(&a16f[a], (c >> 1) & 1, p.status);
                    tc_fence_after();
                    const uint32_t sa = su32(a16 + a * kA16), sb = su32(ringB + slot * kF16B);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t da = smem_desc(sa + j * 256, 128, 1024), db = smem_desc(sb + j * 256, 128, 1024);
                        const uint32_t acc = (s | j) != 0;
                        asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %4, 0;\n\t"
                                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}"
                                     ::"r"(d), "l"(da), "l"(db), "r"(idesc), "r"(acc) : "memory");
                    }
                    tc_commit(&emptyB[slot]);
                    tc_commit(&a16e[a]);
                }
                tc_commit(&accf[buf]);
            }
        }
    } else if (warp < 6) {
        // ================================================================ epilogue (warps 2..5)
        const int q = warp & 3;   // lane quarter this warp may access
        uint32_t it = 0, xb = 0;
        for (int w = blockIdx.x; w < items; w += gridDim.x, ++it) {
            const int tt = w / T, t = w % T;
            const TokTile tile = p.tiles[tt];
            const uint32_t buf = it & 1;
            mbar_wait(&accf[buf], (it >> 1) & 1, p.status);
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * kAccF16;
            if (DUAL) {
                // gate rows (q = 0, 1) and up rows (q = 2, 3) of the same 64 rows of h
                const int hrow = 64 * t + 32 * (q & 1) + lane;
                const bool gate = q < 2;
                float bg = 0.0f, bu = 0.0f;
                if (p.bias) {
                    const uint16_t* bb = p.bias + (size_t)tile.e * p.bias_stride;
                    bg = bf16f(bb[hrow]);
                    bu = bf16f(bb[p.rows + hrow]);
                }
                uint8_t* hb = p.h16 + act16_base(tile, p.rows, 2);
                for (int c0 = 0; c0 < tile.n; c0 += 16, xb ^= 1u) {
                    float v16[16];
                    tc_ld16(taddr + c0, v16);
                    tc_wait_ld();
                    // gate warps keep tokens 0..7 of the chunk, up warps 8..15
                    float* mine = xbuf + (((xb * 2 + (gate ? 0 : 1)) * 2 + (q & 1)) * 32 + lane) * 8;
                    const float* theirs = xbuf + (((xb * 2 + (gate ? 1 : 0)) * 2 + (q & 1)) * 32 + lane) * 8;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        mine[jj] = v16[gate ? 8 + jj : jj];
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    const int cb = c0 + (gate ? 0 : 8);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int n = cb + jj;
                        if (n >= tile.n)
                            break;
                        const float gg = (gate ? v16[jj] : theirs[jj]) + bg;
                        const float uu = (gate ? theirs[jj] : v16[8 + jj]) + bu;
                        const float v = swiglu(gg, uu, p.sw_alpha, p.sw_limit, p.sw_beta);
                        const uint16_t hi = f2bf16_rne(v);
                        const uint16_t lo = f2bf16_rne(v - bf16f(hi));
                        *reinterpret_cast<uint16_t*>(hb + act16_off(2 * tile.npad, n, hrow)) = hi;
                        *reinterpret_cast<uint16_t*>(hb + act16_off(2 * tile.npad, tile.npad + n, hrow)) = lo;
                    }
                }
            } else {
                const int row = t * kRowTile + 32 * q + lane;
                // rows come in multiples of 64, so a warp's 32 rows are all valid or all not
                const bool valid = t * kRowTile + 32 * q < p.rows;
                const float b0 = p.bias && valid ? bf16f(p.bias[(size_t)tile.e * p.bias_stride + row]) : 0.0f;
                for (int c0 = 0; c0 < tile.n; c0 += 16) {
                    float hi16[16], lo16[16];
                    tc_ld16(taddr + c0, hi16);
                    tc_ld16(taddr + tile.npad + c0, lo16);
                    tc_wait_ld();
                    if (!valid)
                        continue;
                    const int nn = tile.n - c0 < 16 ? tile.n - c0 : 16;
                    float* out = p.out + (size_t)(tile.p0 + c0) * p.rows + row;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        if (jj < nn)
                            out[(size_t)jj * p.rows] = (hi16[jj] + lo16[jj]) + b0;
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

}  // namespace

cudaError_t prepare_batched_f16_kernels()
{
    cudaError_t e = cudaFuncSetAttribute(gemm16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF16Smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF16Smem);
    return e;
}

size_t batched_f16_act_bytes(long long rows, int H, int I)
{
    return (size_t)rows * H * 2 + (size_t)rows * I * 4;
}

cudaError_t launch_batched_f16_gemms(const BatchParams& b, int grid, cudaStream_t s)
{
    const long long n8 = (long long)b.M * (b.H / 8);
    pack_x16_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(b.x, b.M, b.H, b.k, b.etile, b.erow, b.tiles, b.ntiles,
                                                                b.x16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    F16Params g{};
    g.w = b.gu;
    g.w_expert = b.gu_expert;
    g.kmajor = 0;
    g.rows = b.I;
    g.K = b.H;
    g.act = b.x16;
    g.tiles = b.tiles;
    g.ntiles = b.ntiles;
    g.bias = b.gu_bias;
    g.bias_stride = 2 * b.I;
    g.h16 = b.h16;
    g.status = b.status;
    g.sw_alpha = b.sw_alpha;
    g.sw_limit = b.sw_limit;
    g.sw_beta = b.sw_beta;
    gemm16_kernel<true><<<grid, kThreadsF16, kF16Smem, s>>>(g);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    g.w = b.dn;
    g.w_expert = b.dn_expert;
    g.kmajor = 1;
    g.rows = b.H;
    g.K = b.I;
    g.act = b.h16;
    g.bias = b.dn_bias;
    g.bias_stride = b.H;
    g.out = b.y;
    g.h16 = nullptr;
    gemm16_kernel<false><<<grid, kThreadsF16, kF16Smem, s>>>(g);
    return cudaGetLastError();
}

}  // namespace moe
