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
//   route_kernel                  top-k + softmax per token
//   plan_kernel                   per-expert stable permutation, token tiles
//   quant_x_kernel                MX(x) into the token tiles
//   gemm_kernel<true>             gate and up tiles, + bias, SwiGLU, MX(h) into
//                                 the token tiles (h never leaves the chip in fp32)
//   gemm_kernel<false>            down tiles, + bias -> y (fp32, slot order)
//   combine_kernel                out = bf16(r + sum_s w_s y_s)
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "moe_internal.h"
#include "route.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

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

// Exclusive scan of three per-expert values over threads 0..255 of the block
// (all 1024 threads call it; threads >= 256 pass zeros); returns the three
// totals through `tot`.
__device__ void scan3_256(int (&v)[3], int (&tot)[3], int (*wsum)[3])
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int x[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            const int y = __shfl_up_sync(0xffffffffu, x[c], off);
            if (lane >= off)
                x[c] += y;
        }
    if (lane == 31 && warp < 8)
        for (int c = 0; c < 3; ++c)
            wsum[warp][c] = x[c];
    __syncthreads();
    if (tid < 32) {
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            int y = tid < 8 ? wsum[tid][c] : 0;
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                const int z = __shfl_up_sync(0xffffffffu, y, off);
                if (tid >= off)
                    y += z;
            }
            if (tid < 8)
                wsum[tid][c] = y;   // inclusive over warps
        }
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const int before = warp > 0 && warp < 8 ? wsum[warp - 1][c] : 0;
        tot[c] = wsum[7][c];
        v[c] = before + x[c] - v[c];
    }
}

// One CTA of 1024 threads.  Entries q = m*k + s (token m, choice s) are ranked
// within their expert in q order (a stable counting sort), experts get
// consecutive slot ranges in expert order, and each expert's slots are cut
// into token tiles of at most kTokTile (the expert's tiles before its last
// are full, so a tile's activation offset follows from the expert's padded
// row offset).
__global__ void __launch_bounds__(1024) plan_kernel(BatchParams p)
{
    __shared__ int cnt[32][kMaxExperts];
    __shared__ int base[kMaxExperts];
    __shared__ int off[kMaxExperts];
    __shared__ int toff[kMaxExperts];
    __shared__ int wsum[8][3];
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
    // per expert: slots n, tiles ceil(n / kTokTile), padded activation rows
    const int n = tid < E ? base[tid] : 0;
    const int full = n / kTokTile, rem = n % kTokTile;
    int v[3] = {n, full + (rem > 0), full * kTokTile + ((rem + 15) & ~15)};
    int tot[3];
    scan3_256(v, tot, wsum);
    if (tid < E) {
        off[tid] = v[0];
        toff[tid] = v[1];
        for (int j = 0; j * kTokTile < n; ++j) {
            const int to = v[1] + j;
            if (to >= p.max_tiles)
                break;
            TokTile t;
            t.e = tid;
            t.p0 = v[0] + j * kTokTile;
            t.n = n - j * kTokTile < kTokTile ? n - j * kTokTile : kTokTile;
            t.npad = (t.n + 15) & ~15;
            t.boff = (long long)(v[2] + j * kTokTile) * 32;
            p.tiles[to] = t;
        }
    }
    const unsigned busy = __ballot_sync(0xffffffffu, n > 0);
    if (lane == 0 && warp < 8)
        wsum[warp][0] = __popc(busy);   // scan3_256 is done with wsum
    __syncthreads();
    if (tid == 0) {
        int nu = 0;
        for (int w = 0; w < 8; ++w)
            nu += wsum[w][0];
        int to = tot[1];
        if (to > p.max_tiles) {
            atomicExch(p.status, MOE_ERR_DEVICE_FAULT);
            to = p.max_tiles;
        }
        *p.ntiles = to;
        if (p.nu_out)
            *p.nu_out = nu;
    }
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
    const uint8_t* w;       // tile-layout weights; expert e at + e * w_expert (DUAL: interleaved gate_up)
    long long w_expert;
    int kmajor;             // the weights are in the k-step-major tile order (the down projection)
    int rows, K;            // output rows (DUAL: rows of h, the projection has 2 * rows), reduction length
    const uint8_t* bq;      // activation codes (tile order)
    const uint8_t* bsf;     // activation scale chunks
    const TokTile* tiles;
    const int* ntiles;
    const uint16_t* bias;   // [E][bias_stride] bf16 or nullptr; DUAL: gate | up
    int bias_stride;
    float* out;             // single: y [slots][rows] fp32
    uint8_t* hq;            // DUAL: MX(h) codes in the down GEMM's activation tile order
    uint8_t* hsf;           // DUAL: MX(h) scale chunks
    int* status;
    float sw_alpha, sw_limit, sw_beta;   // DUAL: the SwiGLU form
};

constexpr int kStageSteps = 8;           // k-steps (64 of K) per pipeline stage
constexpr int kSfCol = 4 * kTokTile;     // first tensor-memory column of the scale sets
constexpr int kRingBytes = 200 * 1024;   // shared-memory stage ring (byte-granular FIFO)
constexpr int kRingSlack = 4096;         // read slack past the ring end (see Stage)
constexpr int kStageSlots = 16;          // stages in flight at most (mbarrier pairs)

struct GemmCfg {
    static constexpr int kSmem = kRingBytes + kRingSlack;
    static constexpr int kAccCols = kTokTile;                 // per accumulator buffer
    static constexpr int kSfSet = 2 * 4 * (kStageSteps / 2);  // tensor-memory columns per scale set
    static_assert(kSfCol + 2 * kSfSet <= 512, "tensor memory: accumulators + two scale sets");
};

// One pipeline stage: `steps` k-steps of R weight rows and npad activation
// rows, with their scale chunks, packed as [A][B][SFA][SFB] and sized to what
// it holds, so that a small token tile leaves the ring to weight bytes.  For
// a partial row tile (R = 64) the MMA still reads 128 rows of the last k-step
// block, up to 2 KB past A; that lands inside the stage or in the ring's slack.
struct Stage {
    uint32_t abytes, bbytes, sfbytes, size;
    __device__ Stage(int steps, int R, int npad)
    {
        const int chunks = (steps + 1) >> 1;
        abytes = steps * R * 32;
        bbytes = steps * npad * 32;
        sfbytes = chunks * kSfChunk;
        size = (abytes + sfbytes + bbytes + sfbytes + 127) & ~127u;
    }
    __device__ uint32_t b() const { return abytes; }
    __device__ uint32_t sfa0() const { return b() + bbytes; }
    __device__ uint32_t sfb() const { return sfa0() + sfbytes; }
};

// FIFO placement of stages in the ring; a stage never straddles the end.
// The producer and the MMA thread run the same sequence of placements.
struct Ring {
    unsigned long long head = 0;   // virtual bytes handed out so far
    uint32_t phys = 0;             // head modulo kRingBytes
    __device__ uint32_t place(uint32_t size, unsigned long long* end)
    {
        if (phys + size > (uint32_t)kRingBytes) {
            head += kRingBytes - phys;
            phys = 0;
        }
        const uint32_t off = phys;
        phys += size;
        head += size;
        *end = head;
        return off;
    }
};

// Persistent: one CTA per SM walks items w = blockIdx.x + i * gridDim.x, item
// w = (token tile w / T, row tile w % T).  Warp 0 feeds the stage ring with
// bulk copies; warp 1 owns tensor memory and issues the MMAs from one thread;
// warps 2..5 (one per lane quarter) drain the accumulators, which are
// double-buffered so the next item's MMAs overlap this item's epilogue.
// DUAL (gate_up): a 128-row tile is 64 gate rows over 64 up rows of the same
// rows of h, so SwiGLU pairs lane quarters 0, 1 with 2, 3 through shared memory.
template <bool DUAL>
__global__ void __launch_bounds__(192, 1) gemm_kernel(GemmParams p)
{
    using C = GemmCfg;
    extern __shared__ __align__(1024) uint8_t smem[];
    // DUAL: per 16-token chunk (double-buffered), gate warps hand over tokens 8..15
    // of their gate sums and up warps tokens 0..7 of their up sums: [buf][gate | up][warp][lane][8]
    __shared__ float xbuf[DUAL ? 2 * 2 * 2 * 32 * 8 : 1];
    __shared__ __align__(8) uint64_t full[kStageSlots], empty[kStageSlots], accf[2], acce[2];
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStageSlots; ++i) {
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

    const int T = DUAL ? p.rows / 64 : ceil_div(p.rows, kRowTile);
    const int KS = p.K / 64, NSTG = ceil_div(KS, kStageSteps), CH = ceil_div(p.K, 128);
    const int prow = DUAL ? 2 * p.rows : p.rows;   // rows of the stored projection
    const int items = *p.ntiles * T;

    if (warp == 0) {
        // The whole warp runs the producer loop; a stage's copies are issued by
        // separate lanes in one instruction (one lane issuing them one after
        // another costs ~0.15 us each, which would bound the stage rate).
        Ring ring;
        unsigned long long ends[kStageSlots];
        unsigned long long rel_end = 0;   // ring bytes released by the consumer
        uint32_t c = 0, rel = 0;          // stages issued / released
        TokTile tile = blockIdx.x < items ? p.tiles[blockIdx.x / T] : TokTile{};
        for (int w = blockIdx.x; w < items; w += gridDim.x) {
            const int tt = w / T, t = w % T;
            // the next item's descriptor is loaded now and used one item later,
            // so its latency never stalls the copy stream
            const int wn = w + gridDim.x;
            const TokTile next = wn < items ? p.tiles[wn / T] : tile;
            const int R = prow - t * kRowTile < kRowTile ? prow - t * kRowTile : kRowTile;
            const uint8_t* we = p.w + tile.e * p.w_expert;
            const uint8_t* b0 = p.bq + tile.boff * KS;
            const uint8_t* sb0 = p.bsf + (long long)tt * CH * kSfChunk;
            for (int j = 0; j < NSTG; ++j, ++c) {
                const int steps = KS - j * kStageSteps < kStageSteps ? KS - j * kStageSteps : kStageSteps;
                const Stage sg(steps, R, tile.npad);
                unsigned long long end;
                const uint32_t off = ring.place(sg.size, &end);
                // wait until the bytes and the slot are free (stages retire in order)
                while (rel < c && (end - rel_end > (unsigned long long)kRingBytes || rel + kStageSlots <= c)) {
                    const uint32_t sl = rel % kStageSlots;
                    mbar_wait(&empty[sl], (rel / kStageSlots) & 1, p.status);
                    rel_end = ends[sl];
                    ++rel;
                }
                const uint32_t slot = c % kStageSlots;
                ends[slot] = end;
                if (lane == 0)
                    mbar_expect_tx(&full[slot], sg.abytes + sg.sfbytes + sg.bbytes + sg.sfbytes);
                __syncwarp();
                const long long soff = (long long)j * (kStageSteps / 2) * kSfChunk;
                const int s0 = j * kStageSteps, ch0 = j * (kStageSteps / 2);
                uint8_t* st = smem + off;
                uint8_t* dst = nullptr;
                const uint8_t* src = nullptr;
                uint32_t n = 0;
                if (!p.kmajor) {
                    // row-tile-major: the stage's k-steps and scale chunks are two runs
                    switch (lane) {
                    case 0: dst = st; src = we + tile_block_off(prow, p.K, t, s0, 0); n = sg.abytes; break;
                    case 1: dst = st + sg.sfa0(); src = we + tile_sf_off(prow, p.K, t, ch0, 0); n = sg.sfbytes; break;
                    default: break;
                    }
                } else if (lane < steps) {
                    // k-step-major: one block per k-step (lanes 0..7), one chunk per
                    // column chunk (lanes 8..11)
                    dst = st + lane * R * 32;
                    src = we + tile_block_off(prow, p.K, t, s0 + lane, 1);
                    n = (uint32_t)R * 32;
                } else if (lane >= kStageSteps && lane < kStageSteps + (steps + 1) / 2) {
                    const int c = lane - kStageSteps;
                    dst = st + sg.sfa0() + c * kSfChunk;
                    src = we + tile_sf_off(prow, p.K, t, ch0 + c, 1);
                    n = kSfChunk;
                }
                if (lane == 16) {
                    dst = st + sg.b(); src = b0 + (long long)j * kStageSteps * tile.npad * 32; n = sg.bbytes;
                } else if (lane == 17) {
                    dst = st + sg.sfb(); src = sb0 + soff; n = sg.sfbytes;
                }
                if (n)
                    bulk_copy(dst, src, n, &full[slot]);
            }
            tile = next;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            Ring ring;
            uint32_t c = 0, it = 0;
            for (int w = blockIdx.x; w < items; w += gridDim.x, ++it) {
                const int t = w % T;
                const TokTile tile = p.tiles[w / T];
                const int R = prow - t * kRowTile < kRowTile ? prow - t * kRowTile : kRowTile;
                const uint32_t buf = it & 1;
                if (it >= 2)
                    mbar_wait(&acce[buf], ((it >> 1) - 1) & 1, p.status);
                tc_fence_after();
                const uint32_t d0 = tmem + buf * C::kAccCols;
                const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(tile.npad >> 3) << 17) |
                                       (1u << 23) | ((uint32_t)(kRowTile >> 4) << 24);
                for (int j = 0; j < NSTG; ++j, ++c) {
                    const int steps = KS - j * kStageSteps < kStageSteps ? KS - j * kStageSteps : kStageSteps;
                    const Stage sg(steps, R, tile.npad);
                    unsigned long long end;
                    const uint32_t st = su32(smem) + ring.place(sg.size, &end);
                    const uint32_t slot = c % kStageSlots;
                    mbar_wait(&full[slot], (c / kStageSlots) & 1, p.status);
                    tc_fence_after();
                    const int chunks = (steps + 1) >> 1;
                    const uint32_t sA0 = st, sB = st + sg.b();
                    const uint32_t sf = tmem + kSfCol + (c & 1) * C::kSfSet;
                    constexpr uint32_t kOp = 4 * (kStageSteps / 2);   // columns per operand's scales
                    const uint32_t sfa0 = sf, sfb = sf + kOp;
                    for (int ch = 0; ch < chunks; ++ch) {
                        tc_cp_sf(sfa0 + 4 * ch, st + sg.sfa0() + ch * kSfChunk);
                        tc_cp_sf(sfb + 4 * ch, st + sg.sfb() + ch * kSfChunk);
                    }
                    for (int i = 0; i < steps; ++i) {
                        const uint32_t id = (uint32_t)(2 * (i & 1));
                        const uint32_t desc = idesc | (id << 4) | (id << 29);
                        const uint64_t bd = smem_desc(sB + i * tile.npad * 32, 128, 256);
                        const uint32_t acc = (j | i) != 0;
                        tc_mma_mxf4(d0, smem_desc(sA0 + i * R * 32, 128, 256), bd, desc,
                                    sfa0 + 4 * (i >> 1), sfb + 4 * (i >> 1), acc);
                    }
                    tc_commit(&empty[slot]);
                }
                tc_commit(&accf[buf]);
            }
        }
    } else {
        const int q = warp & 3;   // lane quarter this warp may access
        uint32_t it = 0, xb = 0;
        for (int w = blockIdx.x; w < items; w += gridDim.x, ++it) {
            const int tt = w / T, t = w % T;
            const TokTile tile = p.tiles[tt];
            const uint32_t buf = it & 1;
            mbar_wait(&accf[buf], (it >> 1) & 1, p.status);
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * C::kAccCols;
            if (DUAL) {
                // h row of this lane: gate rows (q = 0, 1) and up rows (q = 2, 3) of the
                // same 64 rows of h; each warp's 32 rows are one 32-element block of h
                const int hrow = 64 * t + 32 * (q & 1) + lane, kb = hrow >> 5;
                const bool gate = q < 2;
                float bg = 0.0f, bu = 0.0f;
                if (p.bias) {
                    const uint16_t* bb = p.bias + (size_t)tile.e * p.bias_stride;
                    bg = bf16f(bb[hrow]);
                    bu = bf16f(bb[p.rows + hrow]);
                }
                uint8_t* hq = p.hq + tile.boff * (p.rows / 64) + 4 * (lane >> 3);
                uint8_t* hs = p.hsf + (size_t)tt * ceil_div(p.rows, 128) * kSfChunk;
                for (int c0 = 0; c0 < tile.n; c0 += 16, xb ^= 1u) {
                    float v16[16];
                    tc_ld16(taddr + c0, v16);
                    tc_wait_ld();
                    // hand over the other half of the chunk: gate warps keep tokens 0..7,
                    // up warps 8..15
                    float* mine = xbuf + (((xb * 2 + (gate ? 0 : 1)) * 2 + (q & 1)) * 32 + lane) * 8;
                    const float* theirs = xbuf + (((xb * 2 + (gate ? 1 : 0)) * 2 + (q & 1)) * 32 + lane) * 8;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        mine[jj] = v16[gate ? 8 + jj : jj];
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    const int cb = c0 + (gate ? 0 : 8);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        if (cb + jj >= tile.n)
                            break;
                        const float gg = (gate ? v16[jj] : theirs[jj]) + bg;
                        const float uu = (gate ? theirs[jj] : v16[8 + jj]) + bu;
                        const float v = swiglu(gg, uu, p.sw_alpha, p.sw_limit, p.sw_beta);
                        const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
                        const int ef = (int)(amax >> 23);
                        const uint32_t sbyte = ef > 2 ? (uint32_t)(ef - 2) : 0u;
                        const float inv = __uint_as_float((254u - sbyte) << 23);
                        const uint32_t code = amax == 0u ? 0u : (e2m1x2(v * inv, 0.0f) & 0xfu);
                        uint32_t word = code << (4 * (lane & 7));
                        word |= __shfl_xor_sync(0xffffffffu, word, 1);
                        word |= __shfl_xor_sync(0xffffffffu, word, 2);
                        word |= __shfl_xor_sync(0xffffffffu, word, 4);
                        const int n = cb + jj;
                        if ((lane & 7) == 0)
                            *reinterpret_cast<uint32_t*>(hq + act_code_off(tile.npad, n, kb)) = word;
                        if (lane == 0)
                            hs[act_sf_off(n, kb)] = (uint8_t)sbyte;
                    }
                }
            } else {
                const int row = t * kRowTile + 32 * q + lane;
                // rows come in multiples of 64, so a warp's 32 rows are all valid or all not
                const bool valid = t * kRowTile + 32 * q < p.rows;
                const float b0 = p.bias && valid ? bf16f(p.bias[(size_t)tile.e * p.bias_stride + row]) : 0.0f;
                for (int c0 = 0; c0 < tile.n; c0 += 16) {
                    float g[16];
                    tc_ld16(taddr + c0, g);
                    tc_wait_ld();
                    if (!valid)
                        continue;
                    const int nn = tile.n - c0 < 16 ? tile.n - c0 : 16;
                    float* out = p.out + (size_t)(tile.p0 + c0) * p.rows + row;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        if (jj < nn)
                            out[(size_t)jj * p.rows] = g[jj] + b0;
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
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = acc[i] + sum[i];
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = (uint32_t)f2bf16_rne(v[2 * i]) | ((uint32_t)f2bf16_rne(v[2 * i + 1]) << 16);
    *rp = make_uint4(o[0], o[1], o[2], o[3]);
    if (p.out_f32) {
        float4* f = reinterpret_cast<float4*>(p.out_f32 + (size_t)m * p.H + j0);
        f[0] = make_float4(v[0], v[1], v[2], v[3]);
        f[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

// --------------------------------------------------------------- repacking

// Caller row of tile-layout row n: n itself, or the interleaved gate_up order.
__device__ __forceinline__ int src_row(int n, int ilv)
{
    if (!ilv)
        return n;
    const int t = n / kRowTile, r = n % kRowTile;
    return r < 64 ? 64 * t + r : ilv + 64 * t + r - 64;
}

// Caller layout -> tile layout, one projection (N rows of each expert's
// [src_rows][K/2] code matrix).  Work item g < E*N*K/32 moves one 16-byte run
// of codes; g beyond that writes one scale byte.
__global__ void repack_tiles_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                    int E, int src_rows, int N, int K, int ilv, int kmajor, uint8_t* out,
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
            const uint4 v = *reinterpret_cast<const uint4*>(
                codes + ((size_t)e * src_rows + src_row(n, ilv)) * (K / 2) + 16 * c);
            const long long dst = (long long)e * expert_bytes + tile_block_off(N, K, t, c >> 1, kmajor) +
                                  (r >> 3) * 256 + (c & 1) * 128 + (r & 7) * 16;
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
                v = scales[((size_t)e * src_rows + src_row(n, ilv)) * (K / 32) + blk];
            out[(long long)e * expert_bytes + tile_sf_off(N, K, t, ch, kmajor) + b] = v;
        }
    }
}

// Element (n, k) of one projection in caller row order, read back from the
// tile layout the tensor-core kernels stream: its E2M1 code times its E8M0
// scale 2^(s - 127), in fp32 (exact; byte 0 gives 2^-127, byte 255 NaN, and a
// product past the fp32 range overflows to infinity).
__global__ void dequant_tiles_kernel(const uint8_t* __restrict__ tiles, int N, int K, int ilv, int kmajor,
                                     float* __restrict__ out)
{
    const long long total = (long long)N * K;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int nc = (int)(idx / K), k = (int)(idx % K);
        int n = nc;   // row in the tile order
        if (ilv) {
            const int up = nc >= ilv, rr = up ? nc - ilv : nc;
            n = (rr / 64) * kRowTile + (up ? 64 : 0) + rr % 64;
        }
        const int t = n / kRowTile, r = n % kRowTile;
        const int s = k / 64, b = (k % 64) / 2;
        const uint8_t byte = tiles[tile_block_off(N, K, t, s, kmajor) + (r >> 3) * 256 + (b >> 4) * 128 +
                                   (r & 7) * 16 + (b & 15)];
        const uint32_t code = (k & 1) ? byte >> 4 : byte & 0xfu;
        const int blk = k / 32;
        const uint32_t sbyte = tiles[tile_sf_off(N, K, t, blk / 4, kmajor) + (r & 31) * 16 + (r >> 5) * 4 + (blk & 3)];
        const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
        const float v = (code & 8u) ? -mag[code & 7u] : mag[code & 7u];
        const float sc = __uint_as_float(sbyte == 0u ? 0x00400000u : (sbyte == 255u ? 0x7fc00000u : sbyte << 23));
        out[idx] = v * sc;
    }
}

// Top-k and the softmax over it, one warp per token (the debug router and the
// first step of the batched layer).
__global__ void route_kernel(const float* __restrict__ logits, int M, int E, int k, int* idx, float* w)
{
    const int tok = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (tok < M)
        rt::warp_topk(logits + (size_t)tok * E, E, k, idx + (size_t)tok * k, w + (size_t)tok * k);
}

template <bool DUAL>
cudaError_t launch_gemm(const GemmParams& g, int grid, cudaStream_t s)
{
    gemm_kernel<DUAL><<<grid, 192, GemmCfg::kSmem, s>>>(g);
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
                                         GemmCfg::kSmem);
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg::kSmem);
}

cudaError_t launch_batched(const BatchParams& p, int grid, cudaStream_t s, int* launches)
{
    cudaError_t e;
    *launches = 0;
    if ((e = launch_route(p.logits, p.M, p.E, p.k, p.idx, p.wt, s)) != cudaSuccess)
        return e;
    plan_kernel<<<1, 1024, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    if (p.f16) {
        if ((e = launch_batched_f16_gemms(p, grid, s)) != cudaSuccess)
            return e;
        combine_kernel<<<blocks_for((long long)p.M * (p.H / 8), 256), 256, 0, s>>>(p);
        *launches = 6;
        return cudaGetLastError();
    }
    quant_x_kernel<<<blocks_for((long long)p.M * (p.H / 32), 256), 256, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    GemmParams g{};
    g.w = p.gu;
    g.w_expert = p.gu_expert;
    g.kmajor = 0;
    g.rows = p.I;
    g.K = p.H;
    g.bq = p.xq;
    g.bsf = p.xsf;
    g.tiles = p.tiles;
    g.ntiles = p.ntiles;
    g.bias = p.gu_bias;
    g.bias_stride = 2 * p.I;
    g.hq = p.hq;
    g.hsf = p.hsf;
    g.status = p.status;
    g.sw_alpha = p.sw_alpha;
    g.sw_limit = p.sw_limit;
    g.sw_beta = p.sw_beta;
    if ((e = launch_gemm<true>(g, grid, s)) != cudaSuccess)
        return e;
    g.w = p.dn;
    g.w_expert = p.dn_expert;
    g.kmajor = 1;
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
    *launches = 6;
    return cudaGetLastError();
}

cudaError_t launch_repack_tiles(const uint8_t* codes, const uint8_t* scales, int E, int src_rows,
                                int N, int K, int interleave, int kmajor, uint8_t* out, long long expert_bytes,
                                cudaStream_t stream)
{
    const long long work = (long long)E * N * (K / 32) +
                           (long long)E * ceil_div(N, kRowTile) * ceil_div(K, 128) * kSfChunk;
    const long long blocks = (work + 255) / 256 < 65536 ? (work + 255) / 256 : 65536;
    repack_tiles_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, E, src_rows, N, K, interleave, kmajor,
                                                              out, expert_bytes);
    return cudaGetLastError();
}

// Router GEMV of the batched path: logits [M][E] fp32 from x [M][H] bf16 and
// the router rows w [E][H] bf16 followed by the bias [E], one warp per logit.
// The arithmetic is the decode kernel's: a lane-strided fp32 FMA chain over
// 8-element vectors (lo half before hi), a fixed butterfly, then the bias, so
// both paths give the same bits for the same x.
__global__ void router_gemv_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, int M, int H,
                                   int E, float* __restrict__ out)
{
    const long long g = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (g >= (long long)M * E)
        return;
    const int m = (int)(g / E), e = (int)(g % E);
    const uint4* xv = reinterpret_cast<const uint4*>(x + (size_t)m * H);
    const uint4* wv = reinterpret_cast<const uint4*>(w + (size_t)e * H);
    float acc = 0.f;
    for (int i = lane; i < H / 8; i += 32) {
        const uint4 x4 = __ldg(xv + i), w4 = __ldg(wv + i);
        const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w}, ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            acc = fmaf(__uint_as_float(xw[c] << 16), __uint_as_float(ww[c] << 16), acc);
            acc = fmaf(__uint_as_float(xw[c] & 0xffff0000u), __uint_as_float(ww[c] & 0xffff0000u), acc);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0)
        out[(size_t)m * E + e] = acc + bf16f(w[(size_t)E * H + e]);
}

cudaError_t launch_router_gemv(const uint16_t* x, const uint16_t* w, int M, int H, int E, float* out,
                               cudaStream_t stream)
{
    const long long warps = (long long)M * E;
    router_gemv_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(x, w, M, H, E, out);
    return cudaGetLastError();
}

cudaError_t launch_route(const float* logits, int M, int E, int k, int* idx, float* w,
                         cudaStream_t stream)
{
    const int warps = 8;
    route_kernel<<<(M + warps - 1) / warps, warps * 32, 0, stream>>>(logits, M, E, k, idx, w);
    return cudaGetLastError();
}

cudaError_t launch_dequant_tiles(const uint8_t* tiles, int N, int K, int interleave, int kmajor, float* out,
                                 cudaStream_t stream)
{
    const long long total = (long long)N * K;
    dequant_tiles_kernel<<<blocks_for(total, 256), 256, 0, stream>>>(tiles, N, K, interleave, kmajor, out);
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
