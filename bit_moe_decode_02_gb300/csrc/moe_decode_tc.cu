// moe_decode_tc.cu -- the MXFP4 decode layer (M <= 4 tokens) on the
// 5th-generation tensor cores: one persistent launch per layer, one CTA per SM.
//
// The layer is the one of "Sovereign gpt-oss-20B (MXFP4) on Apple Silicon",
// section 3 (top-k routing, per selected expert an MXFP4 gate_up GEMV,
// SwiGLU, an MXFP4 down GEMV, the routing-weighted sum into the residual).
// The weights stay 4-bit all the way into the MMA: tcgen05.mma kind::mxf4
// reads E2M1 codes and E8M0 scales from shared / tensor memory, so no
// instruction per weight runs on the CUDA cores.  That instruction wants FP4
// on the activation side too; an activation vector v (x, or h) is therefore
// fed as a sum of T MXFP4 vectors, v ~ v_1 + ... + v_T, each term one column
// of the MMA's N (token m, term j at column 8m + j; N = 16 for M <= 2, else
// 32).  Term j of a 32-element block has the shared exponent X0 - 2j (X0 the
// OCP MX v1.0 exponent of the block) and the nearest-even E2M1 codes of the
// residual the earlier terms left; every term cuts the residual by at least
// 4, so T = 8 terms leave a relative error near 1e-5 of the block maximum.
// The MMA applies every term's scales, and the epilogue adds a token's columns.
//
// Work unit: 64 rows of h of one selected expert.  Its gate/up weights are one
// 128-row tile (64 gate rows over 64 up rows, the interleaved tile layout), so
// one CTA computes SwiGLU for those rows with nothing exchanged; it folds in
// each token's routing weight, h'_m = w_m h_m, and runs the down projection's
// 64 matching K columns for every output row.  CTA b takes the units
// [b U / G, (b+1) U / G), so no activation ever crosses CTAs: each CTA adds
// its down products into its own fp32 copy of the output, and after one grid
// barrier CTA b sums the CTAs' copies for its slice of the output rows in CTA
// order (results do not depend on timing) and writes
// out = bf16(r + sum + sum_s w_s b_s).
//
// The x terms are built inside the layer: the (token, 32-element block) items
// are dealt over the CTAs, written to global memory and counted; gate/up
// stages carry them once the count is complete.  Weight copies never wait.
//
// The launch signals its dependents at entry, so the next layer's CTAs take
// over each SM as soon as this layer's CTA there exits and set up before they
// wait for this grid to complete.
//
// Warp roles (192 threads): warp 0 streams weights into a byte ring of shared
// memory (each stage's copies issued from separate lanes in one instruction);
// warp 1 owns tensor memory and issues the MMAs; warps 2..5 (one per lane
// quarter) build the x terms and drain the accumulators.  Warps 0 and 1 route.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "moe_internal.h"
#include "route.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kTerms = 8;            // MX terms per activation vector
constexpr int kGuSteps = 8;          // k-steps (64 of K) per gate/up stage
constexpr int kDnStageTiles = 5;     // 128-row down tiles per down stage
constexpr int kSlots = 16;           // stages in flight at most
// tensor memory columns
constexpr int kGuCol = 0;            // gate/up accumulators: 2 buffers x 32
constexpr int kDnCol = 64;           // down accumulators: 2 regions x 160
constexpr int kDnRegion = 160;
constexpr int kSfCol = 384;          // stage scale sets: 2 issuers x 2 sets x 32
constexpr int kSfSet = 32;
constexpr int kTmemCols = 512;
static_assert(kDnCol + 2 * kDnRegion <= kSfCol && kSfCol + 4 * kSfSet <= kTmemCols, "tensor memory");
static_assert(kDnRegion % (kDnStageTiles * 32) == 0, "a region holds whole down stages");
static_assert(kSfSet >= 8 * ((kGuSteps + 1) / 2), "a gate/up stage's A and B scale chunks fit a set");
static_assert(kSfSet >= 4 * (kDnStageTiles + 1), "a down stage's scale chunks fit a set");
constexpr int kThreadsTc = 224;      // producer, MMA issuer A, 4 epilogue warps, MMA issuer B
constexpr int kMmaWarpB = 6;
constexpr int kEpi = 128;            // epilogue threads (warps 2..5)
constexpr int kPend = 16;            // gate/up stages waiting for the x terms
constexpr int kTileA = kRowTile * 32;            // one k-step of a 128-row tile: 4 KB
constexpr int kHTerm = 1024 + kSfChunk;          // h' terms of a unit: one k-step atom + its scale chunk

// MMA N: the rows that hold terms, rounded up to 16; a k-step of terms is
// N rows x 32 bytes (8-row groups 256 bytes apart).
__device__ __forceinline__ int rows_for(int M) { return M * kTerms <= 16 ? 16 : 32; }

// Shared memory past the stage ring: two h'-term buffers, the up-sum exchange
// (2 warps x 32 lanes x float4) and the CTA's fp32 output copy [H][M].
__device__ __forceinline__ uint32_t tail_bytes(int H, int M)
{
    return 2 * kHTerm + 2 * 32 * 16 + (((uint32_t)H * M * 4 + 127) & ~127u);
}

// Items of a CTA with n units, in the order the producer, the MMA issuer and
// the epilogue walk them: gate/up of unit 0, then (gate/up of unit i+1, down
// of unit i) pairs, then the last down -- a unit's SwiGLU epilogue overlaps
// the next unit's gate/up MMAs.
__device__ __forceinline__ void item_at(int k, int n, bool& down, int& i)
{
    if (k == 0) {
        down = false;
        i = 0;
    } else if ((k & 1) && (k + 1) / 2 < n) {
        down = false;
        i = (k + 1) / 2;
    } else {
        down = true;
        i = (k & 1) ? (k - 1) / 2 : k / 2 - 1;
    }
}

// Gate/up stage: [A: steps x 4 KB][SFA: chunks x 512][B: steps x atom][SFB: chunks x 512].
struct GuStage {
    uint32_t abytes, sfbytes, bbytes, sfa, b, sfb, size;
    __device__ GuStage(int steps, int atom)
    {
        abytes = steps * kTileA;
        sfbytes = ((steps + 1) >> 1) * kSfChunk;
        bbytes = steps * atom;
        sfa = abytes;
        b = sfa + sfbytes;
        sfb = b + bbytes;
        size = (sfb + sfbytes + 127) & ~127u;
    }
};
// Down stage of n tiles: [A: n x 4 KB][SFA: n x 512].  A partial tile (64 rows)
// still has a 4 KB slot, so the MMA's 128-row read stays inside the stage.
__device__ __forceinline__ uint32_t dn_stage_size(int n) { return (uint32_t)n * (kTileA + kSfChunk); }

struct RingTc {
    unsigned long long head = 0;
    uint32_t phys = 0;
    __device__ uint32_t place(uint32_t size, uint32_t cap, unsigned long long* end)
    {
        if (phys + size > cap) {
            head += cap - phys;
            phys = 0;
        }
        const uint32_t off = phys;
        phys += size;
        head += size;
        *end = head;
        return off;
    }
};

__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, %0;" ::"r"(kEpi) : "memory"); }
__device__ __forceinline__ void route_barrier() { asm volatile("bar.sync 2, 96;" ::: "memory"); }

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
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Nearest-even E2M1 value of |x| (x already divided by the block scale, so
// |x| < 8), saturating at 6, and its 3-bit magnitude code.  Plain fp32
// arithmetic: rint(y) = (y + 2^23) - 2^23 with round-to-nearest-even adds,
// per grid segment (steps 0.5 below 2, 1 below 4, 2 from 4); the code comes
// from the rounded value's exponent and top mantissa bit (0.5 is the only
// subnormal).  Short latency, unlike the FP4 conversion instructions.
__device__ __forceinline__ float e2m1_rne(float ax, uint32_t& code)
{
    const float big = 8388608.0f;   // 2^23
    const float r05 = __fsub_rn(__fadd_rn(ax * 2.0f, big), big) * 0.5f;
    const float r1 = __fsub_rn(__fadd_rn(ax, big), big);
    const float r2 = fminf(__fsub_rn(__fadd_rn(ax * 0.5f, big), big) * 2.0f, 6.0f);
    const float qv = ax < 2.0f ? r05 : (ax < 4.0f ? r1 : r2);
    const uint32_t bits = __float_as_uint(qv);
    code = qv == 0.0f ? 0u : (qv == 0.5f ? 1u : (bits >> 22) - 252u);
    return qv;
}

// One warp, one 32-element block kb of M tokens m0 .. m0+M-1 (lane i holds
// element i of token m0+t's block in r[t]): kTerms MX terms of each, term j
// of token m to row m * kTerms + j of the k-step atoms at `q` (atom bytes per
// k-step), its E8M0 byte to the scale chunks at `sf`.  Term 0 takes the OCP
// shared exponent X0 = floor(log2 amax) - 2; term j uses X0 - 2j.  A term
// leaves an error of at most 2 * 2^Xj per element (half a step below 6, or
// the saturation from < 8 to 6), i.e. at most 8 * 2^X(j+1), so no later term
// exceeds the E2M1 range and every term cuts the error by at least 4: the
// block maximum is reduced once instead of per term.  The tokens' chains are
// interleaved; packing the codes into bytes and the stores come after.
template <int M>
__device__ __forceinline__ void warp_terms_rows(float (&r)[kMaxTokens], int m0, int kb, uint8_t* q, uint8_t* sf,
                                                int atom, int lane)
{
    uint32_t codes[kMaxTokens] = {0u, 0u, 0u, 0u};   // nibble j = term j's code of this lane's element
    uint32_t sblo[kMaxTokens] = {0u, 0u, 0u, 0u}, sbhi[kMaxTokens] = {0u, 0u, 0u, 0u};   // byte j%4 = scale
    int sb0[kMaxTokens] = {0, 0, 0, 0};
    bool zero[kMaxTokens] = {true, true, true, true};
#pragma unroll
    for (int m = 0; m < kMaxTokens; ++m) {
        if (m < M) {
            const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(r[m])));
            const int ef = (int)(amax >> 23);
            sb0[m] = ef > 2 ? ef - 2 : 0;
            zero[m] = amax == 0u;
        }
    }
#pragma unroll 1
    for (int j = 0; j < kTerms; ++j) {
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m) {
            if (m < M) {
                const uint32_t sb = sb0[m] - 2 * j > 0 ? (uint32_t)(sb0[m] - 2 * j) : 0u;
                const float inv = __uint_as_float((254u - sb) << 23);                          // 2^(127 - sb)
                const float scale = __uint_as_float(sb == 0u ? 0x00400000u : (sb << 23));   // 2^(sb - 127)
                uint32_t mag;
                const float qv = e2m1_rne(fminf(fabsf(r[m]) * inv, 8.0f), mag);
                const uint32_t code = zero[m] ? 0u : (mag | (r[m] < 0.0f ? 8u : 0u));
                codes[m] |= code << (4 * j);
                if (j < 4)
                    sblo[m] |= sb << (8 * j);
                else
                    sbhi[m] |= sb << (8 * (j - 4));
                if (!zero[m])
                    r[m] -= copysignf(qv, r[m]) * scale;
            }
        }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint32_t cm = codes[m], lo = sblo[m], hi = sbhi[m];
#pragma unroll
        for (int j = 0; j < kTerms; ++j) {
            uint32_t word = ((cm >> (4 * j)) & 0xfu) << (4 * (lane & 7));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            word |= __shfl_xor_sync(0xffffffffu, word, 4);
            const int row = (m0 + m) * kTerms + j;
            if ((lane & 7) == 0)
                *reinterpret_cast<uint32_t*>(q + (kb >> 1) * atom + (row >> 3) * 256 + (kb & 1) * 128 +
                                             (row & 7) * 16 + 4 * (lane >> 3)) = word;
            if (lane == 0)
                sf[(kb >> 2) * kSfChunk + row * 16 + (kb & 3)] = (uint8_t)((j < 4 ? lo : hi) >> (8 * (j & 3)));
        }
    }
}

// 1 / sqrt(mean(v^2) + 1e-6) of a bf16 row of n elements (n % 8 == 0), the
// same value on every lane of the warp.
__device__ __forceinline__ float row_inv_rms(const uint16_t* row, int n, int lane)
{
    float a = 0.f;
    for (int i = lane; i < n / 8; i += 32) {
        const uint4 w = __ldcg(reinterpret_cast<const uint4*>(row) + i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int z = 0; z < 4; ++z) {
            const float lo = __uint_as_float(ws[z] << 16), hi = __uint_as_float(ws[z] & 0xffff0000u);
            a = fmaf(lo, lo, a);
            a = fmaf(hi, hi, a);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        a += __shfl_xor_sync(0xffffffffu, a, off);
    return 1.0f / sqrtf(a / (float)n + 1e-6f);
}

struct TcSmem {
    uint64_t full[kSlots], empty[kSlots];
    uint64_t accf[2], acce[2];   // gate/up accumulator buffers: full / drained
    uint64_t dnf[2], dne[2];     // down accumulator regions: full (both issuers) / drained
    uint64_t hbar[2];            // h' terms of a unit written
    uint64_t routed, xready;     // routing done; every CTA's x terms published
    uint32_t tmem_base;
    int sel[kMaxTokens][kMaxTopK];
    float wt[kMaxTokens][kMaxTopK];
    int nu;
    int unit_expert[kMaxUnits];
    unsigned char unit_of[kMaxExperts];
    float wslot[kMaxUnits][kMaxTokens];   // routing weight of token m for expert slot s (0 if not chosen)
};

__global__ void __launch_bounds__(kThreadsTc, 1) decode_tc_kernel(const DecodeTcParams p)
{
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ __align__(8) TcSmem sh;
    // the next layer's CTAs may take each SM as soon as this CTA leaves it
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x, M = p.M;
    const int nrows = rows_for(M), atom = nrows * 32;
    const int KSH = p.H / 64, CHH = ceil_div(p.H, 128), CHI = ceil_div(p.I, 128);
    const int T1 = p.I / 64, T2 = ceil_div(p.H, kRowTile);   // units per expert, down row tiles
    const int TG = kDnRegion / nrows;                           // down tiles per accumulator region
    const int NG = ceil_div(T2, TG);                            // down groups per unit
    const int nblk = p.H / 32, nitems = M * nblk;               // x-term items: (token, 32-element block)
    const int V = M == 1 ? 1 : (M == 2 ? 2 : 4);                // floats per row of a CTA's output copy
    const uint32_t tail_off = ((uint32_t)p.smem_bytes - tail_bytes(p.H, M)) & ~127u;
    const uint32_t ring_cap = tail_off & ~127u;
    uint8_t* hterm = ring + tail_off;                           // [2][kHTerm]
    float4* xch = reinterpret_cast<float4*>(ring + tail_off + 2 * kHTerm);   // [2][32]
    float* oacc = reinterpret_cast<float*>(ring + tail_off + 2 * kHTerm + 2 * 32 * 16);   // [H][M]

    // warm L2 and the TLB for what the first steps read once the previous grid
    // is complete (a prefetch returns no data, so it cannot see a stale value)
    if (warp == 2 && lane < M)
        prefetch_l2(p.logits + (size_t)lane * p.E);
    if (warp >= 3 && warp <= 5 && b < nitems) {
        const int it = b + G * (warp - 3);
        if (it < nitems) {
            const int m = it / nblk, kb = it - m * nblk;
            if (lane == 0)
                prefetch_l2((p.x ? p.x : p.resid) + (size_t)m * p.H + 32 * kb);
        }
    }
    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.accf[i], 1);
            mbar_init(&sh.acce[i], 4);
            mbar_init(&sh.dnf[i], 2);
            mbar_init(&sh.dne[i], 4);
            mbar_init(&sh.hbar[i], 1);
        }
        mbar_init(&sh.routed, 1);
        mbar_init(&sh.xready, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(su32(&sh.tmem_base)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    // everything below reads what the previous grid in the stream wrote (the
    // logits, x, the residual) or shares its workspace
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp < 2 || warp == kMmaWarpB) {
        // ---- routing (warps 0, 1, 6): token m on the (m % 3)-th of them, then the
        // distinct experts in ascending order
#pragma unroll 1
        for (int m = warp == kMmaWarpB ? 2 : warp; m < M; m += 3)
            rt::warp_topk_fit(p.logits + (size_t)m * p.E, p.E, p.k, sh.sel[m], sh.wt[m]);
        route_barrier();
        if (warp == 0) {
            uint32_t bits = 0;
            if (lane < kMaxExperts / 32)
                for (int m = 0; m < M; ++m)
                    for (int s = 0; s < p.k; ++s) {
                        const int e = sh.sel[m][s];
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
                sh.unit_of[e] = (unsigned char)u;
                sh.unit_expert[u] = e;
                ++u;
            }
            const int nu = __shfl_sync(0xffffffffu, incl, 31);
            for (int x = lane; x < nu * kMaxTokens; x += 32)
                sh.wslot[x / kMaxTokens][x % kMaxTokens] = 0.f;
            __syncwarp();
            for (int x = lane; x < M * p.k; x += 32) {
                const int m = x / p.k, k2 = x % p.k;
                sh.wslot[sh.unit_of[sh.sel[m][k2]]][m] = sh.wt[m][k2];
            }
            if (lane == 0)
                sh.nu = nu;
        }
        route_barrier();
        if (warp == 1 && lane == 0)
            mbar_arrive(&sh.routed);   // hands the routing to the epilogue warps
    } else if (warp <= 5) {
        // ---- x terms (warps 2..5): items b + G q + 4 G i, token-major (q = warp - 2)
        const int q = warp - 2, te = tid - 64;
        if (b < nitems) {
            int cm = -1;
            float inv = 1.f;
            for (int it = b + G * q; it < nitems; it += 4 * G) {
                const int m = it / nblk, kb = it - m * nblk;
                float v;
                if (p.x) {
                    v = bf16f(__ldcg(p.x + (size_t)m * p.H + 32 * kb + lane));
                } else {
                    if (m != cm) {
                        inv = row_inv_rms(p.resid + (size_t)m * p.H, p.H, lane);
                        cm = m;
                    }
                    v = bf16f(f2bf16_rne(bf16f(__ldcg(p.resid + (size_t)m * p.H + 32 * kb + lane)) * inv));
                }
                float r4[kMaxTokens] = {v, 0.f, 0.f, 0.f};
                warp_terms_rows<1>(r4, m, kb, p.xt, p.xt + (long long)KSH * atom, atom, lane);
            }
        }
        epi_barrier();
        if (te == 0) {
            // publish this CTA's x terms (every CTA counts itself in), then wait for
            // the whole count and hand it to the producer through an mbarrier, so the
            // producer never waits on a load
            const unsigned long long tgt = count_target(atom_add_release_u64(p.xcnt, 1ull), G);
            int spins = 0;
#pragma unroll 1
            while (ld_acquire_u64(p.xcnt) < tgt) {
                if (++spins > (1 << 24)) {
                    atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                    break;
                }
            }
            mbar_arrive(&sh.xready);
        }
        __syncwarp();   // lane 0 rejoins before the warp's collective instructions
        for (int i = te; i < p.H * M; i += kEpi)
            oacc[i] = 0.f;
        // h'-term rows past M * 8 feed MMA columns nobody reads: give them zero
        // codes and unit-range scales rather than whatever shared memory held
        for (int i = te; i < 2 * kHTerm / 4; i += kEpi)
            reinterpret_cast<uint32_t*>(hterm)[i] = 0u;
        mbar_wait(&sh.routed, 0, p.status);
    }

    const int nu = sh.nu;
    const int U = nu * T1;
    // (products below stay under 2^31: U <= kMaxUnits * kMaxK / 64, G and H small)
    const int u0 = (int)((unsigned)b * U / G), nun = (int)((unsigned)(b + 1) * U / G) - u0;
    const int nact = U < G ? U : G;   // CTAs with units
    const int nitem = 2 * nun;
    if (b == 0 && tid == 0 && p.nu_out)
        *p.nu_out = nu;

    if (warp == 0) {
        // ================================================================ producer
        // Weights stream in item order.  A gate/up stage also carries the x terms
        // of its k-steps; until they are published those two copies wait in a
        // queue, served whenever the producer polls, so weights never wait.
        RingTc ring_alloc;
        unsigned long long ends[kSlots];
        unsigned long long rel_end = 0;
        uint32_t c = 0, rel = 0;
        const uint64_t wpol = l2_evict_first();
        uint32_t pq_off[kPend] = {}, pq_slot[kPend] = {};
        int pq_ks[kPend] = {}, pq_steps[kPend] = {};
        int pq_n = 0;
        bool x_ok = false;
        // the whole warp: once the x terms are all published (a non-blocking test),
        // issue the queued copies
        auto poll = [&]() {
            if (!x_ok && __shfl_sync(0xffffffffu, mbar_test_wait(&sh.xready, 0) ? 1 : 0, 0)) {
                __syncwarp();
                asm volatile("fence.proxy.async.global;" ::: "memory");   // published x terms -> bulk reads
                x_ok = true;
            }
            if (x_ok && pq_n > 0) {
                const int qq = lane >> 1;
                if (qq < pq_n) {
                    const GuStage sg(pq_steps[qq], atom);
                    if ((lane & 1) == 0)
                        bulk_copy(ring + pq_off[qq], p.xt + (long long)pq_ks[qq] * atom, sg.bbytes,
                                  &sh.full[pq_slot[qq]]);
                    else
                        bulk_copy(ring + pq_off[qq] + sg.bbytes,
                                  p.xt + (long long)KSH * atom + (pq_ks[qq] >> 1) * kSfChunk, sg.sfbytes,
                                  &sh.full[pq_slot[qq]]);
                }
                pq_n = 0;
            }
        };
        // the whole warp: claim ring bytes and a slot for a stage (stages retire in order)
        auto claim = [&](uint32_t size, uint32_t& off) -> uint32_t {
            unsigned long long end;
            off = ring_alloc.place(size, ring_cap, &end);
            int spins = 0;
#pragma unroll 1
            while (rel < c && (end - rel_end > (unsigned long long)ring_cap || rel + kSlots <= c)) {
                const uint32_t sl = rel % kSlots;
                if (__shfl_sync(0xffffffffu, mbar_test_wait(&sh.empty[sl], (rel / kSlots) & 1) ? 1 : 0, 0)) {
                    rel_end = ends[sl];
                    ++rel;
                } else {
                    poll();
                    if (++spins > (1 << 22)) {
                        if (lane == 0)
                            atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                        break;
                    }
                }
            }
            const uint32_t slot = c % kSlots;
            ends[slot] = end;
            return slot;
        };
        for (int k = 0; k < nitem; ++k) {
            bool down;
            int i;
            item_at(k, nun, down, i);
            const int unit = u0 + i, s = unit / T1, t = unit % T1;
            const int e = sh.unit_expert[s];
            if (!down) {
                const uint8_t* a0 = p.gu + (long long)e * p.gu_expert + (long long)t * kRowTile * (p.H / 2);
                const uint8_t* s0 = p.gu + (long long)e * p.gu_expert + (long long)(2 * p.I) * (p.H / 2) +
                                    (long long)t * CHH * kSfChunk;
                for (int ks = 0; ks < KSH; ks += kGuSteps, ++c) {
                    const int steps = KSH - ks < kGuSteps ? KSH - ks : kGuSteps;
                    const GuStage sg(steps, atom);
                    uint32_t off;
                    const uint32_t slot = claim(sg.size, off);
                    if (lane == 0)
                        mbar_expect_tx(&sh.full[slot], sg.abytes + sg.sfbytes + sg.bbytes + sg.sfbytes);
                    __syncwarp();
                    uint8_t* st = ring + off;
                    const uint8_t* src = nullptr;
                    uint32_t dsto = 0, n = 0;
                    switch (lane) {
                    case 0: dsto = 0; src = a0 + (long long)ks * kTileA; n = sg.abytes; break;
                    case 1: dsto = sg.sfa; src = s0 + (ks >> 1) * kSfChunk; n = sg.sfbytes; break;
                    case 2: dsto = sg.b; src = p.xt + (long long)ks * atom; n = x_ok ? sg.bbytes : 0u; break;
                    case 3:
                        dsto = sg.sfb;
                        src = p.xt + (long long)KSH * atom + (ks >> 1) * kSfChunk;
                        n = x_ok ? sg.sfbytes : 0u;
                        break;
                    default: break;
                    }
                    if (n) {
                        if (lane < 2)   // weights: read once per call
                            bulk_copy_hint(st + dsto, src, n, &sh.full[slot], wpol);
                        else
                            bulk_copy(st + dsto, src, n, &sh.full[slot]);
                    }
                    if (!x_ok) {
                        if (pq_n == kPend) {   // full: wait for the x terms
#pragma unroll 1
                            for (int w = 0; w < (1 << 22) && pq_n == kPend; ++w)
                                poll();
                            if (pq_n == kPend) {
                                if (lane == 0)
                                    atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                                pq_n = 0;   // give up (those stages will time out)
                            }
                        }
                        pq_off[pq_n] = off + sg.b;
                        pq_slot[pq_n] = slot;
                        pq_ks[pq_n] = ks;
                        pq_steps[pq_n] = steps;
                        ++pq_n;
                    }
                    poll();
                }
            } else {
                // down rows of all tiles, k-step t of K = I (h rows 64t .. 64t+63)
                const uint8_t* d0 = p.dn + (long long)e * p.dn_expert;
                const uint8_t* sd0 = d0 + (long long)p.H * (p.I / 2) + (long long)(t >> 1) * kSfChunk;
                for (int g = 0; g < NG; ++g) {
                    const int ta = g * TG, tb = ta + TG < T2 ? ta + TG : T2;
                    for (int t2 = ta; t2 < tb; t2 += kDnStageTiles, ++c) {
                        const int n = tb - t2 < kDnStageTiles ? tb - t2 : kDnStageTiles;
                        uint32_t off;
                        const uint32_t slot = claim(dn_stage_size(n), off);
                        uint32_t bytes = 0;
                        for (int j = 0; j < n; ++j) {
                            const int R2 = p.H - (t2 + j) * kRowTile < kRowTile ? p.H - (t2 + j) * kRowTile : kRowTile;
                            bytes += (uint32_t)R2 * 32 + kSfChunk;
                        }
                        if (lane == 0)
                            mbar_expect_tx(&sh.full[slot], bytes);
                        __syncwarp();
                        uint8_t* st = ring + off;
                        const int j = lane & 15;
                        if (j < n) {
                            const int tt = t2 + j;
                            const int R2 = p.H - tt * kRowTile < kRowTile ? p.H - tt * kRowTile : kRowTile;
                            if (lane < 16)
                                bulk_copy_hint(st + j * kTileA,
                                          d0 + (long long)tt * kRowTile * (p.I / 2) + (long long)t * R2 * 32,
                                          (uint32_t)R2 * 32, &sh.full[slot], wpol);
                            else
                                bulk_copy_hint(st + n * kTileA + j * kSfChunk, sd0 + (long long)tt * CHI * kSfChunk,
                                               kSfChunk, &sh.full[slot], wpol);
                        }
                    }
                }
            }
        }
#pragma unroll 1
        for (int w = 0; w < (1 << 22) && pq_n > 0; ++w)
            poll();
        if (pq_n > 0 && lane == 0)
            atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
    } else if (warp == 1 || warp == kMmaWarpB) {
        // ================================================================ MMA issuers
        // Issuing a tcgen05 instruction costs one thread ~60-80 cycles.  Issuer A
        // (warp 1) takes the gate/up stages; the down stages, which all wait on
        // the same h' and then run back to back, alternate between A and B
        // (warp 6), each on its own tiles of the region and its own scale sets.
        const int role = warp == 1 ? 0 : 1;
        if (lane == 0) {
            RingTc ring_alloc;
            const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(nrows >> 3) << 17) | (1u << 23) |
                                   ((uint32_t)(kRowTile >> 4) << 24);
            const uint32_t myset = tmem + kSfCol + role * 2 * kSfSet;
            uint32_t c = 0, kk = 0, mine = 0;
            for (int k = 0; k < nitem; ++k) {
                bool down;
                int i;
                item_at(k, nun, down, i);
                const int t = (u0 + i) % T1;
                if (!down) {
                    if (role == 1) {   // issuer A's: only keep the ring placement in step
                        for (int ks = 0; ks < KSH; ks += kGuSteps, ++c) {
                            const int steps = KSH - ks < kGuSteps ? KSH - ks : kGuSteps;
                            unsigned long long end;
                            ring_alloc.place(GuStage(steps, atom).size, ring_cap, &end);
                        }
                        continue;
                    }
                    const uint32_t buf = i & 1;
                    if (i >= 2)
                        mbar_wait(&sh.acce[buf], ((i >> 1) - 1) & 1, p.status);
                    tc_fence_after();
                    const uint32_t d = tmem + kGuCol + buf * 32;
                    bool first = true;
                    for (int ks = 0; ks < KSH; ks += kGuSteps, ++c) {
                        const int steps = KSH - ks < kGuSteps ? KSH - ks : kGuSteps;
                        const GuStage sg(steps, atom);
                        unsigned long long end;
                        const uint32_t st = su32(ring) + ring_alloc.place(sg.size, ring_cap, &end);
                        const uint32_t slot = c % kSlots;
                        mbar_wait(&sh.full[slot], (c / kSlots) & 1, p.status);
                        tc_fence_after();
                        const uint32_t set = myset + (mine++ & 1) * kSfSet;
                        const int chunks = (steps + 1) >> 1;
#pragma unroll 1
                        for (int ch = 0; ch < chunks; ++ch) {
                            tc_cp_sf(set + 4 * ch, st + sg.sfa + ch * kSfChunk);
                            tc_cp_sf(set + kSfSet / 2 + 4 * ch, st + sg.sfb + ch * kSfChunk);
                        }
#pragma unroll 1
                        for (int j = 0; j < steps; ++j) {
                            const uint32_t id = (uint32_t)(2 * (j & 1));
                            tc_mma_mxf4(d, smem_desc(st + j * kTileA, 128, 256), smem_desc(st + sg.b + j * atom, 128, 256),
                                        idesc | (id << 4) | (id << 29), set + 4 * (j >> 1),
                                        set + kSfSet / 2 + 4 * (j >> 1), first ? 0u : 1u);
                            first = false;
                        }
                        tc_commit(&sh.empty[slot]);
                    }
                    tc_commit(&sh.accf[buf]);
                } else {
                    const uint32_t hb = su32(hterm + (i & 1) * kHTerm);
                    mbar_wait(&sh.hbar[i & 1], (i >> 1) & 1, p.status);
                    tc_fence_after();
                    const uint32_t aid = (uint32_t)(2 * (t & 1));   // A scale bytes of k-step t in its chunk
                    int jst = 0;                                     // down stage of this unit
                    for (int g = 0; g < NG; ++g, ++kk) {
                        if (kk >= 2)
                            mbar_wait(&sh.dne[kk & 1], ((kk >> 1) - 1) & 1, p.status);
                        tc_fence_after();
                        const uint32_t dreg = tmem + kDnCol + (kk & 1) * kDnRegion;
                        const int ta = g * TG, tb = ta + TG < T2 ? ta + TG : T2;
                        for (int t2 = ta; t2 < tb; t2 += kDnStageTiles, ++c, ++jst) {
                            const int n = tb - t2 < kDnStageTiles ? tb - t2 : kDnStageTiles;
                            unsigned long long end;
                            const uint32_t st = su32(ring) + ring_alloc.place(dn_stage_size(n), ring_cap, &end);
                            if ((jst & 1) != role)
                                continue;   // the other issuer's stage
                            const uint32_t slot = c % kSlots;
                            mbar_wait(&sh.full[slot], (c / kSlots) & 1, p.status);
                            tc_fence_after();
                            const uint32_t set = myset + (mine++ & 1) * kSfSet;
                            tc_cp_sf(set, hb + 1024);
#pragma unroll 1
                            for (int j = 0; j < n; ++j)
                                tc_cp_sf(set + 4 + 4 * j, st + n * kTileA + j * kSfChunk);
#pragma unroll 1
                            for (int j = 0; j < n; ++j)
                                tc_mma_mxf4(dreg + (t2 - ta + j) * nrows, smem_desc(st + j * kTileA, 128, 256),
                                            smem_desc(hb, 128, 256), idesc | (aid << 29), set + 4 + 4 * j, set, 0u);
                            tc_commit(&sh.empty[slot]);
                        }
                        tc_commit(&sh.dnf[kk & 1]);   // both issuers: the group's region is full
                    }
                }
            }
        }
    } else {
        // ================================================================ epilogue warps
        const int te = tid - 64, q = warp & 3;   // q: the lane quarter this warp may read
        uint32_t kk = 0;
        for (int k = 0; k < nitem; ++k) {
            bool down;
            int i;
            item_at(k, nun, down, i);
            const int unit = u0 + i, s = unit / T1, t = unit % T1;
            if (!down) {
                // ---- gate (rows 0..63) and up (rows 64..127) sums of 64 h rows; the
                // biases are loaded before the accumulator is waited for
                const uint32_t buf = i & 1;
                const int hrow = 64 * t + 32 * (q & 1) + lane;
                const int e = sh.unit_expert[s];
                float bg = 0.f, bu = 0.f;
                if (q < 2 && p.gu_bias) {
                    bg = bf16f(__ldg(p.gu_bias + (size_t)e * 2 * p.I + hrow));
                    bu = bf16f(__ldg(p.gu_bias + (size_t)e * 2 * p.I + p.I + hrow));
                }
                mbar_wait(&sh.accf[buf], (i >> 1) & 1, p.status);
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + kGuCol + buf * 32;
                float sm[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int h16 = 0; h16 < 32; h16 += 16) {
                    if (h16 < nrows) {
                        float d0[16];
                        tc_ld16(taddr + h16, d0);
                        tc_wait_ld();
#pragma unroll
                        for (int col = 0; col < 16; ++col) {
                            const int m = (h16 + col) / kTerms;   // compile-time after unrolling
                            if (m < M)
                                sm[m] += d0[col];
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sh.acce[buf]);
                if (q >= 2)
                    xch[(q - 2) * 32 + lane] = make_float4(sm[0], sm[1], sm[2], sm[3]);
                epi_barrier();
                if (q < 2) {
                    // h'_m = w_m silu(gate + b) (up + b) for h row 64t + 32q + lane: one
                    // 32-element block (k-block q of the down k-step t)
                    const float4 u4 = xch[q * 32 + lane];
                    const float us[kMaxTokens] = {u4.x, u4.y, u4.z, u4.w};
                    float hv[kMaxTokens];
#pragma unroll
                    for (int m = 0; m < kMaxTokens; ++m) {
                        const float g = sm[m] + bg;
                        hv[m] = m < M ? sh.wslot[s][m] * (g / (1.0f + expf(-g))) * (us[m] + bu) : 0.f;
                    }
                    uint8_t* hb = hterm + buf * kHTerm;
                    switch (M) {   // one copy of the code runs
                    case 1: warp_terms_rows<1>(hv, 0, q, hb, hb + 1024, atom, lane); break;
                    case 2: warp_terms_rows<2>(hv, 0, q, hb, hb + 1024, atom, lane); break;
                    case 3: warp_terms_rows<3>(hv, 0, q, hb, hb + 1024, atom, lane); break;
                    default: warp_terms_rows<4>(hv, 0, q, hb, hb + 1024, atom, lane); break;
                    }
                    fence_proxy_async_smem();
                }
                epi_barrier();
                if (te == 0)
                    mbar_arrive(&sh.hbar[buf]);
            } else {
                // ---- down products of unit i into the CTA's output copy
                for (int g = 0; g < NG; ++g, ++kk) {
                    mbar_wait(&sh.dnf[kk & 1], (kk >> 1) & 1, p.status);
                    tc_fence_after();
                    const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + kDnCol + (kk & 1) * kDnRegion;
                    const int ta = g * TG, tb = ta + TG < T2 ? ta + TG : T2;
                    for (int t2 = ta; t2 < tb; ++t2) {
                        float sm[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int h16 = 0; h16 < 32; h16 += 16) {
                            if (h16 < nrows) {
                                float d0[16];
                                tc_ld16(taddr + (t2 - ta) * nrows + h16, d0);
                                tc_wait_ld();
#pragma unroll
                                for (int col = 0; col < 16; ++col) {
                                    const int m = (h16 + col) / kTerms;
                                    if (m < M)
                                        sm[m] += d0[col];
                                }
                            }
                        }
                        const int row = t2 * kRowTile + 32 * q + lane;
                        if (row < p.H)
#pragma unroll
                            for (int m = 0; m < kMaxTokens; ++m)
                                if (m < M)
                                    oacc[row * M + m] += sm[m];
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sh.dne[kk & 1]);
                }
            }
        }
        // ---- the CTA's output copy to its partial slot [H][V] (rows drained by other warps)
        epi_barrier();
        if (nun > 0) {
            float* dst = p.part + (size_t)b * p.H * V;
            for (int row = te; row < p.H; row += kEpi) {
                float v[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m)
                    if (m < M)
                        v[m] = oacc[row * M + m];
                if (V == 1)
                    dst[row] = v[0];
                else if (V == 2)
                    reinterpret_cast<float2*>(dst)[row] = make_float2(v[0], v[1]);
                else
                    reinterpret_cast<float4*>(dst)[row] = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
    }

    // ---- this CTA's output rows [r0, r1): their bias terms sum_s w_s b_s and the
    // residual are loaded before the grid barrier
    const int r0 = (int)((unsigned)b * p.H / G), r1 = (int)((unsigned)(b + 1) * p.H / G);
    const int nr = r1 - r0;
    float bsum[kMaxTokens] = {0.f, 0.f, 0.f, 0.f}, rv[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
    if (tid < nr) {
        const int row = r0 + tid;
        if (p.dn_bias)
            for (int s2 = 0; s2 < nu; ++s2) {
                const float bd = bf16f(__ldg(p.dn_bias + (size_t)sh.unit_expert[s2] * p.H + row));
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m)
                    bsum[m] = fmaf(sh.wslot[s2][m], bd, bsum[m]);
            }
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m)
            if (m < M)
                rv[m] = bf16f(__ldcg(p.resid + (size_t)m * p.H + row));
    }

    // ---- grid barrier: every CTA's output copy is stored (every CTA counts itself in)
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        const unsigned long long tgt = count_target(atom_add_release_u64(p.done, 1ull), G);
        int spins = 0;
#pragma unroll 1
        while (ld_acquire_u64(p.done) < tgt) {
            if (++spins > (1 << 24)) {
                atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                break;
            }
        }
    }
    __syncthreads();

    // ---- output rows [r0, r1): the active CTAs' copies summed in CTA order, split
    // over P thread groups (group g takes CTAs g, g + P, ...), then the groups in order
    if (nr > 0) {
        float4* red = reinterpret_cast<float4*>(ring);   // [P][nr]; the ring is idle now
        const int P = kThreadsTc / nr < 1 ? 1 : kThreadsTc / nr;
        if (tid < P * nr) {
            const int j = tid % nr, g = tid / nr;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            // group g's CTAs: with U >= G every CTA, else the owners of the U units
            auto cta_of = [&](int cc) { return U < G ? (int)(((unsigned)(cc + 1) * G + U - 1) / U) - 1 : cc; };
            // the copies' rows are V floats; one loop per V, so one copy of the code runs
            auto sum_rows = [&](auto vtag) {
                using VT = decltype(vtag);
                constexpr int VW = sizeof(VT) / sizeof(float);
                for (int c0 = g; c0 < nact; c0 += 8 * P) {
                    VT a[8];
#pragma unroll
                    for (int z = 0; z < 8; ++z)
                        if (c0 + z * P < nact)
                            a[z] = __ldcg(reinterpret_cast<const VT*>(p.part + ((size_t)cta_of(c0 + z * P) * p.H + r0 + j) * VW));
#pragma unroll
                    for (int z = 0; z < 8; ++z)
                        if (c0 + z * P < nact) {
                            const float* f = reinterpret_cast<const float*>(&a[z]);
                            acc.x += f[0];
                            if (VW > 1) acc.y += f[VW > 1 ? 1 : 0];
                            if (VW > 2) { acc.z += f[VW > 2 ? 2 : 0]; acc.w += f[VW > 2 ? 3 : 0]; }
                        }
                }
            };
            if (V == 1)
                sum_rows(0.f);
            else if (V == 2)
                sum_rows(make_float2(0.f, 0.f));
            else
                sum_rows(make_float4(0.f, 0.f, 0.f, 0.f));
            red[g * nr + j] = acc;
        }
        __syncthreads();
        if (tid < nr) {
            const int row = r0 + tid;
            float acc[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
            for (int g = 0; g < P; ++g) {
                const float4 a = red[g * nr + tid];
                acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            }
#pragma unroll
            for (int m = 0; m < kMaxTokens; ++m)
                if (m < M)
                    p.resid[(size_t)m * p.H + row] = f2bf16_rne(rv[m] + (acc[m] + bsum[m]));
        }
    }

    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

}  // namespace

cudaError_t prepare_decode_tc(size_t smem)
{
    return cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

size_t decode_tc_static_smem()
{
    cudaFuncAttributes a{};
    return cudaFuncGetAttributes(&a, decode_tc_kernel) == cudaSuccess ? a.sharedSizeBytes : 0;
}

cudaError_t launch_decode_tc(const DecodeTcParams& p, size_t smem, int grid, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel, p);
}

}  // namespace moe
