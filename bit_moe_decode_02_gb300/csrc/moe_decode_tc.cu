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
// 64 matching K columns for every output row.  Each CTA takes q = U / G whole
// units; the U mod G leftover units are cut into pieces (a K range of the
// gate/up, a range of the down tiles) whose CTAs exchange only their gate/up
// partial sums (see make_plan).  Each CTA adds its down products into its own
// fp32 copy of the output, and after one grid barrier CTA b sums the CTAs'
// copies for its slice of the output rows in CTA order (results do not depend
// on timing) and writes out = bf16(r + sum + sum_s w_s b_s).
//
// The x terms are built inside the layer: the (token, 32-element block) items
// are dealt over the CTAs, written to global memory and counted; once the
// count is complete each CTA copies the whole set into shared memory, where it
// stays for the layer.  Weight copies never wait on activations.
//
// The launch signals its dependents at entry, so the next layer's CTAs take
// over each SM as soon as this layer's CTA there exits and set up before they
// wait for this grid to complete.
//
// Warp roles (256 threads): warp 0 streams weights into a byte ring of shared
// memory (a stage's copies issued from separate lanes); warps 1 and 6 issue
// the MMAs, each half of every stage (warp 1 owns tensor memory); warps 2..5
// (one per lane quarter) build the x terms and drain the accumulators; warp 7
// works out the plans before the grid wait and combines a split unit's partial
// sums.  Warps 0, 1 and 6 route.
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
constexpr int kDnStageTiles = 4;     // 128-row down tiles per down stage
constexpr int kSlots = 16;           // stages in flight at most
// tensor memory columns
constexpr int kGuCol = 0;            // gate/up accumulators: 2 buffers x (issuer A | B) x 32
constexpr int kGuBuf = 64;
constexpr int kDnCol = 128;          // down accumulators: 2 regions x 128
constexpr int kDnRegion = 128;
constexpr int kSfCol = 384;          // stage scale sets: 2 issuers x 2 sets x 32
static_assert(kGuCol + 2 * kGuBuf <= kDnCol, "gate/up accumulators");
constexpr int kSfSet = 32;
constexpr int kTmemCols = 512;
static_assert(kDnCol + 2 * kDnRegion <= kSfCol && kSfCol + 4 * kSfSet <= kTmemCols, "tensor memory");
static_assert(kDnRegion % (kDnStageTiles * 32) == 0, "a region holds whole down stages");
static_assert(kSfSet >= 8 * ((kGuSteps + 1) / 2), "a gate/up stage's A and B scale chunks fit a set");
static_assert(kSfSet == 32 && 4 * ((kDnStageTiles + 1) / 2) <= 24 && kSfSet / 2 + 4 * ((kGuSteps + 3) / 4) <= 24,
              "an issuer's stage scale chunks use columns 0..23 of a set; 24..31 hold the h' scales");
constexpr int kThreadsTc = 256;      // producer, MMA issuer A, 4 epilogue warps, MMA issuer B, combiner
constexpr int kMmaWarpB = 6;
constexpr int kCombineWarp = 7;
constexpr int kEpi = 128;            // epilogue threads (warps 2..5)
constexpr int kTileA = kRowTile * 32;            // one k-step of a 128-row tile: 4 KB
constexpr int kHTerm = kHTermBytes;              // h' terms of a unit: one k-step atom + its scale chunk

// MMA N: the rows that hold terms, rounded up to 16; a k-step of terms is
// N rows x 32 bytes (8-row groups 256 bytes apart).
__device__ __forceinline__ int rows_for(int M) { return M * kTerms <= 16 ? 16 : 32; }

// Shared memory past the stage ring: the layer's x terms (H/64 k-step atoms,
// then ceil(H/128) scale chunks, then 2^-S_m of each token), three h'-term buffers (two for whole units,
// one for a split unit's), the up-sum exchange (2 warps x 32 lanes x float4)
// and the CTA's fp32 output copy [H][M].
__device__ __forceinline__ uint32_t xterm_bytes(int H, int atom)
{
    return (uint32_t)(H / 64) * atom + (uint32_t)ceil_div(H, 128) * kSfChunk + 16;
}
__device__ __forceinline__ uint32_t tail_bytes(int H, int M, int atom)
{
    return ((xterm_bytes(H, atom) + 127) & ~127u) + 3 * kHTerm + 2 * 32 * 16 + (((uint32_t)H * M * 4 + 127) & ~127u);
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

// What a CTA does.  With U >= G units and rem = U mod G left over after q
// whole units per CTA, a leftover unit is split in S = min(G / rem, ...) pieces
// (S >= 2), each a K range of its gate/up and a range of its down tiles: piece
// p of leftover unit j goes to CTA j S + p.  The pieces publish their gate/up
// partial sums; every piece's CTA adds all of them in piece order (the same
// fp32 operations everywhere, so the same h') and computes the unit's h' for
// its own down tiles -- a warp of its own does this, so neither the weight
// stream nor the drains wait for the exchange.  Otherwise the units are
// dealt whole, CTA b taking [b U / G, (b+1) U / G).
struct Plan {
    int u0, nun;          // whole units [u0, u0 + nun)
    int piece;            // 1: this CTA holds a piece of a split unit
    int su, sj, pp, S;    // the split unit, its leftover index, the piece, the pieces
    int ks0, ks1, ta, tb; // the piece's gate/up k-steps and down tiles
    int nitem;
};
__device__ __forceinline__ Plan make_plan(int b, int G, int U, int KSH, int CHH, int T2)
{
    Plan pl{};
    const int q = U / G, rem = U - q * G;
    int S = rem > 0 ? G / rem : 0;
    S = S < CHH ? S : CHH;
    S = S < T2 ? S : T2;
    if (q >= 1 && S >= 2) {
        pl.u0 = b * q;
        pl.nun = q;
        if (b < rem * S) {
            pl.piece = 1;
            pl.sj = b / S;
            pl.pp = b - pl.sj * S;
            pl.S = S;
            pl.su = G * q + pl.sj;
            const int c0 = pl.pp * CHH / S, c1 = (pl.pp + 1) * CHH / S;
            pl.ks0 = 2 * c0;
            pl.ks1 = 2 * c1 < KSH ? 2 * c1 : KSH;
            pl.ta = pl.pp * T2 / S;
            pl.tb = (pl.pp + 1) * T2 / S;
        }
    } else {
        pl.u0 = (int)((unsigned)b * U / G);
        pl.nun = (int)((unsigned)(b + 1) * U / G) - pl.u0;
    }
    pl.nitem = 2 * pl.nun + 2 * pl.piece;
    return pl;
}

// Plans for the distinct-expert counts a call can have (nu = k .. min(M k, E)),
// worked out before the routing is known, so the integer divisions of
// make_plan are off the path from the routing to the first weight copy.  The
// fields fit 16 bits: every one is at most U <= kMaxUnits * kMaxK / 64 = 3072.
constexpr int kPlanTab = 32;
struct PackedPlan {
    short v[12];
};
__device__ __forceinline__ PackedPlan pack_plan(const Plan& pl)
{
    PackedPlan q;
    const int f[12] = {pl.u0, pl.nun, pl.piece, pl.su, pl.sj, pl.pp, pl.S, pl.ks0, pl.ks1, pl.ta, pl.tb, pl.nitem};
#pragma unroll
    for (int i = 0; i < 12; ++i)
        q.v[i] = (short)f[i];
    return q;
}
__device__ __forceinline__ Plan unpack_plan(const PackedPlan& q)
{
    Plan pl;
    pl.u0 = q.v[0]; pl.nun = q.v[1]; pl.piece = q.v[2]; pl.su = q.v[3]; pl.sj = q.v[4]; pl.pp = q.v[5];
    pl.S = q.v[6]; pl.ks0 = q.v[7]; pl.ks1 = q.v[8]; pl.ta = q.v[9]; pl.tb = q.v[10]; pl.nitem = q.v[11];
    return pl;
}

enum ItemKind { kGu = 0, kDn = 1, kGuPiece = 2, kDnPiece = 3 };
// Item k of a plan: the piece's gate/up first (its partial sums are published
// early), the whole units' items, the piece's down tiles last.  The epilogue
// combines the pieces' partials only after the last whole unit's gate/up, so
// that unit's SwiGLU never waits for the exchange.
__device__ __forceinline__ void item_of(const Plan& pl, int k, int& kind, int& i)
{
    if (pl.piece && k == 0) {
        kind = kGuPiece;
        i = 0;
    } else if (pl.piece && k == pl.nitem - 1) {
        kind = kDnPiece;
        i = 0;
    } else {
        bool down;
        item_at(k - pl.piece, pl.nun, down, i);
        kind = down ? kDn : kGu;
    }
}

// Gate/up stage: [A: steps x 4 KB][SFA: chunks x 512] (the x terms stay in
// shared memory for the whole layer).
struct GuStage {
    uint32_t abytes, sfbytes, sfa, size;
    __device__ GuStage(int steps)
    {
        abytes = steps * kTileA;
        sfbytes = ((steps + 1) >> 1) * kSfChunk;
        sfa = abytes;
        size = (sfa + sfbytes + 127) & ~127u;
    }
};
// Down stage of n tiles: [A: n x 4 KB][SFA: n x 512].  A partial tile (64 rows)
// still has a 4 KB slot, so the MMA's 128-row read stays inside the stage.
__device__ __forceinline__ uint32_t dn_stage_size(int n) { return (uint32_t)n * (kTileA + kSfChunk); }

struct RingTc {   // (value-initialise: RingTc{} starts at 0)
    unsigned long long head;
    uint32_t phys;
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
    // Packing: an 8 x 8 nibble transpose within each group of 8 lanes (3
    // butterfly exchanges of 16-, 8- and 4-bit fields) leaves lane 8g + i with
    // term i's codes of elements 8g .. 8g+7, one 32-bit store per lane per token;
    // lane i < 8 writes term i's scale byte.
    const int i8 = lane & 7;
#pragma unroll
    for (int m = 0; m < M; ++m) {
        uint32_t x = codes[m];
        uint32_t y = __shfl_xor_sync(0xffffffffu, x, 4);
        x = (lane & 4) ? ((x & 0xFFFF0000u) | (y >> 16)) : ((x & 0x0000FFFFu) | (y << 16));
        y = __shfl_xor_sync(0xffffffffu, x, 2);
        x = (lane & 2) ? ((x & 0xFF00FF00u) | ((y >> 8) & 0x00FF00FFu)) : ((x & 0x00FF00FFu) | ((y << 8) & 0xFF00FF00u));
        y = __shfl_xor_sync(0xffffffffu, x, 1);
        x = (lane & 1) ? ((x & 0xF0F0F0F0u) | ((y >> 4) & 0x0F0F0F0Fu)) : ((x & 0x0F0F0F0Fu) | ((y << 4) & 0xF0F0F0F0u));
        const int row = (m0 + m) * kTerms + i8;
        *reinterpret_cast<uint32_t*>(q + (kb >> 1) * atom + (row >> 3) * 256 + (kb & 1) * 128 + i8 * 16 +
                                     4 * (lane >> 3)) = x;
        if (lane < 8)
            sf[(kb >> 2) * kSfChunk + row * 16 + (kb & 3)] = (uint8_t)((i8 < 4 ? sblo[m] : sbhi[m]) >> (8 * (i8 & 3)));
    }
}

// A bf16 row of n elements (n % 8 == 0, n <= kMaxK) held by a warp: 16-byte
// vector i at lane i % 32, step i / 32 (the loads all in flight together).
constexpr int kRowVec = kMaxK / 8 / 32;
__device__ __forceinline__ void load_row(const uint16_t* row, int n, int lane, uint4 (&v)[kRowVec])
{
#pragma unroll
    for (int z = 0; z < kRowVec; ++z) {
        const int i = lane + 32 * z;
        v[z] = i < n / 8 ? __ldcg(reinterpret_cast<const uint4*>(row) + i) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Element 32 kb + lane of a row held as above: its vector 4 kb + lane / 8 is
// at step (4 kb) / 32 (the same for the four vectors of a block) on lane
// (4 kb) % 32 + lane / 8.
__device__ __forceinline__ uint16_t row_elem(const uint4 (&v)[kRowVec], int kb, int lane)
{
    const int zs = (4 * kb) >> 5;
    uint4 u = v[0];
#pragma unroll
    for (int z = 1; z < kRowVec; ++z)
        if (z == zs)
            u = v[z];
    const int src = ((4 * kb) & 31) + (lane >> 3);
    const uint32_t w0 = __shfl_sync(0xffffffffu, u.x, src), w1 = __shfl_sync(0xffffffffu, u.y, src);
    const uint32_t w2 = __shfl_sync(0xffffffffu, u.z, src), w3 = __shfl_sync(0xffffffffu, u.w, src);
    const int wi = (lane & 7) >> 1;
    const uint32_t w = wi == 0 ? w0 : (wi == 1 ? w1 : (wi == 2 ? w2 : w3));
    return (uint16_t)((lane & 1) ? w >> 16 : w & 0xffffu);
}

// Over a row held as above, the same values on every lane of the warp: the
// largest magnitude (as bf16 bits) and, with want_rms, 1 / sqrt(mean(v^2) + 1e-6).
__device__ __forceinline__ float row_stats(const uint4 (&v)[kRowVec], int n, bool want_rms, uint32_t& amax)
{
    float a = 0.f;
    uint32_t mx = 0u;
#pragma unroll
    for (int z = 0; z < kRowVec; ++z) {
        const uint32_t ws[4] = {v[z].x, v[z].y, v[z].z, v[z].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float lo = __uint_as_float(ws[c] << 16), hi = __uint_as_float(ws[c] & 0xffff0000u);
            a = fmaf(lo, lo, a);
            a = fmaf(hi, hi, a);
            mx = max(mx, max(ws[c] & 0x7fffu, (ws[c] >> 16) & 0x7fffu));
        }
    }
    amax = __reduce_max_sync(0xffffffffu, mx);
    if (!want_rms)
        return 1.f;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        a += __shfl_xor_sync(0xffffffffu, a, off);
    return 1.0f / sqrtf(a / (float)n + 1e-6f);
}

// The power-of-two factor 2^S (S >= 0) that a token's activation is multiplied
// by before it is cut into MX terms, from its largest magnitude amax.  Term j
// of a block has the shared exponent X0 - 2j, and E8M0 holds no exponent below
// -127, so a block with X0 < -113 would lose its last terms.  S = 0 unless
// the token's largest block exponent X0 = floor(log2 amax) - 2 is below -100;
// then S lifts it to -100.  Blocks far below the token's largest lose terms,
// at 2^-13 or less of its largest block's contribution.  The sums are
// multiplied by 2^-S afterwards (exact: both are powers of two, and no sum can
// overflow, since |x| 2^S < 2^-97 and |w| < 2^130).
__device__ __forceinline__ int token_shift(float amax)
{
    const uint32_t u = __float_as_uint(amax);
    if (u == 0u)
        return 0;
    const int e = u >= 0x00800000u ? (int)(u >> 23) - 127 : (31 - __clz((int)u)) - 149;   // floor(log2 amax)
    return -98 - e > 0 ? -98 - e : 0;
}

// Adds the down products of tiles [0, n) of an accumulator region (tile j at
// columns j * nrows, token m's terms at columns 8m .. 8m+7 of it) into the
// output copy oacc [H][M], row row0 + 128 j for this thread.  A TMEM load
// round trip costs far more than the sums, so TB tiles' loads go out before
// one wait: NC columns a tile (8 for one token, 16 for two, 32 for four).  The
// loads are unconditional (a batch never reaches past the region's 128
// columns; columns of absent tiles are read and dropped), the term sums are
// trees and the read-modify-writes of oacc are predicated, so the tiles of a
// batch run side by side instead of one branch after another.
template <int NC, int TB>
__device__ __forceinline__ void drain_region(uint32_t taddr, int n, int nrows, int row0, float* oacc, int H, int M)
{
    constexpr int W = NC < 16 ? NC : 16;   // columns per load instruction
    constexpr int P = NC / W;              // loads per tile
    constexpr int T = NC / 8;              // tokens a tile holds
#pragma unroll 1
    for (int j0 = 0; j0 < n; j0 += TB) {
        float d[TB * P][W];
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const uint32_t a = taddr + (uint32_t)((j0 + j) * nrows);
#pragma unroll
            for (int h = 0; h < P; ++h) {
                if constexpr (W == 8)
                    tc_ld8(a, d[j * P + h]);
                else
                    tc_ld16(a + 16 * h, d[j * P + h]);
            }
        }
        tc_wait_ld();
        float s[TB][T];
#pragma unroll
        for (int j = 0; j < TB; ++j)
#pragma unroll
            for (int m = 0; m < T; ++m) {
                float v[kTerms];
#pragma unroll
                for (int c = 0; c < kTerms; ++c)
                    v[c] = d[j * P + (8 * m + c) / W][(8 * m + c) % W];
                s[j][m] = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
            }
        bool ok[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j)
            ok[j] = j0 + j < n && row0 + (j0 + j) * kRowTile < H;
        if constexpr (NC == 8) {
            float o[TB];
#pragma unroll
            for (int j = 0; j < TB; ++j)
                o[j] = ok[j] ? oacc[row0 + (j0 + j) * kRowTile] : 0.f;
#pragma unroll
            for (int j = 0; j < TB; ++j)
                if (ok[j])
                    oacc[row0 + (j0 + j) * kRowTile] = o[j] + s[j][0];
        } else if constexpr (NC == 16) {
            float2* o2 = reinterpret_cast<float2*>(oacc);
            float2 o[TB];
#pragma unroll
            for (int j = 0; j < TB; ++j)
                o[j] = ok[j] ? o2[row0 + (j0 + j) * kRowTile] : make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < TB; ++j)
                if (ok[j])
                    o2[row0 + (j0 + j) * kRowTile] = make_float2(o[j].x + s[j][0], o[j].y + s[j][1]);
        } else {
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                const int row = row0 + (j0 + j) * kRowTile;
                if (ok[j]) {
                    if (M == 4) {
                        float4* o = reinterpret_cast<float4*>(oacc) + row;
                        const float4 v = *o;
                        *o = make_float4(v.x + s[j][0], v.y + s[j][1], v.z + s[j][2], v.w + s[j][3]);
                    } else {
#pragma unroll
                        for (int m = 0; m < 3; ++m)
                            oacc[row * 3 + m] += s[j][m];
                    }
                }
            }
        }
    }
}

constexpr int kFinSlots = 64;   // output float4s of a CTA's slice whose final terms are prefetched

// The running state of a role across the calls of a launch: every mbarrier
// phase and ring position follows it.  Kept in shared memory between calls (a
// role's threads load it when a call starts, its owner stores it back), so no
// register holds it across the loop over calls.
struct RoleState {
    RingTc rs;                    // producer / MMA issuers: the stage ring
    uint32_t sc;                  // producer / MMA issuers: stages so far
    uint32_t rel;                 // producer: stages released
    unsigned long long rel_end;   // producer: ring position released
    uint32_t kk;                  // MMA issuers / epilogue: down region groups
    uint32_t sfn;                 // MMA issuers: scale-factor sets used
};

struct TcSmem {
    uint64_t full[kSlots], empty[kSlots];
    uint64_t accf[2], acce[2];   // gate/up accumulator buffers: full / drained
    uint64_t dnf[2], dne[2];     // down accumulator regions: full (both issuers) / drained
    uint64_t hbar[2];            // h' terms of a unit written
    uint64_t routed, xfull;      // routing done; the layer's x terms copied in
    uint64_t hsfull;             // the split unit's h' terms copied in
    uint64_t planbar;            // the plan table is written
    uint64_t rlogw, xready;      // in-kernel router: this CTA's logits stored; every CTA's published
    uint64_t rbar;               // in-kernel router: this CTA's router rows copied in
    unsigned epoch;              // this call's tag for the exchange flags (call index + 1)
    uint32_t tmem_base;
    int sel[kMaxTokens][kMaxTopK];
    float wt[kMaxTokens][kMaxTopK];
    int nu;
    int unit_expert[kMaxUnits];
    unsigned char unit_of[kMaxExperts];
    float wslot[kMaxUnits][kMaxTokens];   // routing weight of token m for expert slot s (0 if not chosen)
    float fin[kFinSlots][4];              // r + sum_s w_s b_s of the slice's elements (loaded before the grid barrier)
    PackedPlan plan_tab[kPlanTab];        // plan of nu = k + i distinct experts
    unsigned long long ends[kSlots];      // producer: ring position after each stage in flight
    RoleState role[4];                    // producer, MMA issuer A, MMA issuer B, epilogue
    int gbase, ubase, npc;                // gate/up items, whole units and split-unit calls so far
    uint16_t* cresid;                     // the call's residual buffer
    unsigned long long dtgt, xtgt;        // targets of the last grid barrier and x-term count
};

// The launch's shared state: the stage ring (dynamic), the control block and a
// copy of the parameters (read by every call).
extern __shared__ __align__(1024) uint8_t ring[];
__shared__ __align__(8) TcSmem sh;
__shared__ DecodeTcParams g_p;

// The router GEMV of one CTA: logits of experts e = b, b + G, ... (their
// router rows already in shared memory at wsm, H bf16 each) for tokens m = m0,
// m0 + 3, ... (one warp), written to rlog [M][E].  The input is the layer
// input the x terms are cut from: x, or the normalised residual rounded to
// bf16 exactly as the x terms round it; the warp stages it in shared memory at
// xsm, so that the product loop keeps few registers.  Each logit is a
// lane-strided fp32 FMA chain and a fixed butterfly (the same bits on every
// run), plus the bias.
__device__ __forceinline__ void router_logits(const uint8_t* wsm, uint16_t* xsm, const uint16_t* bias,
                                              const uint16_t* x, const uint16_t* resid, int H, int E, int M, int b,
                                              int G, int m0, int lane, float* rlog)
{
#pragma unroll 1
    for (int m = m0; m < M; m += 3) {
        {
            uint4 rowv[kRowVec];
            load_row((x ? x : resid) + (size_t)m * H, H, lane, rowv);
            float inv = 1.f;
            if (!x) {
                uint32_t ab;
                inv = row_stats(rowv, H, true, ab);
            }
#pragma unroll
            for (int z = 0; z < kRowVec; ++z) {
                const int i = lane + 32 * z;
                if (i < H / 8) {
                    uint4 u = rowv[z];
                    if (!x) {
                        uint32_t* w = &u.x;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t lo = f2bf16_rne(__uint_as_float(w[c] << 16) * inv);
                            const uint32_t hi = f2bf16_rne(__uint_as_float(w[c] & 0xffff0000u) * inv);
                            w[c] = lo | (hi << 16);
                        }
                    }
                    reinterpret_cast<uint4*>(xsm)[i] = u;
                }
            }
        }
        __syncwarp();
#pragma unroll 1
        for (int e = b, r = 0; e < E; e += G, ++r) {
            const uint4* wv = reinterpret_cast<const uint4*>(wsm + (size_t)r * H * 2);
            float acc = 0.f;
#pragma unroll 1
            for (int i = lane; i < H / 8; i += 32) {
                const uint4 x4 = reinterpret_cast<const uint4*>(xsm)[i], w4 = wv[i];
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
                rlog[m * E + e] = acc + bf16f(__ldg(bias + e));
        }
        __syncwarp();
    }
}

// The residual buffer of call c: resid + (c / resid_every) * resid_stride
// (kept in shared memory for the call, so the per-use path has no division).
__device__ __forceinline__ uint16_t* call_resid(const DecodeTcParams& p, int c)
{
    return reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(p.resid) +
                                       (long long)(c / p.resid_every) * p.resid_stride);
}

// One layer call of a launch for one role group: `group` 0 = the routing,
// producer and MMA-issuer warps (0, 1, 6), 1 = the x-term / epilogue warps
// (2..5), 2 = the combiner warp (7).  Each group runs its own loop over the
// calls, so that only its own values are live across the loop; the end of a
// call (bias / residual prefetch, the grid barriers and the reduction) is
// executed by every thread in each group's loop.
template <int GROUP>
__device__ __forceinline__ void decode_call(const int call)
{
    const DecodeTcParams& p = g_p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x, M = p.M;
    const int nrows = rows_for(M), atom = nrows * 32;
    const int KSH = p.H / 64, CHH = ceil_div(p.H, 128), CHI = ceil_div(p.I, 128);
    const int T1 = p.I / 64, T2 = ceil_div(p.H, kRowTile);   // units per expert, down row tiles
    const int TG = kDnRegion / nrows;                           // down tiles per accumulator region
    const int nblk = p.H / 32, nitems = M * nblk;               // x-term items: (token, 32-element block)
    const int V = M == 1 ? 1 : (M == 2 ? 2 : 4);                // floats per row of a CTA's output copy
    const uint32_t tail_off = ((uint32_t)p.smem_bytes - tail_bytes(p.H, M, atom)) & ~127u;
    const uint32_t ring_cap = tail_off;
    uint8_t* xs = ring + tail_off;                              // x terms of the layer
    uint8_t* hterm = xs + ((xterm_bytes(p.H, atom) + 127) & ~127u);   // [3][kHTerm]
    float4* xch = reinterpret_cast<float4*>(hterm + 3 * kHTerm);       // [2][32]
    float* oacc = reinterpret_cast<float*>(hterm + 3 * kHTerm + 2 * 32 * 16);   // [H][M]
    const uint32_t tmem = sh.tmem_base;
    const int nu_hi = (M * p.k < p.E ? M * p.k : p.E) < kMaxUnits ? (M * p.k < p.E ? M * p.k : p.E) : kMaxUnits;
    // this thread's role state (0 producer, 1 / 2 MMA issuers, 3 epilogue)
    const int ri = warp == 0 ? 0 : (warp == 1 ? 1 : (warp == kMmaWarpB ? 2 : 3));
    RoleState st = sh.role[ri];
    int gbase = sh.gbase, ubase = sh.ubase, npc = sh.npc;
    RingTc& rs = st.rs;
    uint32_t& sc = st.sc;
    uint32_t& rel = st.rel;
    unsigned long long& rel_end = st.rel_end;
    uint32_t& kk = st.kk;
    uint32_t& sfn = st.sfn;
    const int layer = (p.layer0 + call) % p.nlayers;
    // this call's tensors (recomputed where used rather than held in registers)
#define cl_gu (p.gu + (long long)layer * p.layer_stride)
#define cl_dn (p.dn + (long long)layer * p.layer_stride)
#define cl_gub (p.gu_bias ? reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.gu_bias) + \
                                                            (long long)layer * p.bias_stride) : nullptr)
#define cl_dnb (p.dn_bias ? reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.dn_bias) + \
                                                            (long long)layer * p.bias_stride) : nullptr)
#define cl_logits reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(p.logits) + \
                                                 (long long)call * p.logits_stride)
#define cl_x (p.x ? reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.x) + \
                                                      (long long)call * p.x_stride) : nullptr)
#define cl_resid sh.cresid
#define cl_f32 (p.out_f32 ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(p.out_f32) + \
                                                     (long long)call * p.out_f32_stride) : nullptr)

    if (GROUP == 0) {
        const float* lgp = cl_logits;
        if (p.router) {
            // ---- router GEMV: logits of this CTA's experts e = b, b + G, ... for
            // every token (token m on the (m % 3)-th of warps 0, 1, 6), from the
            // layer input the x terms are cut from; the x-term publication carries
            // them to every CTA, and the routing waits for it
            const uint16_t* rw = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.router) +
                                                                   (long long)layer * p.router_stride);
            // the ring is idle until the routing is done: its start holds this CTA's
            // router rows (one bulk copy each), then one x row per warp
            const int nre = b < p.E ? (p.E - 1 - b) / G + 1 : 0;
            if (nre > 0) {
                if (warp == 0 && lane == 0) {
                    mbar_expect_tx(&sh.rbar, (uint32_t)(nre * p.H * 2));
                    for (int r = 0; r < nre; ++r)
                        bulk_copy(ring + (size_t)r * p.H * 2, rw + (size_t)(b + r * G) * p.H, (uint32_t)p.H * 2,
                                  &sh.rbar);
                }
                const int wi = warp == kMmaWarpB ? 2 : warp;
                uint16_t* xsm = reinterpret_cast<uint16_t*>(ring + (size_t)(nre + wi) * p.H * 2);
                mbar_wait(&sh.rbar, call & 1, p.status);
                router_logits(ring, xsm, rw + (size_t)p.E * p.H, cl_x, cl_resid, p.H, p.E, M, b, G, wi, lane, p.rlog);
                fence_proxy_async_smem();   // the ring's next writers are bulk copies
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sh.rlogw);
            mbar_wait(&sh.xready, call & 1, p.status);
            lgp = p.rlog;
        }
        // ---- routing (warps 0, 1, 6): token m on the (m % 3)-th of them, then the
        // distinct experts in ascending order
#pragma unroll 1
        for (int m = warp == kMmaWarpB ? 2 : warp; m < M; m += 3)
            rt::warp_topk_fit(lgp + (size_t)m * p.E, p.E, p.k, sh.sel[m], sh.wt[m]);
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
            if (lane == 0)
                sh.nu = nu;
        }
        route_barrier();
        if (warp == 1) {
            // the routing weights by (expert slot, token): read by SwiGLU and the
            // output's bias terms only, so off the producer's path
            const int nu = sh.nu;
            for (int x = lane; x < nu * kMaxTokens; x += 32)
                sh.wslot[x / kMaxTokens][x % kMaxTokens] = 0.f;
            __syncwarp();
            for (int x = lane; x < kMaxTokens * kMaxTopK; x += 32) {
                const int m = x / kMaxTopK, k2 = x % kMaxTopK;
                if (m < M && k2 < p.k)
                    sh.wslot[sh.unit_of[sh.sel[m][k2]]][m] = sh.wt[m][k2];
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sh.routed);   // hands the routing to the epilogue warps
        }
    } else if (GROUP == 1) {
        // ---- x terms (warps 2..5): items b + G q + 4 G i, token-major (q = warp - 2)
        const int q = warp - 2, te = tid - 64;
        if (b < nitems) {
            int cm = -1;
            float inv = 1.f, tmax = 0.f;
            uint4 rowv[kRowVec];
            for (int it = b + G * q; it < nitems; it += 4 * G) {
                const int m = it / nblk, kb = it - m * nblk;
                const uint16_t* row = (cl_x ? cl_x : cl_resid) + (size_t)m * p.H;
                if (!cl_x && m != cm) {
                    // the normalised residual: the token's whole row for its rms (and
                    // its largest |x|: the rounding is monotone, so bf16(max|r| inv))
                    load_row(row, p.H, lane, rowv);
                    uint32_t ab;
                    inv = row_stats(rowv, p.H, true, ab);
                    tmax = bf16f(f2bf16_rne(bf16f((uint16_t)ab) * inv));
                    cm = m;
                }
                const uint16_t raw = cl_x ? __ldcg(row + 32 * kb + lane) : row_elem(rowv, kb, lane);
                float v = cl_x ? bf16f(raw) : bf16f(f2bf16_rne(bf16f(raw) * inv));
                // the token's shift S: 0 when this block's largest |x| is at least
                // 2^-98 (then so is the token's), else from the token's largest |x|
                // (the whole row); every builder of token m finds the same S
                int S = 0;
                if (__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))) < (29u << 23)) {
                    if (cl_x) {
                        uint32_t ab;
                        load_row(row, p.H, lane, rowv);
                        row_stats(rowv, p.H, false, ab);
                        tmax = bf16f((uint16_t)ab);
                    }
                    S = token_shift(tmax);
                }
                if (lane == 0)   // 2^-S of token m
                    reinterpret_cast<float*>(p.xt + (long long)KSH * atom + CHH * kSfChunk)[m] =
                        __uint_as_float((uint32_t)(127 - S) << 23);
                v *= __uint_as_float((uint32_t)(127 + S) << 23);
                float r4[kMaxTokens] = {v, 0.f, 0.f, 0.f};
                warp_terms_rows<1>(r4, m, kb, p.xt, p.xt + (long long)KSH * atom, atom, lane);
            }
        }
        epi_barrier();
        if (te == 0) {
            // publish this CTA's x terms (every CTA counts itself in), then wait for
            // the whole count and hand it to the producer through an mbarrier, so the
            // producer never waits on a load
            // (the first call of the launch learns where the count stands; later
            // calls add without waiting for the old value)
            unsigned long long tgt;
            if (p.router)
                mbar_wait(&sh.rlogw, call & 1, p.status);   // this CTA's logits are stored
            if (call == 0) {
                const unsigned long long old = atom_add_release_u64(p.xcnt, 1ull);
                tgt = count_target(old, G);
                sh.epoch = (unsigned)(old / (unsigned long long)G) + 1u;
            } else {
                red_add_release_u64(p.xcnt, 1ull);
                tgt = sh.xtgt + (unsigned long long)G;
                sh.epoch += 1u;
            }
            sh.xtgt = tgt;
            int spins = 0;
#pragma unroll 1
            while (ld_acquire_u64(p.xcnt) < tgt) {
                if (++spins > p.spin_limit) {
                    atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                    break;
                }
            }
            if (p.router)
                mbar_arrive(&sh.xready);   // every CTA's logits are visible: the routing may read them
            // the whole layer's x terms into shared memory, once
            asm volatile("fence.proxy.async.global;" ::: "memory");   // published x terms -> bulk reads
            const uint32_t ab = (uint32_t)KSH * atom, sb = (uint32_t)CHH * kSfChunk;
            mbar_expect_tx(&sh.xfull, ab + sb + 16);
            bulk_copy(xs, p.xt, ab, &sh.xfull);
            bulk_copy(xs + ab, p.xt + (size_t)KSH * atom, sb + 16, &sh.xfull);
        }
        __syncwarp();   // lane 0 rejoins before the warp's collective instructions
        for (int i = te; i < p.H * M; i += kEpi)
            oacc[i] = 0.f;
        // h'-term rows past M * 8 feed MMA columns nobody reads: give them zero
        // codes and unit-range scales rather than whatever shared memory held
        for (int i = te; i < 3 * kHTerm / 4; i += kEpi)
            reinterpret_cast<uint32_t*>(hterm)[i] = 0u;
        mbar_wait(&sh.routed, call & 1, p.status);
    } else {
        mbar_wait(&sh.routed, call & 1, p.status);
    }

    const int nu = sh.nu;
    const int U = nu * T1;
    // (products below stay under 2^31: U <= kMaxUnits * kMaxK / 64, G and H small)
    mbar_wait(&sh.planbar, 0, p.status);
    const Plan pl = nu - p.k >= 0 && nu - p.k < kPlanTab && nu <= nu_hi ? unpack_plan(sh.plan_tab[nu - p.k])
                                                                        : make_plan(b, G, U, KSH, CHH, T2);
    const int u0 = pl.u0, nun = pl.nun, nitem = pl.nitem;
    const int nact = U < G ? U : G;   // CTAs with units
    if (b == 0 && tid == 0 && p.nu_out)
        p.nu_out[layer] = nu;

    if (GROUP == 0 && warp == 0) {
        // ================================================================ producer
        // Weights stream in item order: every stage is weights only (the x terms
        // and the h' terms are in shared memory), so ring space is all a stage
        // waits for -- but the call's third stage, which also waits for the x terms.
        // The x-term exchange (global stores, a grid count, a bulk copy back) runs
        // while the stream starts, and the first MMA needs its result: only the
        // first 2 stages go out before this CTA holds the call's x terms, so that
        // the exchange does not queue behind the whole ring's weight reads (1, 2
        // and 3 such stages measured 23.7, 23.0 and 23.4 us a layer, no limit 24.0).
        const uint64_t wpol = l2_evict_first();
        uint32_t xwait = 2u;
        // the whole warp: claim ring bytes and a slot for a stage (stages retire in order)
        auto claim = [&](uint32_t size, uint32_t& off) -> uint32_t {
            if (xwait == 0u) {
                mbar_wait(&sh.xfull, call & 1, p.status);
                xwait = 0xffffffffu;
            } else if (xwait != 0xffffffffu) {
                --xwait;
            }
            unsigned long long end;
            off = rs.place(size, ring_cap, &end);
            int spins = 0;
#pragma unroll 1
            while (rel < sc && (end - rel_end > (unsigned long long)ring_cap || rel + kSlots <= sc)) {
                const uint32_t sl = rel % kSlots;
                if (__shfl_sync(0xffffffffu, mbar_test_wait(&sh.empty[sl], (rel / kSlots) & 1) ? 1 : 0, 0)) {
                    rel_end = sh.ends[sl];
                    ++rel;
                } else {
                    if (++spins > (1 << 24)) {
                        if (lane == 0)
                            atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                        break;
                    }
                }
            }
            const uint32_t slot = sc % kSlots;
            __syncwarp();
            if (lane == 0)
                sh.ends[slot] = end;
            __syncwarp();
            return slot;
        };
        for (int k = 0; k < nitem; ++k) {
            int kind, i;
            item_of(pl, k, kind, i);
            const bool piece = kind >= kGuPiece;
            const int unit = piece ? pl.su : u0 + i, s = unit / T1, t = unit % T1;
            const int e = sh.unit_expert[s];
            if (kind == kGu || kind == kGuPiece) {
                const int kA = piece ? pl.ks0 : 0, kB = piece ? pl.ks1 : KSH;
                const uint8_t* a0 = cl_gu + (long long)e * p.gu_expert + (long long)t * kRowTile * (p.H / 2);
                const uint8_t* s0 = cl_gu + (long long)e * p.gu_expert + (long long)(2 * p.I) * (p.H / 2) +
                                    (long long)t * CHH * kSfChunk;
                for (int ks = kA; ks < kB; ks += kGuSteps, ++sc) {
                    const int steps = kB - ks < kGuSteps ? kB - ks : kGuSteps;
                    const GuStage sg(steps);
                    uint32_t off;
                    const uint32_t slot = claim(sg.size, off);
                    if (lane == 0)
                        mbar_expect_tx(&sh.full[slot], sg.abytes + sg.sfbytes);
                    __syncwarp();
                    uint8_t* st = ring + off;
                    if (lane == 0)   // weights: read once per call
                        bulk_copy_hint(st, a0 + (long long)ks * kTileA, sg.abytes, &sh.full[slot], wpol);
                    else if (lane == 1)
                        bulk_copy_hint(st + sg.sfa, s0 + (ks >> 1) * kSfChunk, sg.sfbytes, &sh.full[slot], wpol);
                }
            } else {
                // down rows of tiles [tA, tB), k-step t of K = I (h rows 64t .. 64t+63):
                // in the k-step-major order the tiles of a stage are one run of
                // codes and one run of scale chunks
                const int tA = piece ? pl.ta : 0, tB = piece ? pl.tb : T2;
                const uint8_t* c0 = cl_dn + (long long)e * p.dn_expert + (long long)t * p.H * 32;
                const uint8_t* sc0 = cl_dn + (long long)e * p.dn_expert + (long long)p.H * (p.I / 2) +
                                     (long long)(t >> 1) * T2 * kSfChunk;
                for (int ga = tA; ga < tB; ga += TG) {
                    const int gb = ga + TG < tB ? ga + TG : tB;
                    for (int t2 = ga; t2 < gb; t2 += kDnStageTiles, ++sc) {
                        const int n = gb - t2 < kDnStageTiles ? gb - t2 : kDnStageTiles;
                        const int rows = p.H - t2 * kRowTile < n * kRowTile ? p.H - t2 * kRowTile : n * kRowTile;
                        uint32_t off;
                        const uint32_t slot = claim(dn_stage_size(n), off);
                        if (lane == 0)
                            mbar_expect_tx(&sh.full[slot], (uint32_t)rows * 32 + (uint32_t)n * kSfChunk);
                        __syncwarp();
                        uint8_t* st = ring + off;
                        if (lane == 0)
                            bulk_copy_hint(st, c0 + (long long)t2 * kRowTile * 32, (uint32_t)rows * 32, &sh.full[slot],
                                           wpol);
                        else if (lane == 1)
                            bulk_copy_hint(st + n * kTileA, sc0 + (long long)t2 * kSfChunk, (uint32_t)n * kSfChunk,
                                           &sh.full[slot], wpol);
                    }
                }
            }
        }
    } else if (GROUP == 0) {
        // ================================================================ MMA issuers
        // Issuing a tcgen05 instruction holds its thread ~75-95 cycles (a scale
        // copy as long as an MMA), while the pipe takes one every ~40 cycles from
        // two threads.  So every stage is split between issuer A (warp 1) and B
        // (warp 6): A takes the first half of its scale chunks (gate/up k-step
        // pairs) or down tiles, B the rest, each with its own scale sets and
        // accumulator half / tiles, and both release the stage.  A stage is then
        // consumed in half the time, which is ring space handed back to the
        // weight stream sooner.
        const int role = warp == 1 ? 0 : 1;
        if (lane == 0) {
            const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(nrows >> 3) << 17) | (1u << 23) |
                                   ((uint32_t)(kRowTile >> 4) << 24);
            const uint32_t myset = tmem + kSfCol + role * 2 * kSfSet;
            for (int k = 0; k < nitem; ++k) {
                int kind, i;
                item_of(pl, k, kind, i);
                const bool piece = kind >= kGuPiece;
                const int t = (piece ? pl.su : u0 + i) % T1;
                if (kind == kGu || kind == kGuPiece) {
                    const int gl = piece ? 0 : i + pl.piece;   // gate/up accumulator use in this call
                    const int gi = gbase + gl;                  // ... and since the launch
                    const int kA = piece ? pl.ks0 : 0, kB = piece ? pl.ks1 : KSH;
                    // each issuer adds its half of every stage into its own accumulator half
                    const uint32_t buf = gi & 1;
                    if (gl == 0)
                        mbar_wait(&sh.xfull, call & 1, p.status);   // the call's x terms are in
                    if (gi >= 2)
                        mbar_wait(&sh.acce[buf], ((gi >> 1) - 1) & 1, p.status);
                    tc_fence_after();
                    const uint32_t d = tmem + kGuCol + buf * kGuBuf + role * 32;
                    bool first = true;
                    for (int ks = kA; ks < kB; ks += kGuSteps, ++sc) {
                        const int steps = kB - ks < kGuSteps ? kB - ks : kGuSteps;
                        const GuStage sg(steps);
                        unsigned long long end;
                        const uint32_t st = su32(ring) + rs.place(sg.size, ring_cap, &end);
                        // this issuer's scale chunks [c0, c1) = k-steps [2 c0, min(2 c1, steps))
                        const int chunks = (steps + 1) >> 1, half = (chunks + 1) >> 1;
                        const int c0 = role ? half : 0, c1 = role ? chunks : half;
                        const uint32_t slot = sc % kSlots;
                        if (c0 < c1) {
                            mbar_wait(&sh.full[slot], (sc / kSlots) & 1, p.status);
                            tc_fence_after();
                            const uint32_t set = myset + (sfn++ & 1) * kSfSet;
                            const uint32_t xsf = su32(xs) + KSH * atom + (ks >> 1) * kSfChunk;   // x-term scales
                            // (the hot loop: unrolled, descriptors stepped by adding the byte
                            // offset / 16 to the start-address field)
#pragma unroll
                            for (int ch = 0; ch < (kGuSteps + 3) / 4; ++ch)
                                if (c0 + ch < c1) {
                                    tc_cp_sf(set + 4 * ch, st + sg.sfa + (c0 + ch) * kSfChunk);
                                    tc_cp_sf(set + kSfSet / 2 + 4 * ch, xsf + (c0 + ch) * kSfChunk);
                                }
                            const int j0 = 2 * c0, nj = (2 * c1 < steps ? 2 * c1 : steps) - j0;
                            const uint64_t da = smem_desc(st + j0 * kTileA, 128, 256);
                            const uint64_t db = smem_desc(su32(xs) + (ks + j0) * atom, 128, 256);   // B: x terms
                            const uint32_t id_odd = (2u << 4) | (2u << 29);
#pragma unroll
                            for (int j = 0; j < (kGuSteps + 1) / 2; ++j)
                                if (j < nj) {
                                    tc_mma_mxf4(d, da + (uint64_t)(j * (kTileA >> 4)), db + (uint64_t)(j * (atom >> 4)),
                                                idesc | ((j & 1) ? id_odd : 0u), set + 4 * (j >> 1),
                                                set + kSfSet / 2 + 4 * (j >> 1), (first && j == 0) ? 0u : 1u);
                                }
                            first = false;
                        }
                        tc_commit(&sh.empty[slot]);
                    }
                    tc_commit(&sh.accf[buf]);   // both issuers
                } else {
                    uint32_t hb;
                    if (piece) {
                        hb = su32(hterm + 2 * kHTerm);
                        mbar_wait(&sh.hsfull, npc & 1, p.status);
                    } else {
                        const int ui = ubase + i;
                        hb = su32(hterm + (ui & 1) * kHTerm);
                        mbar_wait(&sh.hbar[ui & 1], (ui >> 1) & 1, p.status);
                    }
                    tc_fence_after();
                    // the unit's h' scale chunk, copied once for all its down tiles into
                    // columns no stage set uses (24..31 of set 0: the two h' buffers,
                    // 24..27 of set 1: the split unit's)
                    const uint32_t hsf = myset + (piece ? (uint32_t)kSfSet + 24u : 24u + 4u * ((ubase + i) & 1));
                    tc_cp_sf(hsf, hb + 1024);
                    const uint32_t aid = (uint32_t)(2 * (t & 1));   // A scale bytes of k-step t in its chunk
                    const int tA = piece ? pl.ta : 0, tB = piece ? pl.tb : T2;
                    for (int ga = tA; ga < tB; ga += TG, ++kk) {
                        const int gb = ga + TG < tB ? ga + TG : tB;
                        if (kk >= 2)
                            mbar_wait(&sh.dne[kk & 1], ((kk >> 1) - 1) & 1, p.status);
                        tc_fence_after();
                        const uint32_t dreg = tmem + kDnCol + (kk & 1) * kDnRegion;
                        for (int t2 = ga; t2 < gb; t2 += kDnStageTiles, ++sc) {
                            const int n = gb - t2 < kDnStageTiles ? gb - t2 : kDnStageTiles;
                            unsigned long long end;
                            const uint32_t st = su32(ring) + rs.place(dn_stage_size(n), ring_cap, &end);
                            // this issuer's tiles [j0, j1) of the stage
                            const int hn = (n + 1) >> 1, j0 = role ? hn : 0, j1 = role ? n : hn;
                            const uint32_t slot = sc % kSlots;
                            if (j0 < j1) {
                                mbar_wait(&sh.full[slot], (sc / kSlots) & 1, p.status);
                                tc_fence_after();
                                const uint32_t set = myset + (sfn++ & 1) * kSfSet;
#pragma unroll
                                for (int j = 0; j < (kDnStageTiles + 1) / 2; ++j)
                                    if (j0 + j < j1)
                                        tc_cp_sf(set + 4 * j, st + n * kTileA + (j0 + j) * kSfChunk);
                                const uint64_t da = smem_desc(st + j0 * kTileA, 128, 256), db = smem_desc(hb, 128, 256);
                                const uint32_t dcol = dreg + (t2 - ga + j0) * nrows;
#pragma unroll
                                for (int j = 0; j < (kDnStageTiles + 1) / 2; ++j)
                                    if (j0 + j < j1)
                                        tc_mma_mxf4(dcol + j * nrows, da + (uint64_t)(j * (kTileA >> 4)), db,
                                                    idesc | (aid << 29), set + 4 * j, hsf, 0u);
                            }
                            tc_commit(&sh.empty[slot]);
                        }
                        tc_commit(&sh.dnf[kk & 1]);   // both issuers: the group's region is full
                    }
                }
            }
        }
    } else if (GROUP == 2) {
        // ================================================================ combiner
        if (pl.piece) {
            // the split unit's h' for this CTA's down tiles: wait for every piece's
            // partial sums (one flag per lane), add them in piece order, SwiGLU,
            // MX terms (lane = h row within each of the two 32-row blocks)
            const int s = pl.su / T1, t = pl.su % T1, e = sh.unit_expert[s];
            // the biases first: HBM is busy with the weight stream, so their
            // latency overlaps the wait for the other pieces
            float bg[2] = {0.f, 0.f}, bu[2] = {0.f, 0.f};
            if (cl_gub)
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    const int hrow = 64 * t + 32 * kb + lane;
                    bg[kb] = bf16f(__ldg(cl_gub + (size_t)e * 2 * p.I + hrow));
                    bu[kb] = bf16f(__ldg(cl_gub + (size_t)e * 2 * p.I + p.I + hrow));
                }
            mbar_wait(&sh.xfull, call & 1, p.status);   // (orders the call tag written before it)
            const unsigned tag = sh.epoch;
            const int b0 = pl.sj * pl.S;   // the CTA of piece 0
            int spins = 0;
            bool all = false;
#pragma unroll 1
            while (!all && ++spins < p.spin_limit)
                all = __all_sync(0xffffffffu, lane >= pl.S || ld_acquire_u32(p.pflag + b0 + lane) == tag);
            if (!all && lane == 0)
                atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
            // gate (rows r) and up (rows 64 + r) sums of both 32-row blocks, every
            // piece's loads in flight together, added in piece order
            float g[2][kMaxTokens] = {}, u[2][kMaxTokens] = {};
            if (M == 1) {
                // token 0 only: one scalar per (piece, block, gate / up), eight pieces'
                // loads in flight together (one round trip for the usual S <= 8)
                for (int p0 = 0; p0 < pl.S; p0 += 8) {
                    float v[8][4];
#pragma unroll
                    for (int z = 0; z < 8; ++z)
                        if (p0 + z < pl.S) {
                            const float* src = p.gpart + (size_t)(b0 + p0 + z) * kRowTile * 4;
#pragma unroll
                            for (int kb = 0; kb < 2; ++kb) {
                                v[z][2 * kb] = __ldcg(src + (32 * kb + lane) * 4);
                                v[z][2 * kb + 1] = __ldcg(src + (64 + 32 * kb + lane) * 4);
                            }
                        }
#pragma unroll
                    for (int z = 0; z < 8; ++z)
                        if (p0 + z < pl.S)
#pragma unroll
                            for (int kb = 0; kb < 2; ++kb) {
                                g[kb][0] += v[z][2 * kb];
                                u[kb][0] += v[z][2 * kb + 1];
                            }
                }
            }
            for (int p0 = 0; M > 1 && p0 < pl.S; p0 += 4) {
                float4 v[4][4];
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    if (p0 + z < pl.S) {
                        const float4* src = reinterpret_cast<const float4*>(p.gpart) + (size_t)(b0 + p0 + z) * kRowTile;
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb) {
                            v[z][2 * kb] = __ldcg(src + 32 * kb + lane);
                            v[z][2 * kb + 1] = __ldcg(src + 64 + 32 * kb + lane);
                        }
                    }
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    if (p0 + z < pl.S)
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb) {
                            const float4 gv = v[z][2 * kb], uv = v[z][2 * kb + 1];
                            g[kb][0] += gv.x; g[kb][1] += gv.y; g[kb][2] += gv.z; g[kb][3] += gv.w;
                            u[kb][0] += uv.x; u[kb][1] += uv.y; u[kb][2] += uv.z; u[kb][3] += uv.w;
                        }
            }
            uint8_t* hb = hterm + 2 * kHTerm;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                float hv[kMaxTokens];
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m) {
                    // a token that did not choose this expert gets exactly 0 (its sums may
                    // even be infinite: the expert's weights were applied to every column)
                    const float gg = g[kb][m] + bg[kb], wt = sh.wslot[s][m];
                    hv[m] = m < M && wt != 0.f ? wt * swiglu(gg, u[kb][m] + bu[kb], p.sw_alpha, p.sw_limit, p.sw_beta)
                                               : 0.f;
                }
                switch (M) {
                case 1: warp_terms_rows<1>(hv, 0, kb, hb, hb + 1024, atom, lane); break;
                case 2: warp_terms_rows<2>(hv, 0, kb, hb, hb + 1024, atom, lane); break;
                case 3: warp_terms_rows<3>(hv, 0, kb, hb, hb + 1024, atom, lane); break;
                default: warp_terms_rows<4>(hv, 0, kb, hb, hb + 1024, atom, lane); break;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sh.hsfull);
        }

    } else {
        // ================================================================ epilogue warps
        const int te = tid - 64, q = warp & 3;   // q: the lane quarter this warp may read
        // SwiGLU of 64 h rows from the gate sums (lane quarters 0, 1) and up sums
        // (2, 3) of token m, times the routing weight, into MX terms at dst: the up
        // sums go through shared memory, then warps q < 2 each write one
        // 32-element block (k-block q of the down k-step)
        auto swiglu_terms = [&](const float (&sm)[kMaxTokens], int s, float bg, float bu, uint8_t* dst) {
            if (q >= 2)
                xch[(q - 2) * 32 + lane] = make_float4(sm[0], sm[1], sm[2], sm[3]);
            epi_barrier();
            if (q < 2) {
                const float4 u4 = xch[q * 32 + lane];
                const float us[kMaxTokens] = {u4.x, u4.y, u4.z, u4.w};
                float hv[kMaxTokens];
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m) {
                    // 0 for a token that did not choose this expert, whatever its sums
                    const float g = sm[m] + bg, wt = sh.wslot[s][m];
                    hv[m] = m < M && wt != 0.f ? wt * swiglu(g, us[m] + bu, p.sw_alpha, p.sw_limit, p.sw_beta) : 0.f;
                }
                switch (M) {   // one copy of the code runs
                case 1: warp_terms_rows<1>(hv, 0, q, dst, dst + 1024, atom, lane); break;
                case 2: warp_terms_rows<2>(hv, 0, q, dst, dst + 1024, atom, lane); break;
                case 3: warp_terms_rows<3>(hv, 0, q, dst, dst + 1024, atom, lane); break;
                default: warp_terms_rows<4>(hv, 0, q, dst, dst + 1024, atom, lane); break;
                }
            }
        };
        // 2^-S_m of each token: the gate/up sums carry the x terms' shift
        float ush[kMaxTokens] = {1.f, 1.f, 1.f, 1.f};
        if (nitem > 0) {
            mbar_wait(&sh.xfull, call & 1, p.status);
#pragma unroll
            for (int m = 0; m < kMaxTokens; ++m)
                if (m < M)
                    ush[m] = reinterpret_cast<const float*>(xs + KSH * atom + CHH * kSfChunk)[m];
        }
        for (int k = 0; k < nitem; ++k) {
            int kind, i;
            item_of(pl, k, kind, i);
            const bool piece = kind >= kGuPiece;
            const int unit = piece ? pl.su : u0 + i, s = unit / T1, t = unit % T1;
            if (kind == kGu || kind == kGuPiece) {
                // ---- gate (rows 0..63) and up (rows 64..127) sums of 64 h rows; the
                // biases are loaded before the accumulator is waited for
                const int gi = gbase + (piece ? 0 : i + pl.piece);   // gate/up accumulator use since the launch
                const uint32_t buf = gi & 1;
                const int hrow = 64 * t + 32 * (q & 1) + lane;
                const int e = sh.unit_expert[s];
                float bg = 0.f, bu = 0.f;
                if (q < 2 && cl_gub) {
                    bg = bf16f(__ldg(cl_gub + (size_t)e * 2 * p.I + hrow));
                    bu = bf16f(__ldg(cl_gub + (size_t)e * 2 * p.I + p.I + hrow));
                }
                mbar_wait(&sh.accf[buf], (gi >> 1) & 1, p.status);
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + kGuCol + buf * kGuBuf;
                const int kA = piece ? pl.ks0 : 0, kB = piece ? pl.ks1 : KSH;
                const bool two = kB - kA >= 3;   // issuer B wrote its half too (some stage has 2+ chunks)
                float sm[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
                float d0[2][16], d1[2][16];   // both halves' loads in flight before one wait
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (16 * h < nrows) {
                        tc_ld16(taddr + 16 * h, d0[h]);
                        if (two)
                            tc_ld16(taddr + 32 + 16 * h, d1[h]);
                    }
                }
                tc_wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (16 * h < nrows) {
#pragma unroll
                        for (int col = 0; col < 16; ++col) {
                            const int m = (16 * h + col) / kTerms;   // compile-time after unrolling
                            if (m < M)
                                sm[m] += two ? d0[h][col] + d1[h][col] : d0[h][col];
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m)
                    sm[m] *= ush[m];
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sh.acce[buf]);
                if (!piece) {
                    const int ui = ubase + i;
                    uint8_t* hb = hterm + (ui & 1) * kHTerm;
                    swiglu_terms(sm, s, bg, bu, hb);
                    if (q < 2)
                        fence_proxy_async_smem();
                    epi_barrier();
                    if (te == 0)
                        mbar_arrive(&sh.hbar[ui & 1]);
                    continue;
                }
                // ---- a piece of a split unit: publish its partial sums (warp 7
                // combines them)
                float4* gp = reinterpret_cast<float4*>(p.gpart) + (size_t)b * kRowTile;
                gp[32 * q + lane] = make_float4(sm[0], sm[1], sm[2], sm[3]);
                epi_barrier();
                if (te == 0)
                    st_release_u32(p.pflag + b, sh.epoch);
            } else {
                // ---- down products of tiles [tA, tB) into the CTA's output copy
                const int tA = piece ? pl.ta : 0, tB = piece ? pl.tb : T2;
                for (int ga = tA; ga < tB; ga += TG, ++kk) {
                    const int gb = ga + TG < tB ? ga + TG : tB;
                    mbar_wait(&sh.dnf[kk & 1], (kk >> 1) & 1, p.status);
                    tc_fence_after();
                    const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + kDnCol + (kk & 1) * kDnRegion;
                    const int row0 = ga * kRowTile + 32 * q + lane;
                    if (M == 1)
                        drain_region<8, 8>(taddr, gb - ga, nrows, row0, oacc, p.H, M);
                    else if (M == 2)
                        drain_region<16, 4>(taddr, gb - ga, nrows, row0, oacc, p.H, M);
                    else
                        drain_region<32, 4>(taddr, gb - ga, nrows, row0, oacc, p.H, M);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sh.dne[kk & 1]);
                }
            }
        }
        // ---- the CTA's output copy to its partial slot [H][V] (rows drained by other warps)
        epi_barrier();
        if (nun > 0 && M != 3) {
            // [H][M] and [H][V] coincide: a straight float4 copy
            const float4* src4 = reinterpret_cast<const float4*>(oacc);
            float4* dst4 = reinterpret_cast<float4*>(p.part + (size_t)b * p.H * V);
            const int n4 = p.H * M / 4;
#pragma unroll 4
            for (int i = te; i < n4; i += kEpi)
                dst4[i] = src4[i];
        } else if (nun > 0) {
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

    // ---- this CTA's slice of the output: float4s [f0, f1) of a copy [H][V] (4 / V
    // rows x V tokens each); the residual and the bias terms sum_s w_s b_s of its
    // elements are loaded before the grid barrier
    const int U4 = p.H * V / 4;
    const int f0 = (int)((unsigned)b * U4 / G), f1 = (int)((unsigned)(b + 1) * U4 / G), nf = f1 - f0;
    // r + sum_s w_s b_s of element z of the slice's float4 j
    auto fin_term = [&](int j, int z) -> float {
        const int el = (f0 + j) * 4 + z, row = el / V, m = el - row * V;
        float v = 0.f;
        if (m < M) {
            if (cl_dnb)
                for (int s2 = 0; s2 < nu; ++s2)
                    v = fmaf(sh.wslot[s2][m], bf16f(__ldg(cl_dnb + (size_t)sh.unit_expert[s2] * p.H + row)), v);
            v += bf16f(__ldcg(cl_resid + (size_t)m * p.H + row));
        }
        return v;
    };
    if (tid < nf && tid < kFinSlots) {
        mbar_wait(&sh.routed, call & 1, p.status);   // the weight slots (warp 1 writes them)
#pragma unroll
        for (int z = 0; z < 4; ++z)
            sh.fin[tid][z] = fin_term(tid, z);
    }

    // ---- grid barrier: every CTA's output copy is stored (every CTA counts itself in).
    // The CTA's copy of the x terms has landed before it arrives (a CTA without
    // units never waits for it otherwise, and the next call rewrites them).
    if (tid == 64)
        mbar_wait(&sh.xfull, call & 1, p.status);
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        // (a debug run may have one CTA skip its arrival, to test that the others give up)
        unsigned long long tgt;
        if (call == 0) {
            tgt = count_target(b == p.skip_cta ? ld_acquire_u64(p.done) : atom_add_release_u64(p.done, 1ull), G);
        } else {
            if (b != p.skip_cta)
                red_add_release_u64(p.done, 1ull);
            tgt = sh.dtgt + (unsigned long long)G;
        }
        sh.dtgt = tgt;
        int spins = 0;
#pragma unroll 1
        while (ld_acquire_u64(p.done) < tgt) {
            if (++spins > p.spin_limit) {
                atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                break;
            }
        }
    }
    __syncthreads();

    // ---- the slice: float4 j of it summed over the active CTAs' copies by warp
    // j mod 8 -- lane l takes CTAs l, l + 32, ... (all its loads in flight at
    // once), then a fixed shuffle tree -- so the order never depends on timing
    {
        auto cta_of = [&](int cc) { return U < G ? (int)(((unsigned)(cc + 1) * G + U - 1) / U) - 1 : cc; };
        const float4* part = reinterpret_cast<const float4*>(p.part);
        for (int j = warp; j < nf; j += kThreadsTc / 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = lane; c0 < nact; c0 += 8 * 32) {
                float4 a[8];
#pragma unroll
                for (int z = 0; z < 8; ++z)
                    if (c0 + 32 * z < nact)
                        a[z] = __ldcg(part + (size_t)cta_of(c0 + 32 * z) * U4 + f0 + j);
#pragma unroll
                for (int z = 0; z < 8; ++z)
                    if (c0 + 32 * z < nact) {
                        acc.x += a[z].x; acc.y += a[z].y; acc.z += a[z].z; acc.w += a[z].w;
                    }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
                acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
                acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
                acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
            }
            // lane z < 4 writes element z of the float4 (its residual and bias terms
            // were loaded by thread j before the barrier: handed over by shuffle)
            const float sums[4] = {acc.x, acc.y, acc.z, acc.w};
            float mine = 0.f;
#pragma unroll
            for (int z = 0; z < 4; ++z)
                if (lane == z)
                    mine = sums[z];
            if (lane < 4) {
                const int el = (f0 + j) * 4 + lane, row = el / V, m = el - row * V;
                if (m < M) {
                    const float v = (j < kFinSlots ? sh.fin[j][lane] : fin_term(j, lane)) + mine;
                    cl_resid[(size_t)m * p.H + row] = f2bf16_rne(v);
                    if (cl_f32)
                        cl_f32[(size_t)m * p.H + row] = v;
                }
            }
        }
    }

    // ---- end of the call: the role states go back to shared memory, and the next
    // call reads its routing and inputs only after every CTA's slice of this
    // output is written
    if (call + 1 < p.ncalls) {
        if (ri == 0) {
            // every stage of this call has been consumed (its MMAs completed before
            // the epilogue's last drain): the producer need not poll their releases
            st.rel = st.sc;
            st.rel_end = st.rs.head;
        }
        if ((ri == 0 && lane == 0) || ((ri == 1 || ri == 2) && lane == 0) || (ri == 3 && tid == 64))
            sh.role[ri] = st;
        if (tid == 0) {
            sh.gbase = gbase + nun + pl.piece;
            sh.ubase = ubase + nun;
            sh.npc = npc + pl.piece;
        }
        __syncthreads();
        if (tid == 0) {
            sh.cresid = call_resid(p, call + 1);   // every thread is past this call's last use
            red_add_release_u64(p.done, 1ull);
            sh.dtgt += (unsigned long long)G;
            wait_count(p.done, sh.dtgt, p.spin_limit, p.status);
        }
        __syncthreads();
    }
#undef cl_gu
#undef cl_dn
#undef cl_gub
#undef cl_dnb
#undef cl_logits
#undef cl_x
#undef cl_resid
#undef cl_f32
}

__global__ void __launch_bounds__(kThreadsTc, 1) decode_tc_kernel(const DecodeTcParams p)
{
    // the next layer's CTAs may take each SM as soon as this CTA leaves it
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x, M = p.M;
    const int nrows = rows_for(M), atom = nrows * 32;
    const int KSH = p.H / 64, CHH = ceil_div(p.H, 128), CHI = ceil_div(p.I, 128);
    const int T1 = p.I / 64, T2 = ceil_div(p.H, kRowTile);   // units per expert, down row tiles
    const int TG = kDnRegion / nrows;                           // down tiles per accumulator region
    const int nblk = p.H / 32, nitems = M * nblk;               // x-term items: (token, 32-element block)
    const int V = M == 1 ? 1 : (M == 2 ? 2 : 4);                // floats per row of a CTA's output copy
    const uint32_t tail_off = ((uint32_t)p.smem_bytes - tail_bytes(p.H, M, atom)) & ~127u;
    const uint32_t ring_cap = tail_off;
    uint8_t* xs = ring + tail_off;                              // x terms of the layer
    uint8_t* hterm = xs + ((xterm_bytes(p.H, atom) + 127) & ~127u);   // [3][kHTerm]
    float4* xch = reinterpret_cast<float4*>(hterm + 3 * kHTerm);       // [2][32]
    float* oacc = reinterpret_cast<float*>(hterm + 3 * kHTerm + 2 * 32 * 16);   // [H][M]

    // warm L2 and the TLB for what the first steps read once the previous grid
    // is complete (a prefetch returns no data, so it cannot see a stale value)
    if (warp == 2 && lane < M && p.logits)   // (the in-kernel router has no given logits)
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
        g_p = p;   // the calls read the parameters from shared memory
        for (int r = 0; r < 4; ++r)
            sh.role[r] = RoleState{};
        sh.gbase = sh.ubase = sh.npc = 0;
        sh.cresid = call_resid(p, 0);
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 2);   // both MMA issuers release every stage
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.accf[i], 2);
            mbar_init(&sh.acce[i], 4);
            mbar_init(&sh.dnf[i], 2);
            mbar_init(&sh.dne[i], 4);
            mbar_init(&sh.hbar[i], 1);
        }
        mbar_init(&sh.routed, 1);
        mbar_init(&sh.xfull, 1);
        mbar_init(&sh.hsfull, 1);
        mbar_init(&sh.planbar, 1);
        mbar_init(&sh.rlogw, 3);   // warps 0, 1 and 6
        mbar_init(&sh.xready, 1);
        mbar_init(&sh.rbar, 1);
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
    // the plan of every distinct-expert count the call can have (lane i: nu =
    // k + i), from the shapes alone, so before the previous grid is waited for
    const int nu_hi = (M * p.k < p.E ? M * p.k : p.E) < kMaxUnits ? (M * p.k < p.E ? M * p.k : p.E) : kMaxUnits;
    if (warp == kCombineWarp) {
        const int nu = p.k + lane;
        if (lane < kPlanTab && nu <= nu_hi)
            sh.plan_tab[lane] = pack_plan(make_plan(b, G, nu * T1, KSH, CHH, T2));
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sh.planbar);
    }
    // everything below reads what the previous grid in the stream wrote (the
    // logits, x, the residual) or shares its workspace
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp < 2 || warp == kMmaWarpB) {
#pragma unroll 1
        for (int call = 0; call < p.ncalls; ++call)
            decode_call<0>(call);
    } else if (warp <= 5) {
#pragma unroll 1
        for (int call = 0; call < p.ncalls; ++call)
            decode_call<1>(call);
    } else {
#pragma unroll 1
        for (int call = 0; call < p.ncalls; ++call)
            decode_call<2>(call);
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
