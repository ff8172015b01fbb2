// moe_decode_tc.cu -- the MXFP4 decode layer (M <= 4 tokens) on the
// 5th-generation tensor cores: one persistent launch, one CTA per SM.
//
// The layer is the one of "Sovereign gpt-oss-20B (MXFP4) on Apple Silicon",
// section 3 (top-k routing, per selected expert an MXFP4 gate_up GEMV,
// SwiGLU, an MXFP4 down GEMV, the routing-weighted sum into the residual).
// The weights stay 4-bit all the way into the MMA: tcgen05.mma kind::mxf4
// reads E2M1 codes and E8M0 scales from shared / tensor memory, so no
// instruction per weight runs on the CUDA cores.  That instruction wants FP4
// on the activation side too; an activation vector v (x, or h) is therefore
// fed as a sum of T MXFP4 vectors, v ~ v_1 + ... + v_T with
// v_j = MX(v - v_1 - ... - v_{j-1}) (OCP MX v1.0 quantiser), each term one
// column of the MMA's N (token m, term j at column 8m + j; N = 16 for M <= 2,
// else 32).  Each term cuts the residual of a 32-element block by a factor
// of at least 4, so T = 8 terms leave a relative error near 1e-6, like fp32
// activations; a bf16 x is usually exact after fewer terms, and a block
// whose residual is zero gets zero terms without further arithmetic.  The
// MMA applies every term's scales, and the epilogue adds a token's columns.
//
// Work: gate_up units (selected expert s, 128-row tile t of gate and of up, a
// K range of H) and down units (s, 128-row tile of down, a K range of I),
// dealt round-robin over the CTAs; the K split gives every SM work when only
// 4 experts are selected.  A unit's fp32 partial sums go to global memory;
// the last unit of a tile to finish (an atomic counter) adds them in a fixed
// order, so results do not depend on timing.  h of an expert's 128 rows is
// published with a release flag; a down unit waits only for the h rows its
// K range covers, while its weights are already streaming into the ring.
// The last down tile of a 128-row slice of the output to finish, across all
// experts, writes out = bf16(r + sum_s w_s y_s) in each token's choice order.
//
// Warp roles (192 threads): warp 0 streams weight tiles into a byte ring of
// shared memory (each stage's copies issued from separate lanes in one
// instruction); warp 1 owns tensor memory and issues the MMAs from one
// thread; warps 2..5 (one per lane quarter) build the activation terms, drain
// the accumulators and run the cross-CTA reductions.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "moe_internal.h"
#include "route.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kRows = 32;          // activation rows: token m, term j at m * kTerms + j
constexpr int kTerms = 8;          // MX terms per activation vector
constexpr int kAtom = kRows * 32;  // bytes of one k-step of activation terms
constexpr int kSteps = 8;          // k-steps (64 of K) per pipeline stage (the producer's issue cost is per stage)
constexpr int kSlots = 16;         // stages in flight at most
constexpr int kAcc = 2 * kRows;    // accumulator columns of one buffer: gate | up (down: issuer A | B)
constexpr int kSfSetCol = 2 * kAcc;   // per-issuer stage scale sets: 2 issuers x 2 sets
constexpr int kSfSetCols = 32;        // one set: A scales (4 chunks) | B scales (4 chunks)
static_assert(kSfSetCols / 2 >= 4 * ((kSteps + 1) / 2), "scale set holds a stage's chunks");
constexpr int kMmaWarpB = 6;
constexpr int kTmemCols = 512;
static_assert(kSfSetCol + 4 * kSfSetCols <= kTmemCols, "tensor memory");
constexpr int kRingSlack = 4096;   // read slack past the ring (partial row tiles)
constexpr int kThreadsTc = 224;    // producer, MMA issuer A, 4 epilogue warps, MMA issuer B
constexpr int kEpi = 128;          // epilogue threads (warps 2..5)
constexpr int kPend = 16;          // queued h-term copies of the producer

// MMA N: the rows that hold terms, rounded up to 16.
__device__ __forceinline__ int rows_for(int M) { return M * kTerms <= 16 ? 16 : 32; }

struct Geometry {
    int KSH, KSI, CHH, CHI, T1, T2;   // k-steps, 128-element chunks and 128-row tiles of H and I
    int nu, KC1, KC2, U1, U2;
};

// Work units, dealt round-robin over the CTAs from one list: U1 gate/up
// pieces (nu*T1 tile pairs in KC1 K pieces), then U2 down pieces (nu*T2
// tiles in KC2 K pieces).  A CTA's down pieces stream into its ring behind
// its pair, so most down weights are resident when h is ready.
__device__ __forceinline__ Geometry geometry(const DecodeTcParams& p, int nu, int G)
{
    Geometry g;
    g.KSH = p.H / 64;
    g.KSI = p.I / 64;
    g.CHH = ceil_div(p.H, 128);
    g.CHI = ceil_div(p.I, 128);
    g.T1 = ceil_div(p.I, kRowTile);
    g.T2 = ceil_div(p.H, kRowTile);
    g.nu = nu;
    const int pairs = nu * g.T1, tiles = nu * g.T2;
    // Gate/up pairs stay whole (a K split makes h wait for the slowest piece, and
    // measured slower); down tiles split so that the list comes to about two
    // units per CTA.
    g.KC1 = 1;
    const int left = 2 * G - pairs;
    const int k2 = left > 0 ? (left + tiles / 2) / tiles : 1;
    g.KC2 = k2 < 1 ? 1 : (k2 > g.CHI ? g.CHI : k2);
    g.U1 = pairs * g.KC1;
    g.U2 = tiles * g.KC2;
    return g;
}

__device__ __forceinline__ int units_of(const Geometry& g, int b, int G)
{
    const int U = g.U1 + g.U2;
    return U > b ? (U - b + G - 1) / G : 0;
}

struct Unit {
    bool down;
    int s, t;           // expert slot, row tile
    int ks0, ks1;       // k-steps [ks0, ks1)
    int R;              // rows of the tile (128, or the remainder)
    int tile;           // pair s * T1 + t, or down tile s * T2 + t
    int pc;             // K piece
    int id;             // unit index within its kind: tile * KC + piece
};

// Unit i of CTA b: list entry b + G * i (a CTA's gate/up pieces precede its down pieces).
__device__ __forceinline__ Unit unit_at(const Geometry& g, const DecodeTcParams& p, int i, int b, int G)
{
    Unit u;
    const int x = b + G * i;
    u.down = x >= g.U1;
    u.id = u.down ? x - g.U1 : x;
    const int KC = u.down ? g.KC2 : g.KC1, T = u.down ? g.T2 : g.T1;
    const int CH = u.down ? g.CHI : g.CHH, KS = u.down ? g.KSI : g.KSH;
    u.pc = u.id % KC;
    u.tile = u.id / KC;
    u.t = u.tile % T;
    u.s = u.tile / T;
    const int c0 = u.pc * CH / KC, c1 = (u.pc + 1) * CH / KC;
    u.ks0 = 2 * c0;
    u.ks1 = 2 * c1 < KS ? 2 * c1 : KS;
    const int rows = u.down ? p.H : p.I;
    u.R = rows - u.t * kRowTile < kRowTile ? rows - u.t * kRowTile : kRowTile;
    return u;
}

// One stage: [A0][A1][SFA0][SFA1][B][SFB] -- A1 / SFA1 the up tile of a pair;
// B / SFB the activation terms of the stage's k-steps (x, or h for down).
// For a partial row tile (R = 64) the MMA still reads 128 rows of a k-step
// block, up to 2 KB past A; that lands in the stage or in the ring's slack.
struct StageTc {
    uint32_t abytes, sfbytes, bbytes, size, sfa0, b, sfb;
    __device__ StageTc(int steps, int R, bool dual)
    {
        abytes = steps * R * 32;
        sfbytes = ((steps + 1) >> 1) * kSfChunk;
        bbytes = steps * kAtom;
        sfa0 = (dual ? 2 : 1) * abytes;
        b = sfa0 + (dual ? 2 : 1) * sfbytes;
        sfb = b + bbytes;
        size = (sfb + sfbytes + 127) & ~127u;
    }
};

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

// One warp, up to 4 groups of four consecutive 32-element blocks.  In group
// w (token m[w], first block kb0[w], nvalid[w] blocks in range), lanes
// 8g .. 8g+7 hold block kb0[w] + g, lane 8g + i its elements 4i .. 4i+3 in
// r[w].  Writes the kTerms MX terms of each block (term j to row 8m + j):
// codes to the k-step atoms at `q`, E8M0 bytes to the scale chunks at `sf`.
// Each term is the OCP MX quantisation of the residual the previous terms
// left; a zero residual gives zero terms.  The groups' chains are independent
// and interleaved (one warp per SM sub-partition has no other latency cover).
template <int NG>
__device__ __forceinline__ void warp_terms(float (&r)[NG][4], const int (&m)[NG], const int (&kb0)[NG],
                                           const int (&nvalid)[NG], uint8_t* q, uint8_t* sf, int lane)
{
    const int g = lane >> 3, sub = lane & 7;
    for (int j = 0; j < kTerms; ++j) {
        uint32_t a[NG];
#pragma unroll
        for (int w = 0; w < NG; ++w)
            a[w] = max(max(__float_as_uint(fabsf(r[w][0])), __float_as_uint(fabsf(r[w][1]))),
                       max(__float_as_uint(fabsf(r[w][2])), __float_as_uint(fabsf(r[w][3]))));
#pragma unroll
        for (int off = 1; off < 8; off <<= 1)
#pragma unroll
            for (int w = 0; w < NG; ++w)
                a[w] = max(a[w], __shfl_xor_sync(0xffffffffu, a[w], off));
        uint32_t half[NG], sb[NG], b0[NG], b1[NG];
#pragma unroll
        for (int w = 0; w < NG; ++w) {
            const int ef = (int)(a[w] >> 23);
            sb[w] = ef > 2 ? (uint32_t)(ef - 2) : 0u;
            const float inv = __uint_as_float((254u - sb[w]) << 23);   // 2^(127 - sb)
            b0[w] = e2m1x2(r[w][0] * inv, r[w][1] * inv);
            b1[w] = e2m1x2(r[w][2] * inv, r[w][3] * inv);
            if (a[w] == 0u)
                b0[w] = b1[w] = 0u;
            half[w] = b0[w] | (b1[w] << 8);
        }
#pragma unroll
        for (int w = 0; w < NG; ++w) {
            const uint32_t other = __shfl_xor_sync(0xffffffffu, half[w], 1);
            const int row = m[w] * kTerms + j, kb = kb0[w] + g;
            if (g < nvalid[w]) {
                if ((sub & 1) == 0)
                    *reinterpret_cast<uint32_t*>(q + (kb >> 1) * kAtom + (row >> 3) * 256 + (kb & 1) * 128 +
                                                 (row & 7) * 16 + 4 * (sub >> 1)) = half[w] | (other << 16);
                if (sub == 0)
                    sf[(kb >> 2) * kSfChunk + row * 16 + (kb & 3)] = (uint8_t)sb[w];
            }
        }
        if (j + 1 < kTerms)
#pragma unroll
            for (int w = 0; w < NG; ++w) {
                const float scale = __uint_as_float(sb[w] == 0u ? 0x00400000u : (sb[w] << 23));   // 2^(sb - 127)
                const float2 e0 = e2m1x2_to_f32(b0[w]), e1 = e2m1x2_to_f32(b1[w]);
                r[w][0] -= e0.x * scale;
                r[w][1] -= e0.y * scale;
                r[w][2] -= e1.x * scale;
                r[w][3] -= e1.y * scale;
            }
    }
}

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

// One warp, one 32-element block kb per token (lane i holds element i of
// token m's block in r[m], m < M): kTerms MX terms of each.  Term 0 takes the
// OCP shared exponent X0 = floor(log2 amax) - 2; term j uses X0 - 2j.  A
// term leaves an error of at most 2 * 2^Xj per element (half a step below 6,
// or the saturation from < 8 to 6), i.e. at most 8 * 2^X(j+1), so no later
// term exceeds the E2M1 range and every term cuts the error by at least 4:
// the block maximum is reduced once instead of per term.  The tokens' chains
// are interleaved; packing the codes into bytes and the stores come after.
__device__ __forceinline__ void warp_terms_rows(float (&r)[kMaxTokens], int M, int kb, uint8_t* q, uint8_t* sf,
                                                int lane)
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
#pragma unroll 1
    for (int m = 0; m < M; ++m) {
        uint32_t cm = codes[0], lo = sblo[0], hi = sbhi[0];
#pragma unroll
        for (int t = 1; t < kMaxTokens; ++t)
            if (m == t) {
                cm = codes[t];
                lo = sblo[t];
                hi = sbhi[t];
            }
#pragma unroll
        for (int j = 0; j < kTerms; ++j) {
            uint32_t word = ((cm >> (4 * j)) & 0xfu) << (4 * (lane & 7));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            word |= __shfl_xor_sync(0xffffffffu, word, 4);
            const int row = m * kTerms + j;
            if ((lane & 7) == 0)
                *reinterpret_cast<uint32_t*>(q + (kb >> 1) * kAtom + (row >> 3) * 256 + (kb & 1) * 128 +
                                             (row & 7) * 16 + 4 * (lane >> 3)) = word;
            if (lane == 0)
                sf[(kb >> 2) * kSfChunk + row * 16 + (kb & 3)] = (uint8_t)((j < 4 ? lo : hi) >> (8 * (j & 3)));
        }
    }
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

struct TcSmem {
    uint64_t full[kSlots], empty[kSlots], accf[2], acce[2], routed;
    uint32_t tmem_base;
    int sel[kMaxTokens][kMaxTopK];
    float wt[kMaxTokens][kMaxTopK];
    int nu;
    int unit_expert[kMaxUnits];
    unsigned char unit_of[kMaxExperts];
    float wslot[kMaxUnits][kMaxTokens];   // routing weight of token m for expert slot s (0 if not chosen)
    int flag;
};

__global__ void __launch_bounds__(kThreadsTc, 1) decode_tc_kernel(const DecodeTcParams p)
{
    extern __shared__ __align__(1024) uint8_t ring[];
    __shared__ __align__(8) TcSmem sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x, M = p.M;
    const int nrows = rows_for(M);
    const uint32_t ring_cap = (uint32_t)(p.smem_bytes - kRingSlack) & ~127u;
    const int KSI = p.I / 64, CHI = ceil_div(p.I, 128), KSH = p.H / 64;
    const long long hstride = (long long)KSI * kAtom + (long long)CHI * kSfChunk;   // h terms of one slot

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 2);   // both issuers
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.accf[i], 2);
            mbar_init(&sh.acce[i], 4);
        }
        mbar_init(&sh.routed, 1);
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
    // The logits were written before the x-term kernel started, which had waited
    // for them: routing may run before this kernel waits for its predecessor.
    if (warp < 2) {
        // ---- routing (warps 0, 1): top-k per token, then the distinct experts in ascending order
        for (int m = warp; m < M; m += 2)
            rt::warp_topk(p.logits + (size_t)m * p.E, p.E, p.k, sh.sel[m], sh.wt[m]);
        asm volatile("bar.sync 2, 64;" ::: "memory");
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
            if (lane == 0) {
                sh.nu = nu;
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            }
        }
        asm volatile("bar.sync 2, 64;" ::: "memory");
        if (warp == 1 && lane == 0)
            mbar_arrive(&sh.routed);   // hands the routing to the other warps
    } else {
        mbar_wait(&sh.routed, 0, p.status);
    }
    const Geometry g = geometry(p, sh.nu, G);
    const int nunits = units_of(g, b, G);
    if (b == 0 && tid == 0 && p.nu_out)
        *p.nu_out = g.nu;

    if (warp == 0) {
        // ================================================================ producer
        // Weight tiles stream in unit order; a pair's stage also carries the x
        // terms of its k-steps.  A down stage's h terms can only be copied once
        // the pairs that produce them have published their flag: such copies
        // wait in a queue that is served whenever the producer would otherwise
        // wait, so the weight stream never stalls on h.
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the x terms are written
        RingTc ring_alloc;
        unsigned long long ends[kSlots];
        unsigned long long rel_end = 0;
        uint32_t c = 0, rel = 0;
        // h-term copies of down stages placed before their pairs were ready, in
        // placement order; every entry names its unit's slot and chunk range
        // (all lanes hold the queue)
        uint32_t pq_off[kPend], pq_slot[kPend];
        int pq_ks[kPend], pq_steps[kPend], pq_s[kPend], pq_c0[kPend], pq_c1[kPend];
        int pq_head = 0, pq_n = 0;
        int ok_s = -1, ok_c0 = 0, ok_c1 = 0;   // the last chunk range found published
        // the whole warp: are all pairs of chunks [c0, c1) of slot s published?
        auto pairs_ready = [&](int s, int c0, int c1) -> bool {
            if (s == ok_s && c0 == ok_c0 && c1 == ok_c1)
                return true;
            bool ok = true;
            for (int ch = c0 + lane; ch < c1; ch += 32)
                ok = ok && ld_acquire_u32(p.hready + s * g.T1 + ch) != 0u;
            if (__all_sync(0xffffffffu, ok)) {
                ok_s = s;
                ok_c0 = c0;
                ok_c1 = c1;
                return true;
            }
            return false;
        };
        // the whole warp: issue the queued copies whose pairs are published, in order
        auto serve = [&]() {
            while (pq_n > 0) {
                const int h0 = pq_head % kPend;
                if (!pairs_ready(pq_s[h0], pq_c0[h0], pq_c1[h0]))
                    return;
                // the run of entries of the same unit, up to 16 (two copies each, one per lane)
                int run = 1;
                while (run < pq_n && run < 16) {
                    const int hq_ = (pq_head + run) % kPend;
                    if (pq_s[hq_] != pq_s[h0] || pq_c0[hq_] != pq_c0[h0] || pq_c1[hq_] != pq_c1[h0])
                        break;
                    ++run;
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");   // published h terms -> bulk reads
                const uint8_t* src = p.ht + (long long)pq_s[h0] * hstride;
                const int q = lane >> 1;
                if (q < run) {
                    const int e = (pq_head + q) % kPend;
                    const StageTc sg(pq_steps[e], kRowTile, false);   // B / SFB sizes do not depend on R
                    if ((lane & 1) == 0)
                        bulk_copy(ring + pq_off[e], src + (long long)pq_ks[e] * kAtom, sg.bbytes, &sh.full[pq_slot[e]]);
                    else
                        bulk_copy(ring + pq_off[e] + sg.bbytes, src + (long long)KSI * kAtom + (pq_ks[e] >> 1) * kSfChunk,
                                  sg.sfbytes, &sh.full[pq_slot[e]]);
                }
                pq_head += run;
                pq_n -= run;
            }
        };
        for (int i = 0; i < nunits; ++i) {
            const Unit u = unit_at(g, p, i, b, G);
            const int e = sh.unit_expert[u.s];
            const int K = u.down ? p.I : p.H, rows = u.down ? p.H : p.I;
            const int CH = u.down ? g.CHI : g.CHH;
            const uint8_t* proj = u.down ? p.dn + (long long)e * p.dn_expert : p.gu + (long long)e * p.gu_expert;
            const uint8_t* a0 = proj + (long long)u.t * kRowTile * (K / 2);
            const uint8_t* s0 = proj + (long long)rows * (K / 2) + (long long)u.t * CH * kSfChunk;
            const long long up = tile_proj_bytes(p.I, p.H);
            bool hready = false;   // down: the pairs of this unit's K range are published
            const int uc0 = u.ks0 >> 1, uc1 = (u.ks1 + 1) >> 1;
            if (u.down) {
                serve();
                hready = pq_n == 0 && pairs_ready(u.s, uc0, uc1);   // stages keep their order
                if (hready)
                    asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            for (int ks = u.ks0; ks < u.ks1; ks += kSteps, ++c) {
                const int steps = u.ks1 - ks < kSteps ? u.ks1 - ks : kSteps;
                const StageTc sg(steps, u.R, !u.down);
                unsigned long long end;
                const uint32_t off = ring_alloc.place(sg.size, ring_cap, &end);
                // wait until the bytes and the slot are free (stages retire in order)
                int spins = 0;
                while (rel < c && (end - rel_end > (unsigned long long)ring_cap || rel + kSlots <= c)) {
                    const uint32_t sl = rel % kSlots;
                    if (__shfl_sync(0xffffffffu, mbar_test_wait(&sh.empty[sl], (rel / kSlots) & 1) ? 1 : 0, 0)) {
                        rel_end = ends[sl];
                        ++rel;
                    } else {
                        serve();
                        if (++spins > (1 << 22)) {
                            if (lane == 0)
                                atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                            break;
                        }
                    }
                }
                const uint32_t slot = c % kSlots;
                ends[slot] = end;
                if (lane == 0)
                    mbar_expect_tx(&sh.full[slot], (u.down ? 1 : 2) * (sg.abytes + sg.sfbytes) + sg.bbytes + sg.sfbytes);
                __syncwarp();
                uint8_t* st = ring + off;
                const long long aoff = (long long)ks * u.R * 32, soff = (long long)(ks >> 1) * kSfChunk;
                const uint8_t* hsrc = p.ht + (long long)u.s * hstride;
                const uint8_t* src = nullptr;
                uint32_t dsto = 0, n = 0;
                switch (lane) {
                case 0: dsto = 0; src = a0 + aoff; n = sg.abytes; break;
                case 1: dsto = sg.sfa0; src = s0 + soff; n = sg.sfbytes; break;
                case 2: if (!u.down) { dsto = sg.abytes; src = a0 + up + aoff; n = sg.abytes; } break;
                case 3: if (!u.down) { dsto = sg.sfa0 + sg.sfbytes; src = s0 + up + soff; n = sg.sfbytes; } break;
                case 4:
                    dsto = sg.b;
                    n = !u.down || hready ? sg.bbytes : 0u;
                    src = u.down ? hsrc + (long long)ks * kAtom : p.xt + (long long)ks * kAtom;
                    break;
                case 5:
                    dsto = sg.sfb;
                    n = !u.down || hready ? sg.sfbytes : 0u;
                    src = u.down ? hsrc + (long long)KSI * kAtom + soff : p.xt + (long long)KSH * kAtom + soff;
                    break;
                default: break;
                }
                if (n)
                    bulk_copy(st + dsto, src, n, &sh.full[slot]);
                if (u.down && !hready) {
                    if (pq_n == kPend) {   // full: wait for the head's pairs
                        for (int w = 0; w < (1 << 22) && pq_n == kPend; ++w)
                            serve();
                        if (pq_n == kPend) {
                            if (lane == 0)
                                atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
                            ++pq_head;   // give up on the oldest entry (its stage will time out)
                            --pq_n;
                        }
                    }
                    const int e = (pq_head + pq_n) % kPend;
                    pq_off[e] = off + sg.b;
                    pq_slot[e] = slot;
                    pq_ks[e] = ks;
                    pq_steps[e] = steps;
                    pq_s[e] = u.s;
                    pq_c0[e] = uc0;
                    pq_c1[e] = uc1;
                    ++pq_n;
                    serve();
                    if (pq_n == 0)
                        hready = true;   // the rest of this unit's stages carry their h terms directly
                }
            }
        }
        for (int w = 0; w < (1 << 22) && pq_n > 0; ++w)
            serve();
        if (pq_n > 0 && lane == 0)
            atomicExch(p.status, MOE_ERR_DEVICE_TIMEOUT);
    } else if (warp == 1 || warp == kMmaWarpB) {
        // ================================================================ MMA issuers
        // Issuing a tcgen05 instruction costs one thread ~60-80 cycles, so two
        // threads share the work: A (warp 1) the gate MMAs, B (warp 6) the up
        // MMAs of a pair; down units alternate their stages between A and B,
        // each into its own half of the accumulator (the drain adds the halves).
        // Each issuer copies its stage scales into its own tensor-memory columns.
        const int role = warp == 1 ? 0 : 1;
        if (lane == 0) {
            RingTc ring_alloc;
            const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(nrows >> 3) << 17) | (1u << 23) |
                                   ((uint32_t)(kRowTile >> 4) << 24);
            const uint32_t myset = tmem + kSfSetCol + role * 2 * kSfSetCols;
            uint32_t c = 0, mine = 0;
            for (int i = 0; i < nunits; ++i) {
                const Unit u = unit_at(g, p, i, b, G);
                const uint32_t buf = i & 1;
                if (i >= 2)
                    mbar_wait(&sh.acce[buf], ((i >> 1) - 1) & 1, p.status);
                tc_fence_after();
                const uint32_t dme = tmem + buf * kAcc + role * kRows;   // this issuer's accumulator half
                bool first = true;
                int jst = 0;
                for (int ks = u.ks0; ks < u.ks1; ks += kSteps, ++c, ++jst) {
                    const int steps = u.ks1 - ks < kSteps ? u.ks1 - ks : kSteps;
                    const StageTc sg(steps, u.R, !u.down);
                    unsigned long long end;
                    const uint32_t st = su32(ring) + ring_alloc.place(sg.size, ring_cap, &end);
                    const uint32_t slot = c % kSlots;
                    mbar_wait(&sh.full[slot], (c / kSlots) & 1, p.status);
                    if (u.down && (jst & 1) != role) {
                        mbar_arrive(&sh.empty[slot]);   // the other issuer owns this down stage
                        continue;
                    }
                    tc_fence_after();
                    const uint32_t sa = st + (u.down || role == 0 ? 0u : sg.abytes);   // gate / up / down A
                    const uint32_t sfa = st + sg.sfa0 + (u.down || role == 0 ? 0u : sg.sfbytes);
                    const uint32_t set = myset + (mine & 1) * kSfSetCols;
                    ++mine;
                    const int chunks = (steps + 1) >> 1;
                    for (int ch = 0; ch < chunks; ++ch) {
                        tc_cp_sf(set + 4 * ch, sfa + ch * kSfChunk);
                        tc_cp_sf(set + kSfSetCols / 2 + 4 * ch, st + sg.sfb + ch * kSfChunk);
                    }
                    for (int j = 0; j < steps; ++j) {
                        const uint32_t id = (uint32_t)(2 * (j & 1));
                        const uint32_t desc = idesc | (id << 4) | (id << 29);
                        tc_mma_mxf4(dme, smem_desc(sa + j * u.R * 32, 128, 256), smem_desc(st + sg.b + j * kAtom, 128, 256),
                                    desc, set + 4 * (j >> 1), set + kSfSetCols / 2 + 4 * (j >> 1), first ? 0u : 1u);
                        first = false;
                    }
                    tc_commit(&sh.empty[slot]);
                }
                tc_commit(&sh.accf[buf]);
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ================================================================ epilogue warps
        const int te = tid - 64, q = warp & 3;
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the residual is this kernel's to write
        const int r = 32 * q + lane;   // row within the tile
        unsigned pend = 0u;   // te == 0: down counter before this CTA's previous piece
        int pend_i = -1;

        // the last piece of output slice t: out = r + sum over expert slots and K
        // pieces of the weighted partials + sum_s w_s b_s, in a fixed order
        auto finish_slice = [&](int t) {
            const int row = t * kRowTile + r;
            if (row < p.H) {
                float acc[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
                const int npc = g.nu * g.KC2;
                for (int z0 = 0; z0 < npc; z0 += 8) {
                    float4 a[8];
#pragma unroll
                    for (int z = 0; z < 8; ++z)
                        if (z0 + z < npc)
                            a[z] = __ldcg(reinterpret_cast<const float4*>(
                                              p.part2 + ((size_t)t * npc + z0 + z) * kRowTile * kMaxTokens) + r);
#pragma unroll
                    for (int z = 0; z < 8; ++z)
                        if (z0 + z < npc) {
                            acc[0] += a[z].x; acc[1] += a[z].y; acc[2] += a[z].z; acc[3] += a[z].w;
                        }
                }
                if (p.dn_bias)
                    for (int s2 = 0; s2 < g.nu; ++s2) {
                        const float bd = bf16f(p.dn_bias[(size_t)sh.unit_expert[s2] * p.H + row]);
#pragma unroll
                        for (int m = 0; m < kMaxTokens; ++m)
                            acc[m] = fmaf(sh.wslot[s2][m], bd, acc[m]);
                    }
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m) {
                    if (m >= M)
                        break;
                    uint16_t* o = p.resid + (size_t)m * p.H + row;
                    *o = f2bf16_rne(bf16f(__ldcg(o)) + acc[m]);
                }
            }
        };

        // h = silu(gate + b) * (up + b) of this warp's 32 rows of pair u (the
        // pieces' partials summed, or the pair's own sums), its MX terms to the
        // slot's h-term buffer, then the pair's release flag
        auto publish_h = [&](const Unit& u, const float (&gs_in)[kMaxTokens], const float (&us_in)[kMaxTokens],
                             bool from_partials) {
            const int row = u.t * kRowTile + r;
            if (u.t * kRowTile + 32 * q < p.I) {   // a warp's 32 rows are all valid or all not
                const int e = sh.unit_expert[u.s];
                const float bg = p.gu_bias ? bf16f(p.gu_bias[(size_t)e * 2 * p.I + row]) : 0.f;
                const float bu = p.gu_bias ? bf16f(p.gu_bias[(size_t)e * 2 * p.I + p.I + row]) : 0.f;
                float gs[kMaxTokens], us[kMaxTokens];
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m) {
                    gs[m] = gs_in[m] + bg;
                    us[m] = us_in[m] + bu;
                }
                if (from_partials)
                    for (int c0 = 0; c0 < g.KC1; c0 += 8) {
                        float4 a[8], c4[8];
#pragma unroll
                        for (int z = 0; z < 8; ++z)
                            if (c0 + z < g.KC1) {
                                const float4* src = reinterpret_cast<const float4*>(
                                    p.part1 + ((size_t)(u.tile * g.KC1 + c0 + z) * 2) * kRowTile * kMaxTokens);
                                a[z] = __ldcg(src + r);
                                c4[z] = __ldcg(src + kRowTile + r);
                            }
#pragma unroll
                        for (int z = 0; z < 8; ++z)
                            if (c0 + z < g.KC1) {
                                gs[0] += a[z].x; gs[1] += a[z].y; gs[2] += a[z].z; gs[3] += a[z].w;
                                us[0] += c4[z].x; us[1] += c4[z].y; us[2] += c4[z].z; us[3] += c4[z].w;
                            }
                    }
                float hv[kMaxTokens];
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m)
                    hv[m] = gs[m] / (1.0f + expf(-gs[m])) * us[m];
                uint8_t* dst = p.ht + (long long)u.s * hstride;
                warp_terms_rows(hv, M, row >> 5, dst, dst + (long long)KSI * kAtom, lane);
            }
            epi_barrier();
            if (te == 0)
                st_release_u32(p.hready + u.tile, 1u);
        };
        const float zero4[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
        // unit pi counted in with counter value `oldv` before it: finish its pair or
        // output slice if it was the last piece
        auto resolve = [&](int pi, unsigned oldv) {
            const Unit pu = unit_at(g, p, pi, b, G);
            const unsigned need = pu.down ? (unsigned)(g.nu * g.KC2) : (unsigned)g.KC1;
            if (te == 0)
                sh.flag = oldv == need - 1u;
            epi_barrier();
            const bool last = sh.flag;
            epi_barrier();
            if (last) {
                if (pu.down)
                    finish_slice(pu.t);
                else
                    publish_h(pu, zero4, zero4, true);
            }
        };

        for (int i = 0; i < nunits; ++i) {
            const Unit u = unit_at(g, p, i, b, G);
            if (u.down && pend_i >= 0 && !unit_at(g, p, pend_i, b, G).down) {
                // a pending gate/up piece is resolved before any down unit is waited
                // for: that down unit may need the very h this CTA has to publish
                epi_barrier();
                resolve(pend_i, pend);
                pend_i = -1;
            }
            // ---- drain: each token's term columns summed
            const uint32_t buf = i & 1;
            mbar_wait(&sh.accf[buf], (i >> 1) & 1, p.status);
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + buf * kAcc;
            const bool two = !u.down || u.ks1 - u.ks0 > kSteps;   // issuer B wrote its half
            float s0[kMaxTokens] = {0.f, 0.f, 0.f, 0.f}, s1[kMaxTokens] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int h16 = 0; h16 < kRows; h16 += 16) {
                if (h16 < nrows) {
                    float d0[16], d1[16];
                    tc_ld16(taddr + h16, d0);
                    if (two)
                        tc_ld16(taddr + kRows + h16, d1);
                    tc_wait_ld();
#pragma unroll
                    for (int col = 0; col < 16; ++col) {
                        const int m = (h16 + col) / kTerms;   // compile-time after unrolling
                        if (m < M) {
                            s0[m] += d0[col];
                            if (!u.down)
                                s1[m] += d1[col];
                            else if (two)
                                s0[m] += d1[col];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sh.acce[buf]);
            if (!u.down && g.KC1 == 1) {   // a whole pair: h right away
                publish_h(u, s0, s1, false);
                continue;
            }
            // ---- a piece: its partials (down: weighted by each token's routing weight
            // for this expert slot), counted into its pair / output slice
            unsigned* cnt;
            if (!u.down) {
                float4* dst = reinterpret_cast<float4*>(p.part1 + ((size_t)u.id * 2) * kRowTile * kMaxTokens);
                dst[r] = make_float4(s0[0], s0[1], s0[2], s0[3]);
                dst[kRowTile + r] = make_float4(s1[0], s1[1], s1[2], s1[3]);
                cnt = p.pair_cnt + u.tile;
            } else {
#pragma unroll
                for (int m = 0; m < kMaxTokens; ++m)
                    s0[m] *= m < M ? sh.wslot[u.s][m] : 0.f;
                reinterpret_cast<float4*>(p.part2 + ((size_t)u.t * g.nu * g.KC2 + u.s * g.KC2 + u.pc) *
                                                        kRowTile * kMaxTokens)[r] = make_float4(s0[0], s0[1], s0[2], s0[3]);
                cnt = p.dn_cnt + u.t;
            }
            epi_barrier();   // the piece's partials are stored
            // whether this was the last piece is read one unit later, so the atomic's
            // latency hides behind the next accumulator wait
            const unsigned prev = pend;
            const int prev_i = pend_i;
            if (te == 0)   // releases the partials; acquires the other pieces' if last
                pend = atom_add_acq_rel(cnt, 1u);
            pend_i = i;
            if (prev_i >= 0)
                resolve(prev_i, prev);
        }
        if (pend_i >= 0) {
            epi_barrier();
            resolve(pend_i, pend);
        }
    }

    // ---- exit: the last CTA out resets the counters for the next call
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(p.exit_cnt, 1u) == (unsigned)G - 1u) {
            for (int i = 0; i < g.nu * g.T1; ++i) {
                p.hready[i] = 0u;
                p.pair_cnt[i] = 0u;
            }
            for (int i = 0; i < g.T2; ++i)
                p.dn_cnt[i] = 0u;
            *p.exit_cnt = 0u;
            __threadfence();
        }
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// x terms of a layer (PDL-chained before the decode kernel): one warp per
// group of 4 blocks of one token, into the buffer the decode kernel copies
// from ([H/64 k-step atoms][ceil(H/128) scale chunks], the shared-memory order).
// With x = nullptr the input is the RMS-normalised residual,
// x = bf16(r / sqrt(mean(r^2) + 1e-6)).
__global__ void __launch_bounds__(128) xterms_kernel(const DecodeTcParams p)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float nrm[4][kMaxTokens];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, M = p.M;
    const uint16_t* xs = p.x ? p.x : p.resid;
    float inv[kMaxTokens] = {1.f, 1.f, 1.f, 1.f};
    if (!p.x) {
        for (int m = 0; m < M; ++m) {
            float a = 0.f;
            for (int i = tid; i < p.H / 2; i += 128) {
                const uint32_t w = __ldcg(reinterpret_cast<const unsigned*>(xs + (size_t)m * p.H) + i);
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
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kMaxTokens; ++m)
            inv[m] = 1.0f / sqrtf((nrm[0][m] + nrm[1][m] + nrm[2][m] + nrm[3][m]) / (float)p.H + 1e-6f);
    }
    const int nkb = p.H / 32, ngr = (nkb + 3) / 4;
    const int x = blockIdx.x * 4 + warp;
    if (x >= M * ngr)
        return;
    const int m = x / ngr, kbg = 4 * (x % ngr);
    float v[1][4];
    uint2 u2 = make_uint2(0u, 0u);
    if (kbg + (lane >> 3) < nkb)
        u2 = __ldcg(reinterpret_cast<const uint2*>(xs + (size_t)m * p.H + 32 * kbg + 4 * lane));
    v[0][0] = __uint_as_float(u2.x << 16);
    v[0][1] = __uint_as_float(u2.x & 0xffff0000u);
    v[0][2] = __uint_as_float(u2.y << 16);
    v[0][3] = __uint_as_float(u2.y & 0xffff0000u);
    if (!p.x) {
        float im = inv[0];
#pragma unroll
        for (int t = 1; t < kMaxTokens; ++t)
            im = m == t ? inv[t] : im;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[0][i] = bf16f(f2bf16_rne(v[0][i] * im));
    }
    const int mm[1] = {m}, kk[1] = {kbg}, nv[1] = {nkb - kbg};
    warp_terms<1>(v, mm, kk, nv, p.xt, p.xt + (long long)(p.H / 64) * kAtom, lane);
}

}  // namespace

cudaError_t prepare_decode_tc(size_t smem)
{
    return cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_decode_tc(const DecodeTcParams& p, size_t smem, int grid, cudaStream_t stream)
{
    const int ngr = (p.H / 32 + 3) / 4;
    cudaLaunchAttribute pre[1];
    pre[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pre[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((p.M * ngr + 3) / 4);
    pc.blockDim = dim3(128);
    pc.stream = stream;
    pc.attrs = pre;
    pc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&pc, xterms_kernel, p);
    if (e != cudaSuccess)
        return e;
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
