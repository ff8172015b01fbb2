// moe_noalloc.cu -- a layer forward that allocates nothing.
//
// Runtimes that hand the library memory they already own -- an inference
// engine with its own pre-sized pool, code that runs while a CUDA graph is
// being captured, a plug-in that must not touch the CUDA allocator -- cannot
// call cudaMalloc, so they cannot create a moe_handle (moe_create allocates
// the resident weight arena and the workspace).  moe_forward_noalloc serves
// them: every input and output is caller memory (the weights in the same
// caller layout that moe_load_experts takes), and the scratch the layer needs
// (h, the per-slot down outputs, the output-tile counters) lives in one
// file-scope __device__ array of fixed size that each GPU holding the library
// keeps until the process exits.
//
// It is a variant of the decode layer with the same arithmetic: every CTA
// routes the tokens itself; a gate_up kernel streams the selected experts'
// gate_up rows with 16-byte loads, decodes E2M1 / int4 in registers against x
// held in registers, reduces the row sums across its threads and writes
// h = silu(gate) * up; a down kernel (chained by programmatic dependent
// launch) multiplies the down rows against h and the last CTA to finish an
// 8-row output tile adds sum_s w_s * y_s to the residual in slot order.  It
// reads the caller layout directly (no load-time repack), so it trades speed
// for needing no prepared weights.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe_noalloc {

constexpr int kMaxTokens = 4;
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 256;
constexpr int kMaxUnits = kMaxTokens * kMaxTopK;
constexpr int kMaxK = 3072;            // largest H or I
constexpr int kThreads = 384;
constexpr int kRowsPerItem = 8;
enum { FMT_MXFP4 = 1, FMT_INT4 = 2 };

// Scratch layout (bytes): h [kMaxTokens][kMaxTopK][kMaxK] fp32, then ypart of
// the same shape, then the output-tile counters [kMaxK / kRowsPerItem].
constexpr size_t kHBytes = (size_t)kMaxTokens * kMaxTopK * kMaxK * sizeof(float);
constexpr size_t kCountOffset = 2 * kHBytes;
constexpr size_t kCountBytes = (size_t)(kMaxK / kRowsPerItem) * sizeof(unsigned);
constexpr size_t kScratchBytes = kCountOffset + kCountBytes;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct LayerParams {
    const uint8_t* gu_codes;   // [E][2I][H/2]
    const uint8_t* gu_scales;  // [E][2I][sbh] bytes per row
    const uint16_t* gu_bias;   // [E][2I] bf16, or nullptr
    const uint8_t* dn_codes;   // [E][H][I/2]
    const uint8_t* dn_scales;  // [E][H][sbi]
    const uint16_t* dn_bias;   // [E][H] bf16, or nullptr
    const float* logits;       // [M][E]
    const uint16_t* x;         // [M][H] bf16 layer input
    uint16_t* resid;           // [M][H] bf16 residual in, result out
    float* h;                  // scratch [M][kmax][I]
    float* ypart;              // scratch [M][kmax][H]
    unsigned int* tile_count;  // scratch [H/8] arrival counters (zero between calls)
    int* nu_out;               // unused here (nullptr)
    int H, I, E, M, k, kmax, group;
    int sbh, sbi;              // scale bytes per row of gate_up / down
};

namespace {


// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Streaming loads of read-only weight bytes: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream8(const void* p)
{
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ void named_barrier(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ __half2 as_half2(uint32_t u)
{
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return h;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f)
{
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&b);
}

// ---------------------------------------------------------------- decoding

// Eight consecutive 4-bit codes (one 32-bit word, element 2b in the low nibble
// of byte b) to fp32, without the scale.
//   MXFP4: FP4 E2M1 values (OCP MX v1.0).
//   int4 : code - 8.
template <int FMT>
__device__ __forceinline__ void decode8(uint32_t w, float (&f)[8])
{
    if constexpr (FMT == FMT_MXFP4) {
        uint32_t h0, h1, h2, h3;
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
            "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
            "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
            "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
            : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
            : "r"(w));
        float2 a = __half22float2(as_half2(h0));
        float2 b = __half22float2(as_half2(h1));
        float2 c = __half22float2(as_half2(h2));
        float2 d = __half22float2(as_half2(h3));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // halves hold elements j and j+4 as fp16 1024 + q; minus 1032 gives q - 8 exactly
            uint32_t t = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
            float2 a = __half22float2(__hsub2(as_half2(t), as_half2(0x64086408u)));
            f[j] = a.x;
            f[j + 4] = a.y;
        }
    }
}

// E8M0 scale byte to fp32: 2^(s-127); 0 -> 2^-127 (subnormal), 255 -> NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t s)
{
    uint32_t bits = s == 0 ? 0x00400000u : (s == 255 ? 0x7fc00000u : (s << 23));
    return __uint_as_float(bits);
}

// The scale that applies to element k0 of a row whose scales start at `srow`.
template <int FMT>
__device__ __forceinline__ float load_scale(const uint8_t* srow, int k0, int group)
{
    if constexpr (FMT == FMT_MXFP4) {
        return e8m0_to_f32(__ldg(srow + (k0 >> 5)));
    } else {
        uint16_t s = __ldg(reinterpret_cast<const unsigned short*>(srow) + k0 / group);
        return __half2float(__ushort_as_half(s));
    }
}

// ---------------------------------------------------------------- reduction

// Warp reduce-scatter: every lane holds S partial values (slot 0..S-1); on
// return lane l holds the warp-wide sum of slot l / (32 / S).
template <int S>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[S])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int n = S / 2, off = 16; n >= 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            float send = upper ? v[i] : v[i + n];
            float keep = upper ? v[i + n] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float t = v[0];
#pragma unroll
    for (int off = 16 / S; off >= 1; off >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, off);
    return t;
}

// ---------------------------------------------------------------- routing

// One warp: top-k of E logits (largest first; ties to the lower index; NaN
// as -inf), then softmax over the k selected.  Lane 0 writes sel[0..k) and
// the weights wt[0..k).
__device__ void warp_topk(const float* __restrict__ lg, int E, int k, int* sel, float* wt)
{
    const int lane = threadIdx.x & 31;
    float v[kMaxExperts / 32];
    uint32_t avail = 0;
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
        const int e = lane + 32 * j;
        float t = -INFINITY;
        if (e < E) {
            t = lg[e];
            if (t != t)
                t = -INFINITY;
            avail |= 1u << j;
        }
        v[j] = t;
    }
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) {
            const int e = lane + 32 * j;
            if (((avail >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < be))) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane)
            avail &= ~(1u << (be >> 5));
        if (lane == 0) {
            sel[s] = be;
            wt[s] = bv;
        }
    }
    __syncwarp();
    const float lmax = wt[0];
    const float l = lane < k ? wt[lane] : -INFINITY;
    const float e = lane < k ? expf(l - lmax) : 0.0f;
    float sum = e;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, off);
    __syncwarp();
    if (lane < k)
        wt[lane] = e / sum;
}

struct RouteSmem {
    int sel[kMaxTokens][kMaxTopK];
    float wt[kMaxTokens][kMaxTopK];
    int nu;                                   // distinct experts
    int unit_expert[kMaxUnits];               // ascending expert index
    unsigned unit_mask[kMaxUnits];            // bit m: token m routed to the unit
    signed char unit_slot[kMaxUnits][kMaxTokens];   // slot of the unit in token m's list
    unsigned char unit_of[kMaxExperts];
};

// All threads: route the M tokens into shared memory and list the units.
__device__ void route_block(const float* __restrict__ logits, int M, int E, int k, RouteSmem& rs)
{
    const int warp = threadIdx.x >> 5;
    if (warp < M)
        warp_topk(logits + (size_t)warp * E, E, k, rs.sel[warp], rs.wt[warp]);
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t bits[kMaxExperts / 32] = {};
        for (int m = 0; m < M; ++m)
            for (int s = 0; s < k; ++s)
                bits[rs.sel[m][s] >> 5] |= 1u << (rs.sel[m][s] & 31);
        int nu = 0;
        for (int wi = 0; wi < kMaxExperts / 32; ++wi) {
            uint32_t b = bits[wi];
            while (b) {
                const int e = wi * 32 + __ffs(b) - 1;
                b &= b - 1;
                rs.unit_of[e] = (unsigned char)nu;
                rs.unit_expert[nu] = e;
                rs.unit_mask[nu] = 0;
                for (int m = 0; m < kMaxTokens; ++m)
                    rs.unit_slot[nu][m] = -1;
                ++nu;
            }
        }
        for (int m = 0; m < M; ++m)
            for (int s = 0; s < k; ++s) {
                const int u = rs.unit_of[rs.sel[m][s]];
                rs.unit_slot[u][m] = (signed char)s;
                rs.unit_mask[u] |= 1u << m;
            }
        rs.nu = nu;
    }
    __syncthreads();
}

// Geometry of the row-parallel split: each thread owns KT consecutive
// elements of K; GW warps span one row ("a group"); NG groups per CTA.
template <int KT>
struct Split {
    int nthr_row, GW, NG, g, wg, tg, k0;
    bool active;
    __device__ Split(int K)
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        nthr_row = K / KT;
        GW = (nthr_row + 31) >> 5;
        NG = (kThreads / 32) / GW;
        g = warp / GW;
        wg = warp % GW;
        tg = wg * 32 + lane;
        active = tg < nthr_row;
        k0 = tg * KT;
    }
};

template <int KT>
struct Codes {
    uint32_t w[kRowsPerItem][KT / 8];
};

template <int KT>
__device__ __forceinline__ void load_row_codes(const uint8_t* p, uint32_t (&w)[KT / 8])
{
    if constexpr (KT == 32) {
        uint4 v = ld_stream16(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
        uint2 v = ld_stream8(p);
        w[0] = v.x; w[1] = v.y;
    }
}

// Partial dot products of one item (kRowsPerItem rows) for the routed tokens.
// part[r * MT + m] = scale_r * sum_{k in slice} W[r][k] x_m[k]
template <int FMT, int MT, int KT>
__device__ __forceinline__ void item_partials(const Codes<KT>& c, const float (&sc)[kRowsPerItem],
                                             const float (&xr)[MT][KT], unsigned mask,
                                             float (&part)[kRowsPerItem * MT])
{
#pragma unroll
    for (int r = 0; r < kRowsPerItem; ++r) {
        float acc0[MT], acc1[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            acc0[m] = 0.0f;
            acc1[m] = 0.0f;
        }
#pragma unroll
        for (int wi = 0; wi < KT / 8; ++wi) {
            float f[8];
            decode8<FMT>(c.w[r][wi], f);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (MT == 1 || ((mask >> m) & 1u)) {
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        acc0[m] = fmaf(f[i], xr[m][8 * wi + i], acc0[m]);
                        acc1[m] = fmaf(f[i + 1], xr[m][8 * wi + i + 1], acc1[m]);
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
            part[r * MT + m] = (acc0[m] + acc1[m]) * sc[r];
    }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// ================================================================ gate_up

template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1) gate_up_kernel(const LayerParams p)
{
    constexpr int KT = MT == 1 ? 32 : 16;
    constexpr int R = kRowsPerItem;
    constexpr int S = R * MT;
    __shared__ RouteSmem rs;
    __shared__ float red[kThreads / 32][2][S];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();   // the previous kernel (the prior layer, or whoever wrote x/logits) is done
    route_block(p.logits, p.M, p.E, p.k, rs);
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.nu_out)
        *p.nu_out = rs.nu;

    // L2 prefetch of the down weights of the selected experts, spread over the grid.
    {
        const size_t cbytes = (size_t)p.H * (p.I / 2), sbytes = (size_t)p.H * p.sbi;
        constexpr uint32_t CH = 16384;
        const int nqc = (int)((cbytes + CH - 1) / CH), nqs = (int)((sbytes + CH - 1) / CH);
        const int nq = nqc + nqs, total = rs.nu * nq;
        for (int q = blockIdx.x + gridDim.x * threadIdx.x; q < total; q += gridDim.x * blockDim.x) {
            const int u = q / nq, r = q % nq;
            const size_t e = rs.unit_expert[u];
            if (r < nqc) {
                const size_t off = (size_t)r * CH;
                prefetch_l2(p.dn_codes + e * cbytes + off, (uint32_t)min((size_t)CH, cbytes - off));
            } else {
                const size_t off = (size_t)(r - nqc) * CH;
                prefetch_l2(p.dn_scales + e * sbytes + off, (uint32_t)min((size_t)CH, sbytes - off));
            }
        }
    }

    const Split<KT> sp(p.H);
    if (sp.g >= sp.NG)
        return;   // warps left over when GW does not divide the CTA; no block barrier follows
    const int bar_id = 1 + sp.g, bar_n = sp.GW * 32;

    // x slice of every token in registers (fp32)
    float xr[MT][KT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const uint16_t* src = p.x + (size_t)m * p.H + sp.k0;
#pragma unroll
        for (int c = 0; c < KT / 8; ++c) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (sp.active && m < p.M)
                v = *reinterpret_cast<const uint4*>(src + 8 * c);
            const uint32_t u4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xr[m][8 * c + 2 * i] = bf16_to_f32((uint16_t)(u4[i] & 0xffffu));
                xr[m][8 * c + 2 * i + 1] = bf16_to_f32((uint16_t)(u4[i] >> 16));
            }
        }
    }

    // Work items: (unit, 4 consecutive gate/up pairs); contiguous ranges per group.
    const int per_unit = p.I / 4;
    const int total = rs.nu * per_unit;
    const int gid = blockIdx.x * sp.NG + sp.g, ngroups = gridDim.x * sp.NG;
    const int it0 = (int)((long long)total * gid / ngroups);
    const int it1 = (int)((long long)total * (gid + 1) / ngroups);
    const size_t row_bytes = (size_t)p.H / 2;

    auto issue = [&](int it, Codes<KT>& c, float (&sc)[R]) {
        const int u = it / per_unit, i0 = (it % per_unit) * 4;
        const size_t e = rs.unit_expert[u];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const size_t row = e * 2 * p.I + (r < 4 ? i0 + r : p.I + i0 + r - 4);
            if (sp.active) {
                load_row_codes<KT>(p.gu_codes + row * row_bytes + sp.k0 / 2, c.w[r]);
                sc[r] = load_scale<FMT>(p.gu_scales + row * p.sbh, sp.k0, p.group);
            } else {
#pragma unroll
                for (int wi = 0; wi < KT / 8; ++wi)
                    c.w[r][wi] = 0u;
                sc[r] = 0.0f;
            }
        }
    };

    Codes<KT> cur, nxt;
    float sc_cur[R], sc_nxt[R];
    if (it0 < it1)
        issue(it0, cur, sc_cur);
    int buf = 0;
    for (int it = it0; it < it1; ++it) {
        if (it + 1 < it1)
            issue(it + 1, nxt, sc_nxt);
        const int u = it / per_unit, i0 = (it % per_unit) * 4;
        const unsigned mask = rs.unit_mask[u];
        float part[S];
        item_partials<FMT, MT, KT>(cur, sc_cur, xr, mask, part);
        if (!sp.active) {
#pragma unroll
            for (int s = 0; s < S; ++s)
                part[s] = 0.0f;
        }
        const float v = warp_reduce_scatter<S>(part);
        if ((lane & (32 / S - 1)) == 0)
            red[warp][buf][lane / (32 / S)] = v;
        named_barrier(bar_id, bar_n);
        if (sp.tg < 4 * MT) {
            const int pr = sp.tg / MT, m = sp.tg % MT;
            const int slot = rs.unit_slot[u][m];
            if (m < p.M && slot >= 0) {
                float ag = 0.0f, au = 0.0f;
                for (int j = 0; j < sp.GW; ++j) {
                    ag += red[sp.g * sp.GW + j][buf][pr * MT + m];
                    au += red[sp.g * sp.GW + j][buf][(4 + pr) * MT + m];
                }
                const size_t e = rs.unit_expert[u];
                const int i = i0 + pr;
                if (p.gu_bias) {
                    ag += bf16_to_f32(p.gu_bias[e * 2 * p.I + i]);
                    au += bf16_to_f32(p.gu_bias[e * 2 * p.I + p.I + i]);
                }
                p.h[((size_t)m * p.kmax + slot) * p.I + i] = silu(ag) * au;
            }
        }
        buf ^= 1;
        cur = nxt;
#pragma unroll
        for (int r = 0; r < R; ++r)
            sc_cur[r] = sc_nxt[r];
    }
}

// ================================================================ down + combine

template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1) down_kernel(const LayerParams p)
{
    constexpr int KT = MT == 1 ? 32 : 16;
    constexpr int R = kRowsPerItem;
    constexpr int S = R * MT;
    __shared__ RouteSmem rs;
    __shared__ float red[kThreads / 32][2][S];
    __shared__ int last_flag[kThreads / 32];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    route_block(p.logits, p.M, p.E, p.k, rs);   // logits were written before gate_up began
    pdl_wait();                                  // h is complete and visible
    pdl_launch_dependents();

    const Split<KT> sp(p.I);
    if (sp.g >= sp.NG)
        return;
    const int bar_id = 1 + sp.g, bar_n = sp.GW * 32;

    const int tiles = p.H / R;
    const int total = rs.nu * tiles;
    const int gid = blockIdx.x * sp.NG + sp.g, ngroups = gridDim.x * sp.NG;
    const int it0 = (int)((long long)total * gid / ngroups);
    const int it1 = (int)((long long)total * (gid + 1) / ngroups);
    const size_t row_bytes = (size_t)p.I / 2;

    float hr[MT][KT];
    int hu = -1;
    int buf = 0;
    for (int it = it0; it < it1; ++it) {
        const int u = it / tiles, jt = it % tiles;
        const size_t e = rs.unit_expert[u];
        const unsigned mask = rs.unit_mask[u];
        if (u != hu) {
            hu = u;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const int slot = m < p.M ? rs.unit_slot[u][m] : -1;
#pragma unroll
                for (int c = 0; c < KT / 4; ++c) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (sp.active && slot >= 0)
                        v = __ldcg(reinterpret_cast<const float4*>(
                            p.h + ((size_t)m * p.kmax + slot) * p.I + sp.k0) + c);
                    hr[m][4 * c] = v.x;
                    hr[m][4 * c + 1] = v.y;
                    hr[m][4 * c + 2] = v.z;
                    hr[m][4 * c + 3] = v.w;
                }
            }
        }
        Codes<KT> c;
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const size_t row = e * p.H + (size_t)jt * R + r;
            if (sp.active) {
                load_row_codes<KT>(p.dn_codes + row * row_bytes + sp.k0 / 2, c.w[r]);
                sc[r] = load_scale<FMT>(p.dn_scales + row * p.sbi, sp.k0, p.group);
            } else {
#pragma unroll
                for (int wi = 0; wi < KT / 8; ++wi)
                    c.w[r][wi] = 0u;
                sc[r] = 0.0f;
            }
        }
        float part[S];
        item_partials<FMT, MT, KT>(c, sc, hr, mask, part);
        if (!sp.active) {
#pragma unroll
            for (int s = 0; s < S; ++s)
                part[s] = 0.0f;
        }
        const float v = warp_reduce_scatter<S>(part);
        if ((lane & (32 / S - 1)) == 0)
            red[warp][buf][lane / (32 / S)] = v;
        named_barrier(bar_id, bar_n);
        if (sp.tg < S) {
            const int r = sp.tg / MT, m = sp.tg % MT;
            const int slot = m < p.M ? rs.unit_slot[u][m] : -1;
            if (slot >= 0) {
                float y = 0.0f;
                for (int j = 0; j < sp.GW; ++j)
                    y += red[sp.g * sp.GW + j][buf][sp.tg];
                const int jrow = jt * R + r;
                if (p.dn_bias)
                    y += bf16_to_f32(p.dn_bias[e * p.H + jrow]);
                p.ypart[((size_t)m * p.kmax + slot) * p.H + jrow] = y;
                __threadfence();
            }
        }
        named_barrier(bar_id, bar_n);
        if (sp.tg == 0) {
            __threadfence();
            const unsigned old = atomicAdd(p.tile_count + jt, 1u);
            last_flag[sp.g] = (old == (unsigned)rs.nu - 1u);
        }
        named_barrier(bar_id, bar_n);
        if (last_flag[sp.g]) {
            // every unit's rows of this tile are in ypart: combine in slot order
            __threadfence();
            if (sp.tg < R * p.M) {
                const int r = sp.tg % R, m = sp.tg / R;
                const int jrow = jt * R + r;
                float acc = 0.0f;
                for (int s = 0; s < p.k; ++s)
                    acc = fmaf(rs.wt[m][s], __ldcg(p.ypart + ((size_t)m * p.kmax + s) * p.H + jrow), acc);
                uint16_t* o = p.resid + (size_t)m * p.H + jrow;
                *o = f32_to_bf16_rn(bf16_to_f32(*o) + acc);
            }
            if (sp.tg == 0)
                p.tile_count[jt] = 0u;
        }
        buf ^= 1;
    }
}


template <int FMT, int MT>
cudaError_t launch_pair(const LayerParams& p, int grid, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, gate_up_kernel<FMT, MT>, p);
    if (err != cudaSuccess)
        return err;
    return cudaLaunchKernelEx(&cfg, down_kernel<FMT, MT>, p);
}

cudaError_t launch_layer(const LayerParams& p, int fmt, int grid, cudaStream_t stream)
{
    const int mt = p.M <= 1 ? 1 : (p.M <= 2 ? 2 : 4);
    if (fmt == FMT_MXFP4) {
        if (mt == 1) return launch_pair<FMT_MXFP4, 1>(p, grid, stream);
        if (mt == 2) return launch_pair<FMT_MXFP4, 2>(p, grid, stream);
        return launch_pair<FMT_MXFP4, 4>(p, grid, stream);
    }
    if (mt == 1) return launch_pair<FMT_INT4, 1>(p, grid, stream);
    if (mt == 2) return launch_pair<FMT_INT4, 2>(p, grid, stream);
    return launch_pair<FMT_INT4, 4>(p, grid, stream);
}

int fail(int code, const char* msg) { return moe::set_error(code, "moe_forward_noalloc: %s", msg); }

// Device address of g_scratch and SM count, looked up once per device.  In
// host code the name g_scratch is only a host-side stand-in for the symbol, so
// its device address has to come from cudaGetSymbolAddress.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_dev[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int device_setup(int dev, unsigned char** scratch, int* sms)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_dev[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
        if (e != cudaSuccess || !ptr)
            return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return fail(MOE_ERR_CUDA, "cudaDeviceGetAttribute failed");
        g_sms[dev] = n;
        g_scratch_dev[dev] = static_cast<unsigned char*>(ptr);
    }
    *scratch = g_scratch_dev[dev];
    *sms = g_sms[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe_noalloc

extern "C" int moe_forward_noalloc(const moe_config* cfg, const void* gu_codes, const void* gu_scales,
                                   const void* gu_bias, const void* dn_codes, const void* dn_scales,
                                   const void* dn_bias, const void* x_bf16, const float* router_logits,
                                   int M, int top_k, void* out_bf16, void* stream)
{
    using namespace moe_noalloc;
    if (!cfg)
        return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
    const int H = cfg->hidden, I = cfg->intermediate, E = cfg->num_experts;
    if (H <= 0 || H % 32 || H > kMaxK || I <= 0 || I % 32 || I > kMaxK)
        return fail(MOE_ERR_INVALID_ARG, "hidden and intermediate must be multiples of 32, at most 3072");
    if (E < 1 || E > kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "num_experts must be in 1..256");
    if (M < 1 || M > kMaxTokens)
        return fail(MOE_ERR_INVALID_ARG, "M must be in 1..4 (the scratch array holds 4 tokens)");
    if (top_k < 1 || top_k > kMaxTopK || top_k > E)
        return fail(MOE_ERR_INVALID_ARG, "top_k must be in 1..min(num_experts, 16)");
    if (cfg->format == MOE_FMT_MXFP4) {
        if (cfg->group != 32)
            return fail(MOE_ERR_INVALID_ARG, "MXFP4 needs group == 32");
    } else if (cfg->format == MOE_FMT_INT4) {
        if (cfg->group < 32 || cfg->group % 32 || H % cfg->group || I % cfg->group)
            return fail(MOE_ERR_INVALID_ARG, "int4 group must be a multiple of 32 dividing H and I");
    } else {
        return fail(MOE_ERR_INVALID_ARG, "unknown format");
    }
    if (!gu_codes || !gu_scales || !dn_codes || !dn_scales || !x_bf16 || !router_logits || !out_bf16)
        return fail(MOE_ERR_INVALID_ARG, "a required pointer is NULL");
    if (cfg->has_bias && (!gu_bias || !dn_bias))
        return fail(MOE_ERR_INVALID_ARG, "has_bias is set but a bias pointer is NULL");
    // x, out and the codes are read and written with 16-byte vector accesses, and
    // the scale arrays are prefetched into L2 in runs that must start on 16-byte
    // boundaries; the biases are bf16 and the logits fp32 loads
    if (((uintptr_t)x_bf16 | (uintptr_t)out_bf16 | (uintptr_t)gu_codes | (uintptr_t)dn_codes |
         (uintptr_t)gu_scales | (uintptr_t)dn_scales) & 15u)
        return fail(MOE_ERR_INVALID_ARG, "x, out and the code and scale arrays must be 16-byte aligned");
    if (((uintptr_t)router_logits & 3u) ||
        (cfg->has_bias && (((uintptr_t)gu_bias | (uintptr_t)dn_bias) & 1u)))
        return fail(MOE_ERR_INVALID_ARG, "router_logits must be 4-byte and the biases 2-byte aligned");
    const uintptr_t xa = (uintptr_t)x_bf16, oa = (uintptr_t)out_bf16, nb = (uintptr_t)M * H * 2;
    if (xa < oa + nb && oa < xa + nb)
        return fail(MOE_ERR_INVALID_ARG, "x overlaps out");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(MOE_ERR_CUDA, "cudaGetDevice failed");
    unsigned char* scratch = nullptr;
    int sms = 0;
    int rc = device_setup(dev, &scratch, &sms);
    if (rc != MOE_OK)
        return rc;
    LayerParams p{};
    p.gu_codes = static_cast<const uint8_t*>(gu_codes);
    p.gu_scales = static_cast<const uint8_t*>(gu_scales);
    p.gu_bias = cfg->has_bias ? static_cast<const uint16_t*>(gu_bias) : nullptr;
    p.dn_codes = static_cast<const uint8_t*>(dn_codes);
    p.dn_scales = static_cast<const uint8_t*>(dn_scales);
    p.dn_bias = cfg->has_bias ? static_cast<const uint16_t*>(dn_bias) : nullptr;
    p.logits = router_logits;
    p.x = static_cast<const uint16_t*>(x_bf16);
    p.resid = static_cast<uint16_t*>(out_bf16);
    p.h = reinterpret_cast<float*>(scratch);
    p.ypart = reinterpret_cast<float*>(scratch + kHBytes);
    p.tile_count = reinterpret_cast<unsigned*>(scratch + kCountOffset);
    p.nu_out = nullptr;
    p.H = H;
    p.I = I;
    p.E = E;
    p.M = M;
    p.k = top_k;
    p.kmax = kMaxTopK;
    p.group = cfg->group;
    p.sbh = cfg->format == MOE_FMT_MXFP4 ? H / 32 : 2 * (H / cfg->group);
    p.sbi = cfg->format == MOE_FMT_MXFP4 ? I / 32 : 2 * (I / cfg->group);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the tile counters must start at zero; a call that was cut short could leave them set
    cudaError_t e = cudaMemsetAsync(p.tile_count, 0, (size_t)(H / kRowsPerItem) * sizeof(unsigned), s);
    if (e == cudaSuccess)
        e = launch_layer(p, cfg->format, sms, s);
    if (e != cudaSuccess)
        return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    return MOE_OK;
}
