// moe_decode_i4.cu -- the packed-int4 decode layer (M <= 4 tokens): one
// persistent launch of one or more layer calls, one CTA per SM.
//
// The layer is the one of "Single-stream int4 decode of a 30B MoE on Apple
// Silicon", sections 1 and 6: symmetric int4 weights, W = (code - 8) * s with
// one fp16 scale s per `group` elements along K, dequantised on chip.  The
// pages' fused kernel dequantises in registers and multiplies (TinyTitan
// tracker, D108 and D110: 16-byte row reads).  Here the codes go straight
// into the A fragments of m16n8k16 f16 MMAs: (1024 + q) - 1032 is q - 8
// exactly in f16, so no instruction per weight runs beyond the decode.  The
// fp16 scales are not powers of two, so they have no exact form as the block
// scales of the 5th-generation tensor cores (E8M0); each group's fp32 MMA sum
// is multiplied by its scale once instead.
//
// Work unit: 64 rows of h of one selected expert -- 4 gate slabs and the 4 up
// slabs of the same rows (16 rows each), and the matching 64 K columns of the
// down projection for every output row -- so SwiGLU is local to the CTA and
// only the output is summed across CTAs.  Units are dealt in contiguous
// ranges, CTA b taking [b U / G, (b+1) U / G).  The weights are stored in the
// order they stream (written at load time):
//   gate/up of unit t: [K/64 segments][8 slabs][32 lanes x 16 bytes] codes,
//                      then [K/64][8][8 x SB] scale entries;
//   down of unit t:    [H/16 slabs][32 lanes x 16 bytes] codes, then
//                      [H/16][8 x SB] scale entries,
// where the 16 code bytes of (slab, lane) cover the four m16n8k16 A fragments
// of one 64-column segment (word j: k16 step j; register i of it = nibbles i
// and i + 4), and an SB-byte entry holds the fp16 scales of rows g and g + 8
// (SB = 8 when group is 32: both 32-element blocks of the segment).  One bulk
// copy moves a stage of a unit: up to 16 gate/up segments or 128 down slabs (64 KB:
// smaller bulk copies stream markedly slower per SM).
//
// 16 warps compute: on a gate/up stage warp w takes slab w mod 8 and every
// other segment of the stage (w / 8 picks which; the two halves' sums are added
// in a fixed order), on a down stage slabs w, w + 16, ...  No warp is kept for
// the stream: thread 0 fills the stage ring once a call is routed, and the last
// warp to finish with a stage refills its slot (a 17th warp would cap the
// registers at 96: one scheduler would hold five warps).  x enters as f16 after an exact power-of-two rescale per token (its
// largest magnitude to [2^14, 2^15)); h' = w h as f16 hi + lo after a
// power-of-two rescale per (unit, token).  Products and sums are fp32.
//
// Calls of one launch are separated by grid barriers: call c + 1 reads its
// routing and inputs only after every CTA's slice of call c's output is
// written.  Every wait is bounded and reports MOE_ERR_DEVICE_TIMEOUT.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "moe_internal.h"
#include "route.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kCw = 16;                    // compute warps (4 per SM sub-partition); no producer
constexpr int kThreadsI4 = kCw * 32;       // warp: the last warp out of a stage issues the next
constexpr int kGuSeg = 16;                 // segments per gate/up stage (64 KB of codes)
constexpr int kDnSlabs = 128;              // slabs per down stage (64 KB of codes)
static_assert(kGuSeg * 4096 <= kI4Codes && kDnSlabs * 512 <= kI4Codes, "a stage's codes fit a slot");
static_assert(kGuSeg * 64 * 8 <= kI4Slot - kI4Codes && kDnSlabs * 8 * 8 <= kI4Slot - kI4Codes,
              "a stage's scale entries fit a slot");
constexpr int kMaxSlotsI4 = 12;
constexpr int kFinI4 = 64;

__device__ __forceinline__ void cw_barrier() { asm volatile("bar.sync 1, %0;" ::"r"(kCw * 32) : "memory"); }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u)
{
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return h;
}

// The four f16x2 A registers of one m16n8k16 MMA from one code word: register
// i holds nibbles i and i + 4.  A nibble q placed in the low bits of an f16
// 0x6400 is 1024 + q, and q - 8 = (1024 + q) - 1032; placed 4 bits up it is
// 1024 + 16 q, and q - 8 = (1024 + 16 q) / 16 - 72 (one fma).  All exact.
__device__ __forceinline__ void decode_i4(uint32_t w, uint32_t (&a)[4])
{
    const uint32_t w8 = w >> 8;
    const __half2 k1032 = u2h(0x64086408u), k16 = u2h(0x2C002C00u), k72 = u2h(0xD480D480u);
    a[0] = h2u(__hsub2(u2h((w & 0x000F000Fu) | 0x64006400u), k1032));
    a[1] = h2u(__hfma2(u2h((w & 0x00F000F0u) | 0x64006400u), k16, k72));
    a[2] = h2u(__hsub2(u2h((w8 & 0x000F000Fu) | 0x64006400u), k1032));
    a[3] = h2u(__hfma2(u2h((w8 & 0x00F000F0u) | 0x64006400u), k16, k72));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Grid barrier (one thread of each CTA): the counter only grows, G per
// barrier; `skip` arrives without adding (debug: the others' waits run out).
__device__ __forceinline__ void grid_sync_i4(unsigned long long* cnt, int G, int limit, int* status, bool skip)
{
    const unsigned long long old = skip ? ld_acquire_u64(cnt) : atom_add_release_u64(cnt, 1ull);
    const unsigned long long tgt = (old / (unsigned long long)G + 1ull) * (unsigned long long)G;
    int spins = 0;
#pragma unroll 1
    while (ld_acquire_u64(cnt) < tgt) {
        if (++spins > limit) {
            atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
            break;
        }
    }
}

// 2^e for e in [-252, 252], as a product of two representable powers of two.
__device__ __forceinline__ float pow2_mul(float v, int e)
{
    const int e1 = e / 2, e2 = e - e1;
    return (v * __uint_as_float((uint32_t)(127 + e1) << 23)) * __uint_as_float((uint32_t)(127 + e2) << 23);
}

// floor(log2 |v|) of a non-zero finite fp32 value (subnormals included).
__device__ __forceinline__ int ilog2f(float v)
{
    const uint32_t u = __float_as_uint(v) & 0x7fffffffu;
    return u >= 0x00800000u ? (int)(u >> 23) - 127 : (31 - __clz((int)u)) - 149;
}

struct I4Smem {
    uint64_t full[kMaxSlotsI4];
    unsigned done[kMaxSlotsI4];           // warps finished with each slot's stages (only grows)
    int sel[kMaxTokens][kMaxTopK];
    float wt[kMaxTokens][kMaxTopK];
    int nu;
    int unit_expert[kMaxUnits];
    unsigned char unit_of[kMaxExperts];
    float wslot[kMaxUnits][kMaxTokens];
    unsigned xmax[kMaxTokens];            // largest |x| per token (fp32 bits)
    float xinv[kMaxTokens];               // 1 / rms of the residual per token (normalised input)
    int xsh[kMaxTokens];                  // power-of-two shift of x per token
    unsigned hmax[2][kMaxTokens];         // largest |h'| per token of a unit (two units alternate)
    float fin[kFinI4][4];
};

// Shared memory past the ring: x as f16 [M][H + 8], the unit's gate/up sums of
// both K halves [2][128][4], h' as f16 hi and lo [2][4][64], the CTA's output
// copy [H][V].
__device__ __forceinline__ uint32_t i4_tail_bytes(int H, int M)
{
    return (uint32_t)M * (H + 8) * 2 + 2 * 128 * 4 * 4 + 2 * 4 * 64 * 2 + (uint32_t)H * 4 * 4;
}
__device__ __forceinline__ int sb_of(int group) { return group == 32 ? 8 : 4; }

extern __shared__ __align__(1024) uint8_t i4ring[];
__shared__ __align__(8) I4Smem si;

__global__ void __launch_bounds__(kThreadsI4, 1) decode_i4_kernel(const DecodeI4Params p)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int G = gridDim.x, b = blockIdx.x, M = p.M, H = p.H, I = p.I;
    const int KS = H / 64, T1 = I / 64, NSL = H / 16;
    const int SB = sb_of(p.group);
    const int V = M == 1 ? 1 : (M == 2 ? 2 : 4);
    const long long gu_unit = (long long)KS * (4096 + 64 * SB), dn_unit = (long long)NSL * (512 + 8 * SB);
    // slots of the stage ring, then the tail
    const uint32_t tail = (i4_tail_bytes(H, M) + 127u) & ~127u;
    const int nslots = min(kMaxSlotsI4, (int)(((uint32_t)p.smem_bytes - tail) / kI4Slot));
    uint8_t* tailp = i4ring + (uint32_t)nslots * kI4Slot;
    __half* xh = reinterpret_cast<__half*>(tailp);                                       // [M][H + 8]
    float* gsum = reinterpret_cast<float*>(tailp + (uint32_t)M * (H + 8) * 2);           // [2][128][4]
    __half* hs16 = reinterpret_cast<__half*>(gsum + 2 * 128 * 4);                         // [2][4][64]
    float* oacc = reinterpret_cast<float*>(hs16 + 2 * 4 * 64);                            // [H][V]

    if (tid == 0) {
        for (int i = 0; i < nslots; ++i) {
            mbar_init(&si.full[i], 1);
            si.done[i] = 0u;
        }
        for (int m = 0; m < kMaxTokens; ++m)
            si.hmax[0][m] = si.hmax[1][m] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");

    uint32_t st_count = 0;   // stages of the launch consumed so far: the ring position (same on every thread)
    int ubase = 0;           // whole units done by this CTA in earlier calls (h' buffers alternate)
#pragma unroll 1
    for (int call = 0; call < p.ncalls; ++call) {
        const int layer = (p.layer0 + call) % p.nlayers;
        const uint8_t* gu = p.gu + (long long)layer * p.layer_stride;
        const uint8_t* dn = p.dn + (long long)layer * p.layer_stride;
        const float* logits = reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(p.logits) +
                                                             (long long)call * p.logits_stride);
        const uint16_t* xin = p.x ? reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.x) +
                                                                     (long long)call * p.x_stride) : nullptr;
        uint16_t* resid = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(p.resid) +
                                                      (long long)(call / p.resid_every) * p.resid_stride);
        float* of32 = p.out_f32 ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(p.out_f32) +
                                                          (long long)call * p.out_f32_stride) : nullptr;
        const uint16_t* gub = p.gu_bias ? reinterpret_cast<const uint16_t*>(
            reinterpret_cast<const uint8_t*>(p.gu_bias) + (long long)layer * p.bias_stride) : nullptr;
        const uint16_t* dnb = p.dn_bias ? reinterpret_cast<const uint16_t*>(
            reinterpret_cast<const uint8_t*>(p.dn_bias) + (long long)layer * p.bias_stride) : nullptr;

        // ---- the stage stream: stage j of this call (unit u0 + j / nsu, its gate/up
        // stages then its down stages) goes into slot (call_base + j) mod nslots.
        // Lane 0 of warp 0 issues the first stage as soon as the routing is known
        // and fills the ring once x is converted; after that, the last warp to
        // finish with a slot's stage issues the stage nslots further on into it.
        const int ngu = (KS + kGuSeg - 1) / kGuSeg, ndn = (NSL + kDnSlabs - 1) / kDnSlabs, nsu = ngu + ndn;
        const uint32_t call_base = st_count;
        auto issue = [&](int j, int ufirst) {
            const int u = ufirst + j / nsu, sl = j % nsu;
            const int e = si.unit_expert[u / T1], t = u % T1;
            const uint8_t* gsrc = gu + (long long)e * p.gu_expert + (long long)t * gu_unit;
            const uint8_t* dsrc = dn + (long long)e * p.dn_expert + (long long)t * dn_unit;
            uint32_t cb, sb2;
            const uint8_t *csrc, *ssrc;
            if (sl < ngu) {
                const int q0 = sl * kGuSeg, n = min(kGuSeg, KS - q0);
                cb = (uint32_t)n * 4096;
                sb2 = (uint32_t)n * 64 * SB;
                csrc = gsrc + (long long)q0 * 4096;
                ssrc = gsrc + (long long)KS * 4096 + (long long)q0 * 64 * SB;
            } else {
                const int s0 = (sl - ngu) * kDnSlabs, n = min(kDnSlabs, NSL - s0);
                cb = (uint32_t)n * 512;
                sb2 = (uint32_t)n * 8 * SB;
                csrc = dsrc + (long long)s0 * 512;
                ssrc = dsrc + (long long)NSL * 512 + (long long)s0 * 8 * SB;
            }
            const uint32_t slot = (call_base + (uint32_t)j) % nslots;
            uint8_t* dst = i4ring + slot * kI4Slot;
            const uint64_t wpol = l2_evict_first();
            mbar_expect_tx(&si.full[slot], cb + sb2);
            bulk_copy_hint(dst, csrc, cb, &si.full[slot], wpol);
            bulk_copy_hint(dst + kI4Codes, ssrc, sb2, &si.full[slot], wpol);
        };
        {
            // ---- token statistics (warp 4 + m: token m): largest |x|, and 1 / rms for
            // the normalised input
            if (warp >= 4 && warp - 4 < M) {
                const int m = warp - 4;
                const uint16_t* row = (xin ? xin : resid) + (size_t)m * H;
                float ss = 0.f;
                uint32_t mx = 0u;
                for (int i = lane; i < H / 8; i += 32) {
                    const uint4 w = __ldcg(reinterpret_cast<const uint4*>(row) + i);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float lo = __uint_as_float(ws[c] << 16), hi = __uint_as_float(ws[c] & 0xffff0000u);
                        ss = fmaf(lo, lo, ss);
                        ss = fmaf(hi, hi, ss);
                        mx = max(mx, max(ws[c] & 0x7fffu, (ws[c] >> 16) & 0x7fffu));
                    }
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, off);
                mx = __reduce_max_sync(0xffffffffu, mx);
                if (lane == 0) {
                    const float inv = xin ? 1.f : 1.0f / sqrtf(ss / (float)H + 1e-6f);
                    float amax = bf16f((uint16_t)mx);
                    if (!xin)
                        amax = bf16f(f2bf16_rne(amax * inv));   // (rounding is monotone)
                    si.xinv[m] = inv;
                    si.xsh[m] = amax > 0.f ? 14 - ilog2f(amax) : 0;
                }
            }
            const float* lgp = logits;
            if (p.router) {
                // ---- router GEMV: this CTA's logits (experts e = b, b + G, ..., one
                // (token, expert) pair a warp) from the layer input (x, or the
                // normalised residual rounded to bf16 as below), with the decode and
                // batched paths' summation order; then a grid barrier publishes them
                cw_barrier();
                const uint16_t* rw = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.router) +
                                                                       (long long)layer * p.router_stride);
                const int nre = b < p.E ? (p.E - 1 - b) / G + 1 : 0;
                if (warp < M * nre) {
                    const int m = warp % M, e = b + (warp / M) * G;
                    const uint4* xv = reinterpret_cast<const uint4*>((xin ? xin : resid) + (size_t)m * H);
                    const uint4* wv = reinterpret_cast<const uint4*>(rw + (size_t)e * H);
                    const float inv = si.xinv[m];
                    float acc = 0.f;
                    for (int i = lane; i < H / 8; i += 32) {
                        const uint4 x4 = __ldcg(xv + i), w4 = __ldg(wv + i);
                        const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w}, ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            float lo = __uint_as_float(xw[c] << 16), hi = __uint_as_float(xw[c] & 0xffff0000u);
                            if (!xin) {
                                lo = bf16f(f2bf16_rne(lo * inv));
                                hi = bf16f(f2bf16_rne(hi * inv));
                            }
                            acc = fmaf(lo, __uint_as_float(ww[c] << 16), acc);
                            acc = fmaf(hi, __uint_as_float(ww[c] & 0xffff0000u), acc);
                        }
                    }
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        acc += __shfl_xor_sync(0xffffffffu, acc, off);
                    if (lane == 0)
                        p.rlog[m * p.E + e] = acc + bf16f(__ldg(rw + (size_t)p.E * H + e));
                }
                cw_barrier();
                if (tid == 0)
                    grid_sync_i4(p.done, G, p.spin_limit, p.status, false);
                cw_barrier();
                lgp = p.rlog;
            }
            // ---- routing (warp m: token m), the distinct experts, the weight table
            if (warp < M)
                rt::warp_topk_fit(lgp + (size_t)warp * p.E, p.E, p.k, si.sel[warp], si.wt[warp]);
            cw_barrier();
            if (warp == 0) {
                uint32_t bits = 0;
                if (lane < kMaxExperts / 32)
                    for (int m = 0; m < M; ++m)
                        for (int s = 0; s < p.k; ++s) {
                            const int e = si.sel[m][s];
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
                    si.unit_of[e] = (unsigned char)u;
                    si.unit_expert[u] = e;
                    ++u;
                }
                const int nu = __shfl_sync(0xffffffffu, incl, 31);
                __syncwarp();
                if (lane == 0) {
                    si.nu = nu;
                    // the ring's first stage goes out now, ahead of the x conversion; the
                    // others wait until its reads of x are done (they would queue behind)
                    const int Uq = nu * T1;
                    const int uf = (int)((long long)b * Uq / G), ul = (int)((long long)(b + 1) * Uq / G);
                    if ((ul - uf) * nsu > 0)
                        issue(0, uf);   // the rest once the x conversion's reads are done
                }
            }
            // x as f16: x 2^S per token (S from the largest |x|), exact for every
            // element within 2^-28 of the largest
            for (int i = tid; i < M * H / 8; i += kCw * 32) {
                const int m = i / (H / 8), c = 8 * (i - m * (H / 8));
                const uint4 w = __ldcg(reinterpret_cast<const uint4*>((xin ? xin : resid) + (size_t)m * H + c));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                const float inv = si.xinv[m];
                const int sh = si.xsh[m];
                uint32_t o[4];
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    float lo = __uint_as_float(ws[z] << 16), hi = __uint_as_float(ws[z] & 0xffff0000u);
                    if (!xin) {
                        lo = bf16f(f2bf16_rne(lo * inv));
                        hi = bf16f(f2bf16_rne(hi * inv));
                    }
                    o[z] = h2u(__floats2half2_rn(pow2_mul(lo, sh), pow2_mul(hi, sh)));
                }
                *reinterpret_cast<uint4*>(xh + m * (H + 8) + c) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            for (int i = tid; i < H * V; i += kCw * 32)
                oacc[i] = 0.f;
            cw_barrier();
            if (tid == 0) {
                const int Uq = si.nu * T1;
                const int uf = (int)((long long)b * Uq / G), ul = (int)((long long)(b + 1) * Uq / G);
                for (int j = 1; j < (ul - uf) * nsu && j < nslots; ++j)
                    issue(j, uf);
            }
            if (warp == 1) {
                const int nu = si.nu;
                for (int x = lane; x < nu * kMaxTokens; x += 32)
                    si.wslot[x / kMaxTokens][x % kMaxTokens] = 0.f;
                __syncwarp();
                for (int x = lane; x < kMaxTokens * kMaxTopK; x += 32) {
                    const int m = x / kMaxTopK, k2 = x % kMaxTopK;
                    if (m < M && k2 < p.k)
                        si.wslot[si.unit_of[si.sel[m][k2]]][m] = si.wt[m][k2];
                }
            }
            cw_barrier();
        }

        const int nu = si.nu, U = nu * T1;
        const int u0 = (int)((long long)b * U / G), u1 = (int)((long long)(b + 1) * U / G);
        if (b == 0 && tid == 0 && p.nu_out)
            p.nu_out[layer] = nu;

        const int ntot = (u1 - u0) * nsu;
        // a warp is through with the stage in `slot`: the last of the kCw refills it
        auto release = [&](uint32_t slot) {
            __syncwarp();
            if (lane == 0) {
                unsigned prev;
                asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                             : "=r"(prev) : "r"(su32(&si.done[slot])) : "memory");
                const int j = (int)(st_count - call_base) + nslots;
                if ((prev + 1u) % kCw == 0u && j < ntot)
                    issue(j, u0);
            }
        };
        {
            // ================================================================ compute warps
            for (int u = u0; u < u1; ++u) {
                const int s = u / T1, t = u % T1, e = si.unit_expert[s];
                // ---- gate / up: warp w takes slab w & 7 (rows: gate 64t + 16 (w & 7), or up
                // 64t + 16 ((w & 7) - 4)) and the even (w < 8) or odd segments of each stage
                const int slab = warp & 7, half = warp >> 3;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int st = 0; st < ngu; ++st, ++st_count) {
                    const uint32_t slot = st_count % nslots;
                    mbar_wait(&si.full[slot], (st_count / nslots) & 1, p.status);
                    const uint8_t* sp = i4ring + slot * kI4Slot;
                    const int q0 = st * kGuSeg, n = min(kGuSeg, KS - q0);
#pragma unroll 8
                    for (int qi = half; qi < n; qi += 2) {
                        const int q = q0 + qi;
                        const uint4 cw = *reinterpret_cast<const uint4*>(sp + qi * 4096 + slab * 512 + lane * 16);
                        const uint8_t* ent = sp + kI4Codes + (qi * 8 + slab) * 8 * SB + g * SB;
                        float sg0, sh0, sg1, sh1;
                        {
                            const uint32_t e0 = *reinterpret_cast<const uint32_t*>(ent);
                            sg0 = __low2float(u2h(e0));
                            sh0 = __high2float(u2h(e0));
                            if (SB == 8) {
                                const uint32_t e1 = *reinterpret_cast<const uint32_t*>(ent + 4);
                                sg1 = __low2float(u2h(e1));
                                sh1 = __high2float(u2h(e1));
                            } else {
                                sg1 = sg0;
                                sh1 = sh0;
                            }
                        }
                        const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
                        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t a[4];
                            decode_i4(w4[j], a);
                            const int k0 = 64 * q + 16 * j + 2 * t4;
                            uint32_t b0 = 0u, b1 = 0u;
                            if (g < M) {
                                b0 = *reinterpret_cast<const uint32_t*>(xh + g * (H + 8) + k0);
                                b1 = *reinterpret_cast<const uint32_t*>(xh + g * (H + 8) + k0 + 8);
                            }
                            if (j < 2)
                                mma16816(d0, a, b0, b1);
                            else
                                mma16816(d1, a, b0, b1);
                        }
                        // one scale per 64 columns (SB = 4) or per 32 (SB = 8: two blocks)
                        acc[0] = fmaf(d0[0], sg0, acc[0]);
                        acc[1] = fmaf(d0[1], sg0, acc[1]);
                        acc[2] = fmaf(d0[2], sh0, acc[2]);
                        acc[3] = fmaf(d0[3], sh0, acc[3]);
                        acc[0] = fmaf(d1[0], sg1, acc[0]);
                        acc[1] = fmaf(d1[1], sg1, acc[1]);
                        acc[2] = fmaf(d1[2], sh1, acc[2]);
                        acc[3] = fmaf(d1[3], sh1, acc[3]);
                    }
                    release(slot);
                }
                // rows 16 slab + g and + 8 of the unit's 128 (gate 0..63, up 64..127), tokens
                // 2 t4, 2 t4 + 1, for this warp's K half
                if (t4 < 2) {
                    float* gs = gsum + half * 128 * 4;
                    gs[(16 * slab + g) * 4 + 2 * t4] = acc[0];
                    gs[(16 * slab + g) * 4 + 2 * t4 + 1] = acc[1];
                    gs[(16 * slab + g + 8) * 4 + 2 * t4] = acc[2];
                    gs[(16 * slab + g + 8) * 4 + 2 * t4 + 1] = acc[3];
                }
                cw_barrier();
                // ---- SwiGLU: thread (row r = tid / 4, token m = tid % 4) of the first 256,
                // h' = w h; the two K halves added in a fixed order
                const int hb = (ubase + u - u0) & 1;
                float hv = 0.f;
                if (tid < 256) {
                    const int r = tid >> 2, m = tid & 3;
                    if (m < M) {
                        const float wt = si.wslot[s][m];
                        const float xs = pow2_mul(1.f, -si.xsh[m]);
                        float gg = (gsum[r * 4 + m] + gsum[128 * 4 + r * 4 + m]) * xs;
                        float uu = (gsum[(64 + r) * 4 + m] + gsum[128 * 4 + (64 + r) * 4 + m]) * xs;
                        if (gub) {
                            gg += bf16f(__ldg(gub + (size_t)e * 2 * I + 64 * t + r));
                            uu += bf16f(__ldg(gub + (size_t)e * 2 * I + I + 64 * t + r));
                        }
                        hv = wt != 0.f ? wt * swiglu(gg, uu, p.sw_alpha, p.sw_limit, p.sw_beta) : 0.f;
                    }
                    uint32_t mx = __float_as_uint(fabsf(hv));
                    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    if (lane < 4)
                        atomicMax(&si.hmax[hb][lane], mx);
                }
                cw_barrier();
                if (tid < 256) {
                    const int r = tid >> 2, m = tid & 3;
                    const float hm = __uint_as_float(si.hmax[hb][m]);
                    const int sh = hm > 0.f ? 14 - ilog2f(hm) : 0;
                    const float hsv = pow2_mul(hv, sh);
                    const __half hi = __float2half_rn(hsv);
                    const __half lo = __float2half_rn(hsv - __half2float(hi));
                    hs16[m * 64 + r] = hi;
                    hs16[4 * 64 + m * 64 + r] = lo;
                    if (tid < kMaxTokens)
                        si.hmax[hb ^ 1][tid] = 0u;   // for the next unit
                }
                cw_barrier();
                // ---- down: this warp's slabs of the unit against h' (hi and lo fragments)
                uint32_t bh[4][2], bl[4][2];
                float hinv[2];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k0 = 16 * j + 2 * t4;
                    const __half* hrow = hs16 + (g < 4 ? g : 0) * 64;
                    const bool ok = g < M;
                    bh[j][0] = ok ? *reinterpret_cast<const uint32_t*>(hrow + k0) : 0u;
                    bh[j][1] = ok ? *reinterpret_cast<const uint32_t*>(hrow + k0 + 8) : 0u;
                    bl[j][0] = ok ? *reinterpret_cast<const uint32_t*>(hrow + 4 * 64 + k0) : 0u;
                    bl[j][1] = ok ? *reinterpret_cast<const uint32_t*>(hrow + 4 * 64 + k0 + 8) : 0u;
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int m = 2 * t4 + c;
                    const float hm = m < kMaxTokens ? __uint_as_float(si.hmax[hb][m]) : 0.f;
                    hinv[c] = hm > 0.f ? pow2_mul(1.f, ilog2f(hm) - 14) : 0.f;
                }
                for (int st = 0; st < ndn; ++st, ++st_count) {
                    const uint32_t slot = st_count % nslots;
                    mbar_wait(&si.full[slot], (st_count / nslots) & 1, p.status);
                    const uint8_t* sp = i4ring + slot * kI4Slot;
                    const int s0 = st * kDnSlabs, n = min(kDnSlabs, NSL - s0);
#pragma unroll 8
                    for (int si2 = warp; si2 < n; si2 += kCw) {
                        const int sl = s0 + si2;
                        const uint4 cw = *reinterpret_cast<const uint4*>(sp + si2 * 512 + lane * 16);
                        const uint8_t* ent = sp + kI4Codes + si2 * 8 * SB + g * SB;
                        const uint32_t e0 = *reinterpret_cast<const uint32_t*>(ent);
                        const uint32_t e1 = SB == 8 ? *reinterpret_cast<const uint32_t*>(ent + 4) : e0;
                        const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
                        float dh0[4] = {0.f, 0.f, 0.f, 0.f}, dh1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t a[4];
                            decode_i4(w4[j], a);
                            if (j < 2) {
                                mma16816(dh0, a, bh[j][0], bh[j][1]);
                                mma16816(dh0, a, bl[j][0], bl[j][1]);
                            } else {
                                mma16816(dh1, a, bh[j][0], bh[j][1]);
                                mma16816(dh1, a, bl[j][0], bl[j][1]);
                            }
                        }
                        const float sg0 = __low2float(u2h(e0)), sh0 = __high2float(u2h(e0));
                        const float sg1 = __low2float(u2h(e1)), sh1 = __high2float(u2h(e1));
                        if (t4 < 2) {
                            const int r0 = 16 * sl + g, r1 = r0 + 8;
                            const float y00 = fmaf(dh1[0], sg1, dh0[0] * sg0) * hinv[0];
                            const float y01 = fmaf(dh1[1], sg1, dh0[1] * sg0) * hinv[1];
                            const float y10 = fmaf(dh1[2], sh1, dh0[2] * sh0) * hinv[0];
                            const float y11 = fmaf(dh1[3], sh1, dh0[3] * sh0) * hinv[1];
                            const int m0 = 2 * t4;
                            if (m0 < M) {
                                oacc[r0 * V + m0] += y00;
                                oacc[r1 * V + m0] += y10;
                            }
                            if (m0 + 1 < M) {
                                oacc[r0 * V + m0 + 1] += y01;
                                oacc[r1 * V + m0 + 1] += y11;
                            }
                        }
                    }
                    release(slot);
                }
            }
            cw_barrier();
            // ---- the CTA's output copy to its partial slot [H][V]
            if (u1 > u0) {
                const float4* src4 = reinterpret_cast<const float4*>(oacc);
                float4* dst4 = reinterpret_cast<float4*>(p.part + (size_t)b * H * V);
                for (int i = tid; i < H * V / 4; i += kCw * 32)
                    dst4[i] = src4[i];
            }
        }
        ubase += u1 - u0;

        // ---- this CTA's slice of the output: float4s [f0, f1) of a copy [H][V];
        // r + sum_s w_s b_s of its elements are loaded before the grid barrier
        const int U4 = H * V / 4;
        const int f0 = (int)((long long)b * U4 / G), f1 = (int)((long long)(b + 1) * U4 / G), nf = f1 - f0;
        auto fin_term = [&](int j, int z) -> float {
            const int el = (f0 + j) * 4 + z, row = el / V, m = el - row * V;
            float v = 0.f;
            if (m < M) {
                if (dnb)
                    for (int s2 = 0; s2 < nu; ++s2)
                        v = fmaf(si.wslot[s2][m], bf16f(__ldg(dnb + (size_t)si.unit_expert[s2] * H + row)), v);
                v += bf16f(__ldcg(resid + (size_t)m * H + row));
            }
            return v;
        };
        if (tid < nf && tid < kFinI4)
#pragma unroll
            for (int z = 0; z < 4; ++z)
                si.fin[tid][z] = fin_term(tid, z);
        __syncthreads();
        if (tid == 0)
            grid_sync_i4(p.done, G, p.spin_limit, p.status, b == p.skip_cta);
        __syncthreads();
        // every CTA with units holds a copy: CTA c has units iff [c U / G, (c+1) U / G) is not empty
        {
            const float4* part = reinterpret_cast<const float4*>(p.part);
            for (int j = warp; j < nf; j += kThreadsI4 / 32) {
                // lane l takes CTAs l, l + 32, ... (all its loads in flight at once),
                // then a fixed shuffle tree: the order never depends on timing
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c0 = lane; c0 < G; c0 += 8 * 32) {
                    float4 a[8];
                    bool has[8];
#pragma unroll
                    for (int z = 0; z < 8; ++z) {
                        const int c = c0 + 32 * z;
                        has[z] = c < G && (long long)(c + 1) * U / G > (long long)c * U / G;
                        if (has[z])
                            a[z] = __ldcg(part + (size_t)c * U4 + f0 + j);
                    }
#pragma unroll
                    for (int z = 0; z < 8; ++z)
                        if (has[z]) {
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
                const float sums[4] = {acc.x, acc.y, acc.z, acc.w};
                float mine = 0.f;
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    if (lane == z)
                        mine = sums[z];
                if (lane < 4) {
                    const int el = (f0 + j) * 4 + lane, row = el / V, m = el - row * V;
                    if (m < M) {
                        const float v = (j < kFinI4 ? si.fin[j][lane] : fin_term(j, lane)) + mine;
                        resid[(size_t)m * H + row] = f2bf16_rne(v);
                        if (of32)
                            of32[(size_t)m * H + row] = v;
                    }
                }
            }
        }
        if (call + 1 < p.ncalls) {
            __syncthreads();
            if (tid == 0)
                grid_sync_i4(p.done, G, p.spin_limit, p.status, false);
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- load time

// Caller layout -> the int4 unit layout of one projection for E experts.
// proj 0: gate_up [2I][H] (gate rows 0..I-1, up rows I..2I-1); proj 1: down [H][I].
// Work item: one 32-bit code word, or one SB-byte scale entry.
__global__ void repack_i4_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int E,
                                 int H, int I, int group, int proj, uint8_t* __restrict__ out, long long expert_bytes)
{
    const int SB = sb_of(group), T1 = I / 64, KS = H / 64, NSL = H / 16;
    const int K = proj == 0 ? H : I;             // caller row length in elements
    const int nsc = K / group;                   // caller scales per row
    const long long unit = proj == 0 ? (long long)KS * (4096 + 64 * SB) : (long long)NSL * (512 + 8 * SB);
    const long long cwords = proj == 0 ? (long long)T1 * KS * 8 * 128 : (long long)T1 * NSL * 128;
    const long long nent = proj == 0 ? (long long)T1 * KS * 8 * 8 : (long long)T1 * NSL * 8;
    const long long per_e = cwords + nent;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < (long long)E * per_e;
         idx += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(idx / per_e);
        long long r = idx % per_e;
        const bool is_code = r < cwords;
        if (!is_code)
            r -= cwords;
        int t, q, j, lane, jj, gg, sl;
        long long row0, dst;
        if (proj == 0) {
            if (is_code) {
                jj = (int)(r % 4); r /= 4;
                lane = (int)(r % 32); r /= 32;
            } else {
                gg = (int)(r % 8); r /= 8;
            }
            j = (int)(r % 8); r /= 8;
            q = (int)(r % KS);
            t = (int)(r / KS);
            const long long base = (long long)e * expert_bytes + (long long)t * unit;
            row0 = j < 4 ? 64 * t + 16 * j : I + 64 * t + 16 * (j - 4);
            dst = is_code ? base + (long long)q * 4096 + j * 512 + lane * 16 + jj * 4
                          : base + (long long)KS * 4096 + ((long long)q * 8 + j) * 8 * SB + gg * SB;
        } else {
            if (is_code) {
                jj = (int)(r % 4); r /= 4;
                lane = (int)(r % 32); r /= 32;
            } else {
                gg = (int)(r % 8); r /= 8;
            }
            sl = (int)(r % NSL);
            t = (int)(r / NSL);
            q = t;   // the unit's 64 columns of K = I
            const long long base = (long long)e * expert_bytes + (long long)t * unit;
            row0 = 16 * sl;
            dst = is_code ? base + (long long)sl * 512 + lane * 16 + jj * 4
                          : base + (long long)NSL * 512 + (long long)sl * 8 * SB + gg * SB;
        }
        const int rows = proj == 0 ? 2 * I : H;
        const uint8_t* cbase = codes + (size_t)e * rows * (K / 2);
        if (is_code) {
            const int g = lane >> 2, t4 = lane & 3;
            const uint8_t* r0 = cbase + (size_t)(row0 + g) * (K / 2);
            const uint8_t* r1 = r0 + 8 * (size_t)(K / 2);
            auto nib = [](const uint8_t* row, int k) -> uint32_t { return (row[k >> 1] >> (4 * (k & 1))) & 0xfu; };
            const int c = 64 * q + 16 * jj + 2 * t4;
            const uint32_t word = nib(r0, c) | (nib(r1, c) << 4) | (nib(r0, c + 8) << 8) | (nib(r1, c + 8) << 12) |
                                  (nib(r0, c + 1) << 16) | (nib(r1, c + 1) << 20) | (nib(r0, c + 9) << 24) |
                                  (nib(r1, c + 9) << 28);
            *reinterpret_cast<uint32_t*>(out + dst) = word;
        } else {
            const uint16_t* sbase = scales + (size_t)e * rows * nsc;
            const size_t ra = (size_t)(row0 + gg), rb = ra + 8;
            uint16_t* d16 = reinterpret_cast<uint16_t*>(out + dst);
            if (SB == 4) {
                const int gi = 64 * q / group;
                d16[0] = sbase[ra * nsc + gi];
                d16[1] = sbase[rb * nsc + gi];
            } else {
                d16[0] = sbase[ra * nsc + 2 * q];
                d16[1] = sbase[rb * nsc + 2 * q];
                d16[2] = sbase[ra * nsc + 2 * q + 1];
                d16[3] = sbase[rb * nsc + 2 * q + 1];
            }
        }
    }
}

// Element (n, k) of one projection in caller order, read back from the unit
// layout with the kernel's decode: (q - 8) times its fp16 scale, in fp32.
__global__ void dequant_i4_kernel(const uint8_t* __restrict__ w, int H, int I, int group, int proj,
                                  float* __restrict__ out)
{
    const int SB = sb_of(group), KS = H / 64, NSL = H / 16;
    const int N = proj == 0 ? 2 * I : H, K = proj == 0 ? H : I;
    const long long unit = proj == 0 ? (long long)KS * (4096 + 64 * SB) : (long long)NSL * (512 + 8 * SB);
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < (long long)N * K;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx / K), k = (int)(idx % K);
        long long code_at, ent_at;
        int rr;
        const int kk = k % 64, jj = kk / 16, kc = kk % 16;
        if (proj == 0) {
            const bool up = n >= I;
            const int nn = up ? n - I : n, t = nn / 64, j = (up ? 4 : 0) + (nn % 64) / 16, q = k / 64;
            rr = nn % 16;
            const long long base = (long long)t * unit;
            code_at = base + (long long)q * 4096 + j * 512;
            ent_at = base + (long long)KS * 4096 + ((long long)q * 8 + j) * 8 * SB;
        } else {
            const int sl = n / 16, t = k / 64;
            rr = n % 16;
            const long long base = (long long)t * unit;
            code_at = base + (long long)sl * 512;
            ent_at = base + (long long)NSL * 512 + (long long)sl * 8 * SB;
        }
        const int g = rr & 7, hi = rr >> 3, t4 = (kc & 7) >> 1, second = kc >= 8;
        const uint32_t word = *reinterpret_cast<const uint32_t*>(w + code_at + (4 * g + t4) * 16 + jj * 4);
        const int reg = 2 * second + hi;
        const uint32_t q4 = (word >> ((kc & 1) ? 16 + 4 * reg : 4 * reg)) & 0xfu;
        const uint16_t* ent = reinterpret_cast<const uint16_t*>(w + ent_at + g * SB);
        const float s = __half2float(__ushort_as_half(SB == 4 ? ent[hi] : ent[hi + 2 * (kk / 32)]));
        out[idx] = (float)((int)q4 - 8) * s;
    }
}

}  // namespace

long long i4_unit_bytes(int H, int group, int proj)
{
    const int SB = group == 32 ? 8 : 4;
    return proj == 0 ? (long long)(H / 64) * (4096 + 64 * SB) : (long long)(H / 16) * (512 + 8 * SB);
}

size_t decode_i4_static_smem()
{
    cudaFuncAttributes a{};
    return cudaFuncGetAttributes(&a, decode_i4_kernel) == cudaSuccess ? a.sharedSizeBytes : 0;
}

cudaError_t prepare_decode_i4(size_t smem)
{
    return cudaFuncSetAttribute(decode_i4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_decode_i4(const DecodeI4Params& p, size_t smem, int grid, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsI4);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_i4_kernel, p);
}

cudaError_t launch_repack_i4(const uint8_t* codes, const uint16_t* scales, int E, int H, int I, int group, int proj,
                             uint8_t* out, long long expert_bytes, cudaStream_t stream)
{
    const long long per_e = proj == 0 ? (long long)(I / 64) * (H / 64) * 8 * (128 + 8)
                                      : (long long)(I / 64) * (H / 16) * (128 + 8);
    const long long work = (long long)E * per_e;
    const long long blocks = (work + 255) / 256 < 65536 ? (work + 255) / 256 : 65536;
    repack_i4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, E, H, I, group, proj, out, expert_bytes);
    return cudaGetLastError();
}

cudaError_t launch_dequant_i4(const uint8_t* w, int H, int I, int group, int proj, float* out, cudaStream_t stream)
{
    const long long total = (long long)(proj == 0 ? 2 * I : H) * (proj == 0 ? H : I);
    const long long blocks = (total + 255) / 256 < 8192 ? (total + 255) / 256 : 8192;
    dequant_i4_kernel<<<(unsigned)blocks, 256, 0, stream>>>(w, H, I, group, proj, out);
    return cudaGetLastError();
}

}  // namespace moe
