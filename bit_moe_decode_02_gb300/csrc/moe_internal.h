// moe_internal.h -- declarations shared by the C-ABI layer (moe_api.cu) and
// the kernels.  Not part of the public interface.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr int kMaxTokens = 4;      // decode M
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 256;
constexpr int kMaxUnits = kMaxTokens * kMaxTopK;   // distinct experts of one layer call
constexpr int kMaxK = 3072;        // largest H or I

// Record the calling thread's error message (read by moe_last_error) and
// return `code`.
int set_error(int code, const char* fmt, ...);

// ------------------------------------------------------------------ batched
// Calls with M > kMaxTokens run per-expert grouped GEMMs on the tensor cores
// (tcgen05.mma kind::mxf4: MXFP4 weights x MXFP4-quantised activations, fp32
// accumulators in tensor memory).  Weights are kept once, in a "tile" layout
// made for that instruction, which the decode kernels stream as well.
//
// Tile layout of one projection W [N][K] (N, K multiples of 64).  Row tile t
// covers rows 128t .. 128t + R_t - 1 (R_t = 128, or N % 128 for the last one),
// k-step s covers K = 64s .. 64s + 63.
//   codes  an R_t x 32-byte block per (t, s) in the canonical no-swizzle
//          K-major order -- row r, byte b at (r/8)*256 + (b/16)*128 + (r%8)*16
//          + b%16 (8x16-byte core matrices; K-direction stride 128, row-group
//          stride 256) -- at t*128*K/2 + s*R_t*32 (row-tile-major: gate_up)
//          or at s*N*32 + t*128*32 (k-step-major: down).
//   scales at N*K/2 + (t*C + c)*512 (row-tile-major) or N*K/2 + (c*T + t)*512
//          (k-step-major), C = ceil(K/128), T = ceil(N/128): chunk c of tile t
//          holds the E8M0 bytes of K-blocks 4c..4c+3 of the tile's 128 rows,
//          row r = i + 32j and block kb at i*16 + j*4 + kb (the order a
//          32x128-bit tensor-memory copy replicated to the four lane quarters
//          expects).
// A decode unit of gate_up is one row tile over all of K, and of down one
// k-step over all rows: each order makes a unit's bytes one contiguous run.
// The gate_up matrix [2I][K] (gate rows 0..I-1, up rows I..2I-1) is stored as
// one projection of 2I rows in the interleaved row order: tile t holds gate rows
// 64t .. 64t+63 as its rows 0..63 and up rows 64t .. 64t+63 as its rows
// 64..127, so one 128-row MMA gives gate and up of the same 64 rows of h.
// Activations (x, h) use the same two orders per token tile: codes
// [k-step][npad rows x 32 bytes], scales [chunk][512].
constexpr int kMaxBatchTokens = 8192;
constexpr int kTokTile = 96;       // tokens of one MMA (N), a multiple of 16
constexpr int kRowTile = 128;      // weight rows of one MMA (M)
constexpr int kSfChunk = 512;

inline __host__ __device__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline __host__ __device__ long long tile_proj_bytes(int N, int K)
{
    return (long long)N * K / 2 + (long long)ceil_div(N, kRowTile) * ceil_div(K, 128) * kSfChunk;
}
// Byte offsets, within one expert's projection, of the R_t x 32-byte
// block (row tile t, k-step s) and of scale chunk (row tile t, 128-column
// chunk ch).  Row-tile-major (kmajor = 0): a tile's k-steps follow one
// another, so one row tile over all of K is contiguous (gate_up: a decode unit
// is one row tile).  K-step-major (kmajor = 1): the tiles of one k-step follow
// one another (rows 0 .. N-1 of k-step s are contiguous, and so are the scale
// chunks of one column chunk), so one k-step over all rows is contiguous
// (down: a decode unit is one k-step of every row).
inline __host__ __device__ long long tile_block_off(int N, int K, int t, int s, int kmajor)
{
    const int R = N - t * kRowTile < kRowTile ? N - t * kRowTile : kRowTile;
    return kmajor ? (long long)s * N * 32 + (long long)t * kRowTile * 32
                  : (long long)t * kRowTile * (K / 2) + (long long)s * R * 32;
}
inline __host__ __device__ long long tile_sf_off(int N, int K, int t, int ch, int kmajor)
{
    const int T = ceil_div(N, kRowTile), CH = ceil_div(K, 128);
    return (long long)N * (K / 2) + (long long)(kmajor ? ch * T + t : t * CH + ch) * kSfChunk;
}

inline int max_tok_tiles(int Mk, int E) { return E + ceil_div(Mk, kTokTile); }

struct TokTile {
    int e;          // expert
    int p0;         // first permuted slot
    int n;          // tokens (slots) in the tile, 1..kTokTile
    int npad;       // n rounded up to a multiple of 16 (the MMA's N)
    long long boff; // byte offset of the tile's codes in an activation buffer, per 64 of K
};

struct BatchParams {
    const uint8_t* gu;          // interleaved tile layout: expert e at + e*gu_expert
    const uint8_t* dn;          // expert e at + e*dn_expert
    long long gu_expert, dn_expert;
    const uint16_t* gu_bias;    // [E][2I] bf16, or nullptr
    const uint16_t* dn_bias;    // [E][H] bf16, or nullptr
    const float* logits;        // [M][E]
    const uint16_t* x;          // [M][H] bf16
    uint16_t* resid;            // [M][H] bf16 in/out
    // workspace
    int* idx;                   // [M][k] selected experts
    float* wt;                  // [M][k] routing weights
    int* slot;                  // [M*k] permuted slot of each (token, choice)
    int* etile;                 // [M*k] token tile of each (token, choice)
    int* erow;                  // [M*k] row inside that tile
    int* ntiles;                // [1]
    TokTile* tiles;             // [max_tok_tiles]
    uint8_t* xq;                // activation codes, tile order (boff * H/64 per tile)
    uint8_t* xsf;               // [tile][ceil(H/128)][512]
    uint8_t* hq;
    uint8_t* hsf;               // [tile][ceil(I/128)][512]
    float* y;                   // [M*k][H], slot order
    int* status;
    int* nu_out;                // experts with at least one token (written by plan_kernel)
    float* out_f32;             // [M][H] fp32 result before the bf16 rounding, or nullptr
    int H, I, E, M, k;
    int max_tiles;
    // bf16 numerics (moe_batched_f16.cu): bf16 activation tiles of x and of h
    // (hi and lo rows), or f16 = 0 for the MXFP4 activations above
    int f16;
    uint8_t* x16;
    uint8_t* h16;
    float sw_alpha, sw_limit, sw_beta;   // the SwiGLU form (alpha, limit, offset; 1, +inf, 0: plain)
};

// Enqueue the batched layer (route, plan, quantise x, gate_up GEMM + SwiGLU +
// quantise h, down GEMM, combine) on `stream`; `grid` = SM count.
cudaError_t launch_batched(const BatchParams& p, int grid, cudaStream_t stream, int* launches);
cudaError_t prepare_batched_kernels();
// The bf16 variant's two GEMMs and the x packing that feeds them (after route
// and plan, before combine); the bytes of its activation tiles for `rows`
// padded rows.
cudaError_t launch_batched_f16_gemms(const BatchParams& p, int grid, cudaStream_t stream);
cudaError_t prepare_batched_f16_kernels();
size_t batched_f16_act_bytes(long long rows, int H, int I);
// Caller layout [E][N][K/2] codes + [E][N][K/32] E8M0 -> tile layout (one projection
// per expert of N rows of a caller matrix with `src_rows` rows).  Tile row n comes
// from caller row n, or with `interleave` = I > 0 (N = 2I) from the interleaved
// gate_up order: row 64t + r (r < 64) or I + 64t + r - 64 of tile t; `kmajor`
// picks the k-step-major order.
cudaError_t launch_repack_tiles(const uint8_t* codes, const uint8_t* scales, int E, int src_rows,
                                int N, int K, int interleave, int kmajor, uint8_t* out, long long expert_bytes,
                                cudaStream_t stream);
// MX quantisation of n fp32 values (n % 32 == 0) into natural order codes/scales.
cudaError_t launch_mx_quantize(const float* in, long long n, uint8_t* codes, uint8_t* scales,
                               cudaStream_t stream);
// The h codes of the last batched call, back in [M*k][I/2] / [M*k][I/32] order.
cudaError_t launch_untile_h(const BatchParams& p, uint8_t* codes, uint8_t* scales,
                            cudaStream_t stream);

// ------------------------------------------------------ tensor-core decode
// The MXFP4 decode layer (M <= 4) on tcgen05 kind::mxf4 (moe_decode_tc.cu);
// weights in the tile layout above.  One persistent launch per layer, chained
// to the previous grid with programmatic dependent launch.

struct DecodeTcParams {
    // One launch runs `ncalls` layer calls in sequence: call c uses resident layer
    // (layer0 + c) mod nlayers and its own inputs and outputs (base + c * stride,
    // strides in bytes; a stride of 0 reuses the same buffer, as the stack does
    // with its residual).  Call c + 1 reads nothing before call c's output is
    // complete (a grid barrier separates them).
    const uint8_t* gu;          // layer 0's interleaved tile layout: expert e at + e*gu_expert
    const uint8_t* dn;          // layer 0's down tiles: expert e at + e*dn_expert
    long long layer_stride;     // bytes from one layer's tiles to the next
    long long gu_expert, dn_expert;
    const uint16_t* gu_bias;    // layer 0's [E][2I] bf16 (gate | up), or nullptr
    const uint16_t* dn_bias;    // layer 0's [E][H] bf16, or nullptr
    long long bias_stride;      // bytes from one layer's biases to the next
    const float* logits;        // [M][E] per call
    const uint16_t* x;          // [M][H] bf16 per call, or nullptr: RMS-normalise resid
    uint16_t* resid;            // [M][H] bf16 in/out per call
    float* out_f32;             // [M][H] fp32 result before the bf16 rounding per call, or nullptr
    long long logits_stride, x_stride, resid_stride, out_f32_stride;
    int resid_every;            // calls per residual buffer: call c uses resid + (c / resid_every) * resid_stride
    float sw_alpha, sw_limit, sw_beta;   // the SwiGLU form (alpha, limit, offset; 1, +inf, 0: plain)
    int ncalls, layer0, nlayers;
    float* part;                // [G][H][4] each CTA's fp32 copy of the expert output
    uint8_t* xt;                // x terms of the layer: [H/64][N rows x 32 B][ceil(H/128)][512]
    float* gpart;               // [G][128][4] gate/up partial sums of split-unit pieces
    unsigned* pflag;            // [G] piece partial published: the call's tag
    unsigned long long* xcnt;   // [1] x-term publications, G per call (only grows)
    unsigned long long* done;   // [1] grid-barrier arrivals, G per barrier (only grows)
    int* status;
    int* nu_out;                // [nlayers] distinct experts of the last call on each layer
    int H, I, E, M, k;
    int smem_bytes;             // dynamic shared memory of the layer kernel
    int spin_limit;             // polls before a cross-CTA wait gives up (kSpinLimit by default)
    int skip_cta;               // debug: this CTA skips its grid-barrier arrival (-1: none)
    // In-kernel router: layer 0's router weights bf16 [E][H] followed by the
    // bias bf16 [E] (router_stride bytes from one layer's to the next), or
    // nullptr when the caller gives the logits.  The call's logits go to rlog
    // [kMaxTokens][E] (the last call's stay there).
    const uint16_t* router;
    long long router_stride;
    float* rlog;
};
constexpr int kSpinLimit = 1 << 24;

constexpr int kHTermBytes = 1024 + kSfChunk;   // one k-step of activation terms + its scale chunk
// x terms of a layer: k-step atoms, scale chunks, then 16 bytes holding 2^-S_m
// for each token m (S_m >= 0: the power-of-two shift the token's terms carry)
inline size_t tc_terms_bytes(int K)
{
    return (size_t)(K / 64) * 1024 + (size_t)ceil_div(K, 128) * kSfChunk + 16;
}
inline size_t tc_part_bytes(int G, int H) { return (size_t)G * H * 4 * sizeof(float); }
constexpr int kTcCounterWords = 3;   // xcnt, done, the streaming probe's barrier (64-bit)
cudaError_t prepare_decode_tc(size_t smem);
size_t decode_tc_static_smem();
cudaError_t launch_decode_tc(const DecodeTcParams& p, size_t smem, int grid, cudaStream_t stream);

// ------------------------------------------------------------ int4 decode
// The packed-int4 decode layer (M <= 4) on m16n8k16 f16 MMAs (moe_decode_i4.cu),
// weights in the unit layout described there; calls and strides as for
// DecodeTcParams.
struct DecodeI4Params {
    const uint8_t* gu;          // layer 0's gate/up units: expert e at + e*gu_expert
    const uint8_t* dn;          // layer 0's down units: expert e at + e*dn_expert
    long long layer_stride, gu_expert, dn_expert;
    const uint16_t* gu_bias;    // layer 0's [E][2I] bf16, or nullptr
    const uint16_t* dn_bias;    // layer 0's [E][H] bf16, or nullptr
    long long bias_stride;
    const float* logits;
    const uint16_t* x;          // or nullptr: RMS-normalise resid
    uint16_t* resid;
    float* out_f32;
    long long logits_stride, x_stride, resid_stride, out_f32_stride;
    int resid_every;            // calls per residual buffer: call c uses resid + (c / resid_every) * resid_stride
    float sw_alpha, sw_limit, sw_beta;   // the SwiGLU form (alpha, limit, offset; 1, +inf, 0: plain)
    int ncalls, layer0, nlayers;
    float* part;                // [G][H][4] each CTA's fp32 copy of the expert output
    unsigned long long* done;   // [1] grid-barrier arrivals (only grows)
    int* status;
    int* nu_out;                // [nlayers]
    int H, I, E, M, k, group;
    int smem_bytes;
    int spin_limit, skip_cta;
    const uint16_t* router;     // in-kernel router (as for the MXFP4 decode), or nullptr
    long long router_stride;
    float* rlog;
};
constexpr int kI4Slot = 73728;    // one stage: up to 64 KB of codes, then up to 8 KB of scales
constexpr int kI4Codes = 65536;
// bytes of one unit (64 rows of h) of gate/up (proj 0) or down (proj 1)
long long i4_unit_bytes(int H, int group, int proj);
size_t decode_i4_static_smem();
cudaError_t prepare_decode_i4(size_t smem);
cudaError_t launch_decode_i4(const DecodeI4Params& p, size_t smem, int grid, cudaStream_t stream);
cudaError_t launch_repack_i4(const uint8_t* codes, const uint16_t* scales, int E, int H, int I, int group, int proj,
                             uint8_t* out, long long expert_bytes, cudaStream_t stream);
cudaError_t launch_dequant_i4(const uint8_t* w, int H, int I, int group, int proj, float* out, cudaStream_t stream);

// Debug kernels.
// One expert projection of the tile layout back to fp32 in caller row order
// (gate_up: interleave = I, rows [0, I) gate and [I, 2I) up; down: 0).
// Load-time layout conversions (moe_loader.cu): [E][K][N] 4-bit codes ->
// [E][N][K]; [E][R][C] elements of esz bytes -> [E][C][R]; gate/up rows
// alternating -> gate rows then up rows (rows of row_bytes bytes, R rows).
cudaError_t launch_transpose_nibbles(const uint8_t* src, uint8_t* dst, int E, int N, int K, cudaStream_t s);
cudaError_t launch_transpose_elems(const uint8_t* src, uint8_t* dst, int E, int R, int C, int esz, cudaStream_t s);
cudaError_t launch_deinterleave_rows(const uint8_t* src, uint8_t* dst, int E, int R, long long row_bytes,
                                     cudaStream_t s);
// The streaming floor probe (moe_probe.cu): n regions of `bytes` bytes, region r
// at base + r * region_stride, read one after another by `grid` CTAs with bulk
// copies and a grid barrier (counter cnt) between regions.
cudaError_t launch_stream_read(const uint8_t* base, long long region_stride, long long bytes, int nregions,
                               unsigned long long* cnt, int spin_limit, int* status, int grid, cudaStream_t s);
// Router GEMV logits [M][E] = x [M][H] . W^T + b (w: W bf16 [E][H] then b [E]),
// fp32 with the decode kernel's summation order.
cudaError_t launch_router_gemv(const uint16_t* x, const uint16_t* w, int M, int H, int E, float* out,
                               cudaStream_t stream);
cudaError_t launch_dequant_tiles(const uint8_t* tiles, int N, int K, int interleave, int kmajor, float* out,
                                 cudaStream_t stream);
cudaError_t launch_dequant(int fmt, int group, const uint8_t* slabs, int N, int K, int slab_bytes,
                           float* out, cudaStream_t stream);
cudaError_t launch_route(const float* logits, int M, int E, int k, int* idx, float* w,
                         cudaStream_t stream);

}  // namespace moe
