// moe_internal.h -- declarations shared by the C-ABI layer (moe_api.cu) and
// the kernels (moe_decode.cu).  Not part of the public interface.
//
// Resident weight layout ("slabs").  Every expert projection W [N][K] is
// stored as N/16 slabs of 16 consecutive rows.  A slab is
//     [codes: K/64 segments x 32 lanes x 16 bytes][scales: K/64 x 8 x SB bytes]
// where the 16 code bytes of (segment q, lane l) are exactly the A operands of
// lane l for the four m16n8k16 MMAs that cover K = 64q .. 64q+63 (g = l/4,
// t = l%4; word j holds rows g and g+8, elements 16j + {2t, 2t+1, 2t+8, 2t+9}),
// and the SB scale bytes of (segment q, g) are the scales of rows g and g+8
// for that segment.  A slab is contiguous, so one bulk copy moves it.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr int kMaxTokens = 4;      // decode M
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 256;
constexpr int kMaxUnits = kMaxTokens * kMaxTopK;   // distinct experts of one layer call
constexpr int kMaxK = 3072;        // largest H or I (12 warps x 4 segments x 64)
constexpr int kComputeWarps = 12;  // MMA warps of the layer kernel
constexpr int kThreads = (kComputeWarps + 2) * 32;   // + a producer and a signalling warp
constexpr int kMaxSegPerWarp = kMaxK / 64 / kComputeWarps;
constexpr int kSlabRows = 16;
constexpr int kMaxSlots = 8;       // depth of the shared-memory slab ring
constexpr int kSmemBudget = 220 * 1024;    // dynamic shared memory of the layer kernel
constexpr int kRedBytes = 2 * kComputeWarps * 32 * kMaxTokens * 4;
constexpr int kXfragBytes = kComputeWarps * kMaxSegPerWarp * 4 * 32 * 8;   // x MMA fragments

enum { FMT_MXFP4 = 1, FMT_INT4 = 2 };

// Scale bytes per (segment, g) entry: MXFP4 4 (two E8M0 blocks x two rows),
// int4 with one group per segment or more 4 (one fp16 x two rows), int4 with
// 32-element groups 8 (two fp16 x two rows).
inline __host__ __device__ int scale_entry_bytes(int fmt, int group)
{
    return fmt == FMT_MXFP4 ? 4 : (group == 32 ? 8 : 4);
}
inline __host__ __device__ int slab_bytes(int K, int sb) { return 8 * K + (K / 64) * 8 * sb; }

struct LayerParams {
    const uint8_t* gu;          // gate_up slabs of expert 0; expert e at + e * gu_expert_bytes
    const uint8_t* dn;          // down slabs
    const uint16_t* gu_bias;    // [E][2I] bf16, or nullptr
    const uint16_t* dn_bias;    // [E][H] bf16, or nullptr
    const uint32_t* special;    // [E][2]: 1 if a projection holds an E8M0 byte 0 or 255
    const float* logits;        // [M][E]
    const uint16_t* x;          // [M][H] bf16 layer input, or nullptr: normalise resid
    uint16_t* resid;            // [M][H] bf16 residual in, result out
    float* h;                   // workspace [M][kmax][I]
    float* ypart;               // workspace [M][kmax][H]
    unsigned* done;             // [kMaxUnits] gate_up slab-pairs finished per unit (zero between calls)
    unsigned* hmax;             // [kMaxUnits][kMaxTokens] bits of max |h| (zero between calls)
    unsigned* slab_cnt;         // [H/16] units finished per down slab (zero between calls)
    unsigned* exit_cnt;         // [1] CTAs finished (zero between calls)
    int* status;                // device status word
    int* nu_out;                // distinct experts of this call (written by CTA 0)
    float* out_f32;             // [M][H] fp32 result before the bf16 rounding, or nullptr
    long long gu_expert_bytes, dn_expert_bytes;
    int gu_slab_bytes, dn_slab_bytes;
    int H, I, E, M, k, kmax, mmax, group;
    int nslots, slot_bytes;
};

// Counters of one handle: done | hmax | slab_cnt | exit.
inline size_t counter_words(int H) { return kMaxUnits + kMaxUnits * kMaxTokens + H / kSlabRows + 1; }

// Launch the layer kernel on `stream` (programmatic dependent launch towards
// the preceding kernel).  grid = one CTA per SM.
cudaError_t launch_layer(const LayerParams& p, int fmt, int grid, cudaStream_t stream);
// Dynamic shared memory the layer kernel needs, and its one-time set-up.
size_t layer_smem_bytes(const LayerParams& p);
cudaError_t prepare_layer_kernel(int fmt, int group, size_t smem, int* blocks_per_sm);

// Caller layout -> slabs for E experts of one projection ([E][N][K/2] codes,
// [E][N][K/32] u8 or [E][N][K/group] fp16 scales).  special[e * 2 + proj]
// gets 1 if an E8M0 byte is 0 or 255.
cudaError_t launch_repack(int fmt, int group, const uint8_t* codes, const uint8_t* scales, int E,
                          int N, int K, uint8_t* out, long long expert_bytes, int slab_bytes,
                          uint32_t* special, int proj, cudaStream_t stream);

// Record the calling thread's error message (read by moe_last_error) and
// return `code`.
int set_error(int code, const char* fmt, ...);

// ------------------------------------------------------------------ batched
// Calls with M > kMaxTokens run per-expert grouped GEMMs on the tensor cores
// (tcgen05.mma kind::mxf4: MXFP4 weights x MXFP4-quantised activations, fp32
// accumulators in tensor memory).  Weights are kept a second time in a "tile"
// layout made for that instruction.
//
// Tile layout of one projection W [N][K] (N, K multiples of 64).  Row tile t
// covers rows 128t .. 128t + R_t - 1 (R_t = 128, or N % 128 for the last one),
// k-step s covers K = 64s .. 64s + 63.
//   codes  at t*128*K/2 + s*R_t*32: an R_t x 32-byte block in the canonical
//          no-swizzle K-major order -- row r, byte b at
//          (r/8)*256 + (b/16)*128 + (r%8)*16 + b%16 (8x16-byte core matrices;
//          K-direction stride 128, row-group stride 256).
//   scales at N*K/2 + (t*C + c)*512, C = ceil(K/128): chunk c holds the E8M0
//          bytes of K-blocks 4c..4c+3 of the tile's 128 rows, row r = i + 32j
//          and block kb at i*16 + j*4 + kb (the order a 32x128-bit tensor-memory
//          copy replicated to the four lane quarters expects).
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
};

// Enqueue the batched layer (route, plan, quantise x, gate_up GEMM + SwiGLU +
// quantise h, down GEMM, combine) on `stream`; `grid` = SM count.
cudaError_t launch_batched(const BatchParams& p, int grid, cudaStream_t stream, int* launches);
cudaError_t prepare_batched_kernels();
// Caller layout [E][N][K/2] codes + [E][N][K/32] E8M0 -> tile layout (one projection
// per expert of N rows of a caller matrix with `src_rows` rows).  Tile row n comes
// from caller row n, or with `interleave` = I > 0 (N = 2I) from the interleaved
// gate_up order: row 64t + r (r < 64) or I + 64t + r - 64 of tile t.
cudaError_t launch_repack_tiles(const uint8_t* codes, const uint8_t* scales, int E, int src_rows,
                                int N, int K, int interleave, uint8_t* out, long long expert_bytes,
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
    const uint8_t* gu;          // interleaved tile layout: expert e at + e*gu_expert
    const uint8_t* dn;          // tile layout: expert e at + e*dn_expert
    long long gu_expert, dn_expert;
    const uint16_t* gu_bias;    // [E][2I] bf16 (gate | up), or nullptr
    const uint16_t* dn_bias;    // [E][H] bf16, or nullptr
    const float* logits;        // [M][E]
    const uint16_t* x;          // [M][H] bf16, or nullptr: RMS-normalise resid
    uint16_t* resid;            // [M][H] bf16 in/out
    float* part;                // [G][H][4] each CTA's fp32 copy of the expert output
    uint8_t* xt;                // x terms of the layer: [H/64][N rows x 32 B][ceil(H/128)][512]
    float* gpart;               // [G][128][4] gate/up partial sums of split-unit pieces
    unsigned* pflag;            // [G] piece partial published: the call's tag
    unsigned long long* xcnt;   // [1] x-term publications, G per call (only grows)
    unsigned long long* done;   // [1] output copies stored, G per call (only grows)
    int* status;
    int* nu_out;
    float* out_f32;             // [M][H] fp32 result before the bf16 rounding, or nullptr
    int H, I, E, M, k;
    int smem_bytes;             // dynamic shared memory of the layer kernel
    int spin_limit;             // polls before a cross-CTA wait gives up (kSpinLimit by default)
    int skip_cta;               // debug: this CTA skips its grid-barrier arrival (-1: none)
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
constexpr int kTcCounterWords = 2;   // xcnt, done (64-bit)
cudaError_t prepare_decode_tc(size_t smem);
size_t decode_tc_static_smem();
cudaError_t launch_decode_tc(const DecodeTcParams& p, size_t smem, int grid, cudaStream_t stream);

// Debug kernels.
// One expert projection of the tile layout back to fp32 in caller row order
// (gate_up: interleave = I, rows [0, I) gate and [I, 2I) up; down: 0).
cudaError_t launch_dequant_tiles(const uint8_t* tiles, int N, int K, int interleave, float* out,
                                 cudaStream_t stream);
cudaError_t launch_dequant(int fmt, int group, const uint8_t* slabs, int N, int K, int slab_bytes,
                           float* out, cudaStream_t stream);
cudaError_t launch_route(const float* logits, int M, int E, int k, int* idx, float* w,
                         cudaStream_t stream);

}  // namespace moe
