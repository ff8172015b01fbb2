// moe_internal.h -- declarations shared by the C-ABI layer (moe_api.cu) and
// the kernels (moe_decode.cu).  Not part of the public interface.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr int kMaxTokens = 4;      // decode M
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 256;
constexpr int kMaxUnits = kMaxTokens * kMaxTopK;   // distinct experts of one layer
constexpr int kMaxK = 4096;        // largest H or I
constexpr int kThreads = 384;      // threads per CTA of the decode kernels
constexpr int kRowsPerItem = 8;    // rows of one work item (4 gate/up pairs, or 8 down rows)

enum { FMT_MXFP4 = 1, FMT_INT4 = 2 };

// One layer's resident weights and the per-call pointers of a decode forward.
struct LayerParams {
    const uint8_t* gu_codes;   // [E][2I][H/2]
    const uint8_t* gu_scales;  // [E][2I][sbh] bytes per row
    const uint16_t* gu_bias;   // [E][2I] bf16, or nullptr
    const uint8_t* dn_codes;   // [E][H][I/2]
    const uint8_t* dn_scales;  // [E][H][sbi]
    const uint16_t* dn_bias;   // [E][H] bf16, or nullptr
    const float* logits;       // [M][E]
    const uint16_t* x;         // [M][H] bf16 layer input, or nullptr: normalise resid
    uint16_t* resid;           // [M][H] bf16 residual in, result out
    float* h;                  // workspace [M][kmax][I]
    float* ypart;              // workspace [M][kmax][H]
    unsigned int* tile_count;  // workspace [H/8] arrival counters (zero between calls)
    int* nu_out;               // distinct experts of this call (written by CTA 0)
    int H, I, E, M, k, kmax, group;
    int sbh, sbi;              // scale bytes per row of gate_up / down
};

// Launch the two kernels of one decode layer on `stream` (programmatic
// dependent launch between them and towards the preceding kernel).
cudaError_t launch_layer(const LayerParams& p, int fmt, int num_sms, cudaStream_t stream);

// Debug kernels.
cudaError_t launch_dequant(int fmt, const uint8_t* codes, const uint8_t* scales, int N, int K,
                           int group, float* out, cudaStream_t stream);
cudaError_t launch_route(const float* logits, int M, int E, int k, int* idx, float* w,
                         cudaStream_t stream);

}  // namespace moe
