// moe_loader.cu -- load-time conversions of checkpoint layouts into the
// caller layout the repack kernels take (rows [N] of K elements, gate rows
// before up rows).  They run once per layer on the device copy of the
// caller's tensors; nothing here is on the forward path.
//
// The pages verify the MXFP4 reader's orientation against the reference
// checkpoint ("Sovereign gpt-oss-20B (MXFP4) on Apple Silicon", section 3:
// "transpose orientation verified"); these conversions let a checkpoint that
// stores a projection in the other orientation ([K][N]), or gate and up rows
// alternating, be loaded as is.
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_internal.h"

namespace moe {
namespace {

// [E][K][N] 4-bit codes (two per byte, the element with the even index along
// N in the low nibble) -> [E][N][K] (the even index along K low).  One thread
// per output byte.
__global__ void transpose_nibbles_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E, int N,
                                         int K)
{
    const long long per = (long long)N * (K / 2), total = (long long)E * per;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
         g += (long long)gridDim.x * blockDim.x) {
        const long long e = g / per, r = g % per;
        const int n = (int)(r / (K / 2)), k = 2 * (int)(r % (K / 2));
        const uint8_t* s = src + e * per;
        const int sh = 4 * (n & 1);
        const uint32_t lo = (s[((long long)k * N + n) >> 1] >> sh) & 0xfu;
        const uint32_t hi = (s[((long long)(k + 1) * N + n) >> 1] >> sh) & 0xfu;
        dst[g] = (uint8_t)(lo | (hi << 4));
    }
}

// [E][R][C] elements of esz bytes -> [E][C][R].
__global__ void transpose_elems_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E, int R,
                                       int C, int esz)
{
    const long long per = (long long)R * C, total = (long long)E * per;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
         g += (long long)gridDim.x * blockDim.x) {
        const long long e = g / per, r = g % per;
        const int c = (int)(r / R), i = (int)(r % R);   // output element (c, i)
        const uint8_t* s = src + (e * per + (long long)i * C + c) * esz;
        uint8_t* d = dst + g * esz;
        for (int b = 0; b < esz; ++b)
            d[b] = s[b];
    }
}

// Rows of row_bytes bytes, per expert: gate/up alternating (source row 2j is
// gate row j, 2j + 1 up row j) -> gate rows 0 .. R/2-1, then up rows.
__global__ void deinterleave_rows_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E, int R,
                                         long long row_bytes)
{
    const long long per = (long long)R * row_bytes, total = (long long)E * per;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
         g += (long long)gridDim.x * blockDim.x) {
        const long long e = g / per, r = g % per;
        const int row = (int)(r / row_bytes);
        const long long b = r % row_bytes;
        const int srow = row < R / 2 ? 2 * row : 2 * (row - R / 2) + 1;
        dst[g] = src[e * per + (long long)srow * row_bytes + b];
    }
}

unsigned grid_for(long long n)
{
    const long long b = (n + 255) / 256;
    return (unsigned)(b < 65536 ? (b > 0 ? b : 1) : 65536);
}

}  // namespace

cudaError_t launch_transpose_nibbles(const uint8_t* src, uint8_t* dst, int E, int N, int K, cudaStream_t s)
{
    transpose_nibbles_kernel<<<grid_for((long long)E * N * (K / 2)), 256, 0, s>>>(src, dst, E, N, K);
    return cudaGetLastError();
}

cudaError_t launch_transpose_elems(const uint8_t* src, uint8_t* dst, int E, int R, int C, int esz, cudaStream_t s)
{
    transpose_elems_kernel<<<grid_for((long long)E * R * C), 256, 0, s>>>(src, dst, E, R, C, esz);
    return cudaGetLastError();
}

cudaError_t launch_deinterleave_rows(const uint8_t* src, uint8_t* dst, int E, int R, long long row_bytes,
                                     cudaStream_t s)
{
    deinterleave_rows_kernel<<<grid_for((long long)E * R * row_bytes), 256, 0, s>>>(src, dst, E, R, row_bytes);
    return cudaGetLastError();
}

}  // namespace moe
