// bf16 GEMV decode stand-in for the interference measurement (see kvx_standin.h).
//
// One warp per row, grid-stride over rows. The default grid gives each warp
// about 8 rows, so CTAs come and go like a real decode kernel's and the
// scheduler can place them around other kernels' CTAs. A row of 2,560 bf16 is
// 320 16-byte words:
// each lane issues its 10 loads back to back (5 KiB per warp in flight), then
// multiplies with x, kept in shared memory as fp32, and the warp reduces with
// shuffles. The weights are read once with no reuse, so the loads bypass L1.
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "kvx_standin.h"

namespace {

constexpr int kMaxWordsPerLane = 16;  // cols <= 16 * 32 * 8 = 4096

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(256) kvx_standin_gemv_kernel(const uint4 *__restrict__ W,
                                                               const uint16_t *__restrict__ x,
                                                               float *__restrict__ y, uint64_t rows,
                                                               uint32_t cols)
{
    extern __shared__ float xs[];
    for (uint32_t i = threadIdx.x; i < cols; i += blockDim.x)
        xs[i] = __uint_as_float((uint32_t)x[i] << 16);
    __syncthreads();

    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t words = cols >> 3;          // 16-byte words per row
    const uint32_t per_lane = words >> 5;      // cols is a multiple of 256
    const uint64_t wpb = blockDim.x >> 5;
    const uint64_t nwarps = (uint64_t)gridDim.x * wpb;
    for (uint64_t r = (uint64_t)blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += nwarps) {
        const uint4 *row = W + r * words;
        uint4 v[kMaxWordsPerLane];
#pragma unroll
        for (int j = 0; j < kMaxWordsPerLane; ++j)
            if ((uint32_t)j < per_lane)
                v[j] = ld_stream(row + j * 32 + lane);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxWordsPerLane; ++j) {
            if ((uint32_t)j < per_lane) {
                const float *xv = xs + (j * 32 + lane) * 8;
                acc = fmaf(bf16_lo(v[j].x), xv[0], acc);
                acc = fmaf(bf16_hi(v[j].x), xv[1], acc);
                acc = fmaf(bf16_lo(v[j].y), xv[2], acc);
                acc = fmaf(bf16_hi(v[j].y), xv[3], acc);
                acc = fmaf(bf16_lo(v[j].z), xv[4], acc);
                acc = fmaf(bf16_hi(v[j].z), xv[5], acc);
                acc = fmaf(bf16_lo(v[j].w), xv[6], acc);
                acc = fmaf(bf16_hi(v[j].w), xv[7], acc);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0)
            y[r] = acc;
    }
}

}  // namespace

extern "C" kvx_status kvx_standin_gemv_bf16(uint64_t W, uint64_t x, uint64_t y, uint64_t rows,
                                            uint32_t cols, int ctas, void *stream)
{
    if (!W || !x || !y || rows == 0 || cols == 0 || cols % 256 || cols > 4096 || ctas < 0)
        return KVX_ERR_INVALID_ARG;
    if ((W | x | y) & 15u)
        return KVX_ERR_ALIGN;
    if (ctas == 0) {  // 8 warps per CTA, about 8 rows per warp
        const uint64_t want = (rows + 63) / 64;
        ctas = (int)(want < (1u << 30) ? want : (1u << 30));
    }
    kvx_standin_gemv_kernel<<<ctas, 256, cols * sizeof(float), static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint4 *>(W), reinterpret_cast<const uint16_t *>(x),
        reinterpret_cast<float *>(y), rows, cols);
    return cudaGetLastError() == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}
