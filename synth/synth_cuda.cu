/*
 * Seeded synthetic inputs, GPU side.
 *
 * Test and benchmark infrastructure only.  It computes the same values as
 * synth_host.c (see the definition there: SplitMix64 outputs, an Irwin-Hall
 * sum of four 32-bit uniforms, one int64->fp32 conversion and one fp32
 * multiply, each rounded to nearest even, then round-to-nearest-even to
 * binary16 or bfloat16).  It is compiled into its own library and shares no
 * code with the optimizer-step kernels.
 */
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__device__ __forceinline__ float value_at(uint64_t key, uint64_t i, float scale)
{
    uint64_t a = mix64(key + (2u * i + 1u) * kGamma);
    uint64_t b = mix64(key + (2u * i + 2u) * kGamma);
    uint64_t s = (a & 0xFFFFFFFFULL) + (a >> 32) + (b & 0xFFFFFFFFULL) + (b >> 32);
    long long c = (long long)s - 8589934590LL;
    return __fmul_rn(__ll2float_rn(c), scale);
}

__global__ void fill_f32_kernel(uint64_t key, uint64_t first, int64_t n, float scale, float *out)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = value_at(key, first + (uint64_t)i, scale);
}

__global__ void fill_half_kernel(uint64_t key, uint64_t first, int64_t n, float scale, int dtype,
                                 uint16_t *out)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        float x = value_at(key, first + (uint64_t)i, scale);
        out[i] = dtype == 0 ? __half_as_ushort(__float2half_rn(x))
                            : __bfloat16_as_ushort(__float2bfloat16_rn(x));
    }
}

__global__ void round_half_kernel(const float *x, int64_t n, int dtype, uint16_t *out)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = dtype == 0 ? __half_as_ushort(__float2half_rn(x[i]))
                            : __bfloat16_as_ushort(__float2bfloat16_rn(x[i]));
}

unsigned grid_for(int64_t n)
{
    int64_t blocks = (n + 255) / 256;
    return (unsigned)(blocks < 152 * 16 ? (blocks > 0 ? blocks : 1) : 152 * 16);
}

} // namespace

extern "C" {

/* All pointers are device pointers; n may be 0.  Returns a cudaError_t. */
int synth_gpu_fill_f32(uint64_t key, uint64_t first, int64_t n, float scale, float *out,
                       cudaStream_t stream)
{
    if (n <= 0)
        return 0;
    fill_f32_kernel<<<grid_for(n), 256, 0, stream>>>(key, first, n, scale, out);
    return (int)cudaGetLastError();
}

int synth_gpu_fill_half(uint64_t key, uint64_t first, int64_t n, float scale, int dtype,
                        uint16_t *out, cudaStream_t stream)
{
    if (n <= 0)
        return 0;
    fill_half_kernel<<<grid_for(n), 256, 0, stream>>>(key, first, n, scale, dtype, out);
    return (int)cudaGetLastError();
}

int synth_gpu_round_half(const float *x, int64_t n, int dtype, uint16_t *out, cudaStream_t stream)
{
    if (n <= 0)
        return 0;
    round_half_kernel<<<grid_for(n), 256, 0, stream>>>(x, n, dtype, out);
    return (int)cudaGetLastError();
}

} // extern "C"
