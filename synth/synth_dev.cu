// Device implementation of the seeded generator declared in synth.h (same streams, same bits
// as synth.c: integer hashing plus correctly rounded fp32 operations only).
#include <cuda_runtime.h>

#include "synth.h"

#define SYN_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr unsigned long long kGolden = 0x9E3779B97F4A7C15ULL;

__host__ __device__ __forceinline__ unsigned long long mix(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ unsigned long long base_of(unsigned long long seed, unsigned stream) {
  return mix(seed ^ ((unsigned long long)stream << 32) ^ 0x243F6A8885A308D3ULL);
}

__device__ __forceinline__ float std_normal(unsigned long long base, unsigned long long i) {
  int s = 0;
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    unsigned long long z = mix(base + (3 * i + w + 1) * kGolden);
#pragma unroll
    for (int q = 0; q < 4; ++q) s += (int)((z >> (16 * q)) & 0xFFFFu);
  }
  s -= 393210;
  return __fmul_rn(__int2float_rn(s), 1.0f / 65536.0f);
}

__device__ __forceinline__ unsigned short to_bf16(float f) {
  unsigned u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (unsigned short)(u >> 16);
}

__global__ void normal_bf16_kernel(unsigned long long base, long long offset, long long n, float sigma,
                                   const float* __restrict__ mu, long long mu_len, unsigned short* __restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    unsigned long long g = (unsigned long long)(offset + i);
    float y = __fmul_rn(std_normal(base, g), sigma);
    if (mu) y = __fadd_rn(y, mu[g % (unsigned long long)mu_len]);
    out[i] = to_bf16(y);
  }
}

__global__ void normal_f32_kernel(unsigned long long base, long long offset, long long n, float sigma,
                                  float* __restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    out[i] = __fmul_rn(std_normal(base, (unsigned long long)(offset + i)), sigma);
}

__global__ void uniform_f32_kernel(unsigned long long base, long long offset, long long n, float lo, float span,
                                   float* __restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    unsigned long long z = mix(base + ((unsigned long long)(offset + i) + 1) * kGolden);
    float u = __fmul_rn(__ull2float_rn(z >> 40), 1.0f / 16777216.0f);
    out[i] = __fadd_rn(__fmul_rn(u, span), lo);
  }
}

unsigned grid_for(long long n) {
  long long b = (n + 255) / 256;
  if (b > 152LL * 64) b = 152LL * 64;
  if (b < 1) b = 1;
  return (unsigned)b;
}

}  // namespace

SYN_API int syn_normal_bf16_dev(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma,
                                const float* mu_dev, int64_t mu_len, uint16_t* out_dev, void* cuda_stream) {
  if (n <= 0) return 0;
  normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      base_of(seed, stream), offset, n, sigma, mu_dev, mu_len, (unsigned short*)out_dev);
  return (int)cudaGetLastError();
}

SYN_API int syn_normal_f32_dev(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma,
                               float* out_dev, void* cuda_stream) {
  if (n <= 0) return 0;
  normal_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(base_of(seed, stream), offset, n, sigma,
                                                                         out_dev);
  return (int)cudaGetLastError();
}

SYN_API int syn_uniform_f32_dev(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float lo, float hi,
                                float* out_dev, void* cuda_stream) {
  if (n <= 0) return 0;
  float span = hi - lo;
  uniform_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(base_of(seed, stream), offset, n, lo, span,
                                                                          out_dev);
  return (int)cudaGetLastError();
}
