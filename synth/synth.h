/*
 * Seeded synthetic inputs for the MoE layer workloads: host and device implementations of one
 * counter-based generator. Holds no arithmetic of the MoE method itself; it only draws numbers.
 *
 * Generator: the SplitMix64 sequence (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014). Element i of stream (seed, stream) is the SplitMix64
 * output function applied to base + (i + 1) * 0x9E3779B97F4A7C15, where base is the output
 * function applied to seed ^ (stream << 32) ^ 0x243F6A8885A308D3.
 *
 * Normal draws: the sum of twelve uniform 16-bit integers taken from three consecutive words
 * (the Irwin-Hall construction with mean 0 and variance 1), as an exact fp32 value, times
 * sigma (one fp32 rounding), plus an optional per-column shift mu (one fp32 rounding), then
 * rounded to bf16 to nearest even where a bf16 tensor is asked for. Uniform draws: the top 24
 * bits of one word scaled to [0, 1) exactly, then u * (hi - lo) + lo with two fp32 roundings.
 * Every operation is an exact integer operation or one correctly rounded fp32 operation, so
 * the host and device implementations give identical bits.
 */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* Host: out[i] = element (offset + i) of the stream, i in [0, n). mu may be NULL; otherwise
 * element j gets mu[j % mu_len] added (a per-column shift of a row-major [rows, mu_len]). */
void syn_normal_bf16(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma, const float* mu,
                     int64_t mu_len, uint16_t* out);
void syn_normal_f32(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma, float* out);
void syn_uniform_f32(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float lo, float hi, float* out);

/* Device: the same streams written to device memory on a CUDA stream (cudaStream_t passed as
 * void*). Return 0 on success, a CUDA error code otherwise. */
int syn_normal_bf16_dev(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma, const float* mu_dev,
                        int64_t mu_len, uint16_t* out_dev, void* cuda_stream);
int syn_normal_f32_dev(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma, float* out_dev,
                       void* cuda_stream);
int syn_uniform_f32_dev(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float lo, float hi,
                        float* out_dev, void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif
