/* Host implementation of the seeded generator declared in synth.h. */
#include "synth.h"

#include <string.h>

#define SYN_API __attribute__((visibility("default")))
#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t syn_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t syn_base(uint64_t seed, uint32_t stream) {
  return syn_mix(seed ^ ((uint64_t)stream << 32) ^ 0x243F6A8885A308D3ULL);
}

static uint64_t syn_word(uint64_t base, uint64_t i) { return syn_mix(base + (i + 1) * SYN_GOLDEN); }

/* Irwin-Hall: twelve uniform 16-bit draws, centred; exact in fp32 (|S| < 2^19). */
static float syn_std_normal(uint64_t base, uint64_t i) {
  int32_t s = 0;
  for (int w = 0; w < 3; ++w) {
    uint64_t z = syn_word(base, 3 * i + (uint64_t)w);
    for (int q = 0; q < 4; ++q) s += (int32_t)((z >> (16 * q)) & 0xFFFFu);
  }
  s -= 393210; /* 12 * 65535 / 2 */
  return (float)s * (1.0f / 65536.0f);
}

static uint16_t syn_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

SYN_API void syn_normal_bf16(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma,
                             const float* mu, int64_t mu_len, uint16_t* out) {
  uint64_t base = syn_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t g = (uint64_t)(offset + i);
    float v = syn_std_normal(base, g);
    float y = v * sigma;
    if (mu) {
      float m = mu[g % (uint64_t)mu_len];
      y = y + m;
    }
    out[i] = syn_f32_to_bf16(y);
  }
}

SYN_API void syn_normal_f32(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float sigma, float* out) {
  uint64_t base = syn_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float v = syn_std_normal(base, (uint64_t)(offset + i));
    out[i] = v * sigma;
  }
}

SYN_API void syn_uniform_f32(uint64_t seed, uint32_t stream, int64_t offset, int64_t n, float lo, float hi,
                             float* out) {
  uint64_t base = syn_base(seed, stream);
  float span = hi - lo;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float u = (float)(syn_word(base, (uint64_t)(offset + i)) >> 40) * (1.0f / 16777216.0f);
    float y = u * span;
    out[i] = y + lo;
  }
}
