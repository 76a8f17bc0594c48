// Device code of the dispatch copy (step 2, inference guide 6.4, section 3.1: each token's hidden state
// is copied once per chosen expert; Perplexity "Quantization": FP8 activations are scaled per 1x128
// vector at run time), shared by the standalone gather kernels (dispatch.cu) and the fused
// small-batch route-and-dispatch kernel (fused.cu): a copied row, its e4m3 codes and its scales are the
// same on either path.
//
// The unit of work is one warp on one piece of one token's row (an item): 2 KB of a bf16 row, or 1024
// elements of a row quantised to e4m3. Splitting rows into items, instead of a warp per token, keeps
// enough loads in flight when there are few tokens (a decode batch of 256 has 256 rows).
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace dp {

constexpr int kBf16ItemVec = 128;  // uint4 (8 bf16 each) per bf16 item: 1024 elements
constexpr int kFp8ItemElems = 1024;

__host__ __device__ __forceinline__ int bf16_items_per_row(int h) { return (h / 8 + kBf16ItemVec - 1) / kBf16ItemVec; }
__host__ __device__ __forceinline__ int fp8_items_per_row(int h) { return (h + kFp8ItemElems - 1) / kFp8ItemElems; }

// Copy item `it` (token it / items-per-row, piece it % items-per-row) of x to the token's k rows
// (inv_pos[t, j] >= 0) and, with `shared`, to row R + t. Lane l moves uint4 c0 + l + 32 u, u < 4.
__device__ __forceinline__ void gather_bf16_item(const uint4* __restrict__ x, const int32_t* __restrict__ inv_pos,
                                                 uint4* __restrict__ xd, int h, int k, int R, int shared, int64_t it,
                                                 int lane) {
  const int per = bf16_items_per_row(h);
  const int64_t t = it / per;
  const int hv = h / 8;
  const int c0 = (int)(it - t * per) * kBf16ItemVec;
  const int my_row = lane < k ? inv_pos[t * k + lane] : -1;
  const uint4* src = x + t * hv;
  uint4 v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = c0 + lane + 32 * u;
    if (c < hv) v[u] = src[c];
  }
  for (int j = 0; j < k; ++j) {
    const int r = __shfl_sync(0xffffffffu, my_row, j);
    if (r < 0) continue;
    uint4* dst = xd + (int64_t)r * hv;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + lane + 32 * u;
      if (c < hv) dst[c] = v[u];
    }
  }
  if (shared) {
    uint4* dst = xd + (int64_t)(R + t) * hv;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + lane + 32 * u;
      if (c < hv) dst[c] = v[u];
    }
  }
}

// FP8 item: 1024 elements of token t's row in passes of 256 (lanes 0-15 one 128-element block, 16-31
// the next); every block is quantised once (amax over its 16 lanes, scale = amax / 448, 1 for an
// all-zero block, codes e4m3(v / scale) rounded to nearest even with saturation), then its codes and
// scale are written to the token's k rows (and the shared expert's row).
__device__ __forceinline__ void gather_fp8_item(const uint4* __restrict__ x, const int32_t* __restrict__ inv_pos,
                                                uint8_t* __restrict__ xd, float* __restrict__ xs, int h, int k, int R,
                                                int shared, int64_t it, int lane) {
  const int per = fp8_items_per_row(h);
  const int64_t t = it / per;
  const int hv = h / 8;
  const int hb = h / 128;
  const int e0 = (int)(it - t * per) * kFp8ItemElems;
  const int my_row = lane < k ? inv_pos[t * k + lane] : -1;
  const uint4* src = x + t * hv;
  for (int p = 0; p < kFp8ItemElems / 256 && e0 + 256 * p < h; ++p) {
    const int c = (e0 + 256 * p) / 8 + lane;  // this lane's uint4 of the pass
    const uint4 v = src[c];
    const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                        bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint32_t q[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t code = __nv_cvt_float_to_fp8(__fdiv_rn(f[i], scale), __NV_SATFINITE, __NV_E4M3);
      q[i / 4] |= code << (8 * (i % 4));
    }
    const uint2 qv = make_uint2(q[0], q[1]);
    const int blk = (c * 8) / 128;
    const bool scale_writer = (lane & 15) == 0;
    for (int j = 0; j <= k; ++j) {
      int r;
      if (j < k) {
        r = __shfl_sync(0xffffffffu, my_row, j);
        if (r < 0) continue;
      } else {
        if (!shared) break;
        r = R + (int)t;
      }
      *reinterpret_cast<uint2*>(xd + (int64_t)r * h + c * 8) = qv;
      if (scale_writer) xs[(int64_t)r * hb + blk] = scale;
    }
  }
}

}  // namespace dp
}  // namespace moe
