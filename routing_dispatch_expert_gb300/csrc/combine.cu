// Step 4 of the layer: combine, and the static FP8 weight quantiser.
//
// Ultralytics glossary "Expert Parallelism", step 4, and inference guide 6.4, section 3.1, step 4:
// expert outputs return to their token and are summed with the route weights. Guide 6.4,
// section 7: the shared expert acts like one more expert every token picks (weight 1). The route
// weights were already applied in the down-projection epilogue, so combine is a gather-sum:
//   y[t] = bf16( sum_j yd[inv_pos[t, j]] + yd[T*k + t] ),  fp32 in slot order, rounded once.
//
// Perplexity "Quantization": weights are quantised statically per 128x128 tile.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace cb {

__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ yd, const int32_t* __restrict__ inv_pos,
                                                      uint4* __restrict__ y, int T, int h, int k, int R, int shared) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int hv = h / 8;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const int my_row = lane < k ? inv_pos[(int64_t)t * k + lane] : -1;
    for (int c = lane; c < hv; c += 64) {
      const bool two = c + 32 < hv;
      float acc[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
      auto add = [&](int r) {
        const uint4* src = yd + (int64_t)r * hv;
        uint4 v0 = src[c];
        uint4 v1 = two ? src[c + 32] : make_uint4(0, 0, 0, 0);
        const uint32_t a[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[u][2 * i] += bf16_lo(a[4 * u + i]);
            acc[u][2 * i + 1] += bf16_hi(a[4 * u + i]);
          }
      };
#pragma unroll 4
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_row, j);
        if (r >= 0) add(r);
      }
      if (shared) add(R + t);
      uint4* dst = y + (int64_t)t * hv;
      dst[c] = make_uint4(pack_bf16x2(acc[0][0], acc[0][1]), pack_bf16x2(acc[0][2], acc[0][3]),
                          pack_bf16x2(acc[0][4], acc[0][5]), pack_bf16x2(acc[0][6], acc[0][7]));
      if (two)
        dst[c + 32] = make_uint4(pack_bf16x2(acc[1][0], acc[1][1]), pack_bf16x2(acc[1][2], acc[1][3]),
                                 pack_bf16x2(acc[1][4], acc[1][5]), pack_bf16x2(acc[1][6], acc[1][7]));
    }
  }
}

// k <= KMAX: all k (+1 shared) rows of a 256-element chunk are loaded before any is added, so a warp
// keeps k + 1 independent 16-byte loads per lane in flight; the sum is still taken in slot order. The
// unit of work is one warp on PIECE consecutive 256-element chunks of one token's row, so that a batch
// of few tokens (decode) still spreads over every SM.
constexpr int PIECE = 4;
template <int KMAX>
__global__ void __launch_bounds__(256) combine_small_k_kernel(const uint4* __restrict__ yd,
                                                              const int32_t* __restrict__ inv_pos,
                                                              uint4* __restrict__ y, int T, int h, int k, int R,
                                                              int shared) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (gridDim.x * blockDim.x) >> 5;
  const int hv = h / 8;
  const int per = (hv / 32 + PIECE - 1) / PIECE;  // pieces per row (h is a multiple of 256)
  for (int64_t it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < (int64_t)T * per; it += warps) {
    const int t = (int)(it / per);
    const int c_lo = (int)(it - (int64_t)t * per) * PIECE * 32;
    const int c_hi = min(hv, c_lo + PIECE * 32);
    const int my_row = lane < k ? inv_pos[(int64_t)t * k + lane] : -1;
    int rows[KMAX + 1];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) rows[j] = __shfl_sync(0xffffffffu, my_row, j);  // -1 past k
    rows[KMAX] = shared ? R + t : -1;
    for (int c = c_lo + lane; c < c_hi; c += 32) {
      uint4 v[KMAX + 1];
#pragma unroll
      for (int j = 0; j <= KMAX; ++j)
        v[j] = rows[j] >= 0 ? yd[(int64_t)rows[j] * hv + c] : make_uint4(0, 0, 0, 0);
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j <= KMAX; ++j) {
        if (rows[j] < 0) continue;
        const uint32_t a[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] += bf16_lo(a[i]);
          acc[2 * i + 1] += bf16_hi(a[i]);
        }
      }
      y[(int64_t)t * hv + c] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                          pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
  }
}

// one CTA per 128x128 tile: amax, scale = amax / 448 (1 if zero), codes rounded to nearest even
__global__ void __launch_bounds__(256) quantize_weight_kernel(const uint4* __restrict__ w, int64_t rows, int64_t cols,
                                                              uint2* __restrict__ q, float* __restrict__ s) {
  __shared__ float red[8];
  const int64_t tiles_c = cols / 128, tiles_r = rows / 128;
  const int64_t tile = blockIdx.x;
  const int64_t b = tile / (tiles_r * tiles_c);
  const int64_t tr = (tile / tiles_c) % tiles_r, tc = tile % tiles_c;
  const int64_t cv = cols / 8;  // uint4 per row
  const uint4* base = w + b * rows * cv + tr * 128 * cv + tc * 16;
  uint4 v[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = threadIdx.x + 256 * i;  // 2048 uint4 per tile: row e / 16, chunk e % 16
    v[i] = base[(e / 16) * cv + (e % 16)];
    const uint32_t a[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(a[j])), fabsf(bf16_hi(a[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) s[tile] = scale;
  uint2* qbase = q + b * rows * cv + tr * 128 * cv + tc * 16;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = threadIdx.x + 256 * i;
    const uint32_t a[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t out[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(bf16_lo(a[j]), scale), __NV_SATFINITE, __NV_E4M3);
      uint32_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(bf16_hi(a[j]), scale), __NV_SATFINITE, __NV_E4M3);
      out[j / 2] |= (c0 | (c1 << 8)) << (16 * (j % 2));
    }
    qbase[(e / 16) * cv + (e % 16)] = make_uint2(out[0], out[1]);
  }
}

}  // namespace cb

cudaError_t launch_combine(const void* yd, const int32_t* inv_pos, void* y, int T, int h, int k, int shared,
                           cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  // small k: one warp per piece of a row; larger k: one warp per token
  const int64_t units = k <= 8 ? (int64_t)T * ((h / 256 + cb::PIECE - 1) / cb::PIECE) : T;
  int64_t blocks = cdiv(units, 8);
  if (blocks > (int64_t)num_sms() * 16) blocks = (int64_t)num_sms() * 16;
  if (k <= 8)
    cb::combine_small_k_kernel<8><<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(yd), inv_pos,
                                                                         reinterpret_cast<uint4*>(y), T, h, k, T * k,
                                                                         shared);
  else
    cb::combine_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(yd), inv_pos,
                                                              reinterpret_cast<uint4*>(y), T, h, k, T * k, shared);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weights(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, float* s,
                                    cudaStream_t stream) {
  const int64_t tiles = batch * (rows / 128) * (cols / 128);
  if (tiles == 0) return cudaSuccess;
  cb::quantize_weight_kernel<<<(unsigned)tiles, 256, 0, stream>>>(reinterpret_cast<const uint4*>(w), rows, cols,
                                                                   reinterpret_cast<uint2*>(q), s);
  return cudaGetLastError();
}

}  // namespace moe
