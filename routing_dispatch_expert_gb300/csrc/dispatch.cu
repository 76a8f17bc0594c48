// Dispatch as a local permute.
//
// Perplexity "MoE Router": dense dispatch/combine needs the routing information aggregated per
// expert rather than per token. Inference guide 6.4, section 3.1, step 2: each token's hidden state is
// copied k times, once for each chosen expert. Perplexity "Quantization": activations are quantised
// at run time per 1x128 vector (FP8 layer).
//
// Four kernels, all deterministic (integer atomics only, whose results do not depend on order):
//   1. histogram   per 512-token block: counts of each expert      -> hist[block][E]
//   2. scan        one CTA: per-expert running sum over blocks, exclusive scan over experts
//                  -> counts (clamped to the capacity), offsets, and the within-expert rank of every
//                  (block, expert)
//   3. rank        per 512-token block: per-warp lane masks of each expert give every (token, slot)
//                  its row, rows of an expert in ascending token order -> inv_pos, row_token,
//                  row_weight
//   4. gather      one warp per item (a 1024-element piece of one token's row): the piece is read
//                  once and written to the token's k rows (and to the shared expert's row), as bf16
//                  or as e4m3 with 1x128 scales (dispatch_impl.cuh).
#include <cuda_fp8.h>

#include "common.cuh"
#include "dispatch_impl.cuh"
#include "kernels.h"

namespace moe {

namespace dp {
constexpr int TPB = 512;  // tokens per histogram / rank block
constexpr int WARPS = TPB / 32;

__global__ void __launch_bounds__(TPB) hist_kernel(const int32_t* __restrict__ idx, int T, int k, int E,
                                                   int32_t* __restrict__ hist, int* status) {
  extern __shared__ int32_t sh[];
  for (int e = threadIdx.x; e < E; e += TPB) sh[e] = 0;
  __syncthreads();
  const int64_t t = (int64_t)blockIdx.x * TPB + threadIdx.x;
  if (t < T) {
    bool bad = false;
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      if (e >= 0 && e < E)
        atomicAdd(&sh[e], 1);
      else
        bad = true;
    }
    if (bad) atomicOr(status, MOE_STATUS_BAD_EXPERT_INDEX);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += TPB) hist[(int64_t)blockIdx.x * E + e] = sh[e];
}

// hist[b][e] becomes the number of earlier tokens (blocks < b) that chose e, i.e. the rank within
// expert e of block b's first such token; counts are clamped to the capacity `cap`. With a placement
// the counts and offsets are per physical slot: replica i of an expert with R replicas and c kept rows
// gets the rows of ranks i, i + R, i + 2R, ... < c.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* __restrict__ hist, int nblk, int E, int cap,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int n_slots, const int32_t* __restrict__ slot_expert,
                                                    const int32_t* __restrict__ slot_replica,
                                                    const int32_t* __restrict__ replicas,
                                                    int32_t* __restrict__ expert_counts) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t kept[1024];
  const int e = threadIdx.x;  // E <= 1024, n_slots <= 1024
  int run = 0;
  if (e < E) {
    for (int b = 0; b < nblk; ++b) {
      int c = hist[(int64_t)b * E + e];
      hist[(int64_t)b * E + e] = run;
      run += c;
    }
    run = min(run, cap);
    if (n_slots == 0)
      counts[e] = run;
    else
      expert_counts[e] = kept[e] = run;
  }
  const int n = n_slots == 0 ? E : n_slots;
  if (n_slots != 0) {
    __syncthreads();
    run = 0;
    if (e < n_slots) {
      const int ex = slot_expert[e], i = slot_replica[e], r = replicas[ex], c = kept[ex];
      run = c > i ? (c - i + r - 1) / r : 0;
      counts[e] = run;
    }
  }
  // exclusive scan of run over experts
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = warp_tot[lane];
    int iv = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, iv, o);
      if (lane >= o) iv += u;
    }
    warp_tot[lane] = iv - v;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int excl = warp_tot[w] + incl - run;
  if (e < n) offsets[e] = excl;
  if (e == n - 1) offsets[n] = excl + run;
}

__global__ void __launch_bounds__(TPB) rank_kernel(const int32_t* __restrict__ idx, const float* __restrict__ topk_w,
                                                   const int32_t* __restrict__ base, const int32_t* __restrict__ offsets,
                                                   int T, int k, int E, int cap, int32_t* __restrict__ inv_pos,
                                                   int32_t* __restrict__ row_token, float* __restrict__ row_weight,
                                                   int n_slots, int max_replicas, const int32_t* __restrict__ replicas,
                                                   const int32_t* __restrict__ replica_slot) {
  extern __shared__ uint32_t smem[];
  uint32_t* masks = smem;                                        // [WARPS][E]
  int32_t* wbase = reinterpret_cast<int32_t*>(smem + WARPS * E);  // [WARPS][E]
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < WARPS * E; i += TPB) masks[i] = 0;
  __syncthreads();
  const int64_t t = (int64_t)blockIdx.x * TPB + threadIdx.x;
  const bool tv = t < T;
  if (tv)
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      if (e >= 0 && e < E) atomicOr(&masks[w * E + e], 1u << lane);
    }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += TPB) {
    int run = base[(int64_t)blockIdx.x * E + e];
    for (int ww = 0; ww < WARPS; ++ww) {
      wbase[ww * E + e] = run;
      run += __popc(masks[ww * E + e]);
    }
  }
  __syncthreads();
  if (tv) {
    const uint32_t lt = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      int row = -1;
      if (e >= 0 && e < E) {
        const int rank = wbase[w * E + e] + __popc(masks[w * E + e] & lt);  // earlier tokens choosing e
        if (rank < cap) {
          if (n_slots == 0) {
            row = offsets[e] + rank;
          } else {  // round-robin over the expert's replicas
            const int r = replicas[e];
            row = offsets[replica_slot[e * max_replicas + rank % r]] + rank / r;
          }
          row_token[row] = (int32_t)t;
          row_weight[row] = topk_w[t * k + j];
        }
      }
      inv_pos[t * k + j] = row;
    }
  }
}

// The dispatch copies: one warp per item (a piece of one token's row), items in token order.
__global__ void __launch_bounds__(256) gather_bf16_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv_pos,
                                                          uint4* __restrict__ xd, int T, int h, int k, int R,
                                                          int shared) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)T * bf16_items_per_row(h);
  for (int64_t it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += warps)
    gather_bf16_item(x, inv_pos, xd, h, k, R, shared, it, lane);
}

__global__ void __launch_bounds__(256) gather_fp8_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv_pos,
                                                         uint8_t* __restrict__ xd, float* __restrict__ xs, int T, int h,
                                                         int k, int R, int shared) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)T * fp8_items_per_row(h);
  for (int64_t it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += warps)
    gather_fp8_item(x, inv_pos, xd, xs, h, k, R, shared, it, lane);
}

// Load balance of one step from its counts (S <= 1024 experts or slots): the busiest expert's rows,
// the experts with rows, the kept rows (offsets[S]) and the dropped assignments, and busiest / mean.
__global__ void __launch_bounds__(1024) balance_kernel(const int32_t* __restrict__ counts,
                                                       const int32_t* __restrict__ offsets, int S, int64_t assignments,
                                                       moe_balance_stats* out) {
  __shared__ int32_t wmax[32];
  const int e = threadIdx.x, lane = e & 31, w = e >> 5;
  const int c = e < S ? counts[e] : 0;
  const int active = __syncthreads_count(c > 0);
  int m = c;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wmax[w] = m;
  __syncthreads();
  if (w == 0) {
    m = wmax[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
      const int kept = offsets[S];
      out->max_rows = m;
      out->active = active;
      out->kept = kept;
      out->dropped = (int32_t)(assignments - kept);
      // max / (kept / S) = max * S / kept: exact in fp64 (both factors below 2^31 and 2^10), one division
      out->max_over_mean = kept > 0 ? (float)((double)m * (double)S / (double)kept) : 0.f;
    }
  }
}

}  // namespace dp

cudaError_t launch_balance(const int32_t* counts, const int32_t* offsets, int S, int64_t assignments,
                           moe_balance_stats* out, cudaStream_t stream) {
  dp::balance_kernel<<<1, 1024, 0, stream>>>(counts, offsets, S, assignments, out);
  return cudaGetLastError();
}

int dispatch_blocks(int T) { return (int)cdiv(T, dp::TPB); }
size_t dispatch_scratch_ints(int T, int E) { return (size_t)dispatch_blocks(T) * (size_t)E; }

cudaError_t launch_dispatch(const DispatchDesc& d, cudaStream_t stream) {
  if (d.T == 0) {
    // no tokens: offsets must still describe E empty experts
    const int n = d.n_slots ? d.n_slots : d.E;
    cudaError_t e = cudaMemsetAsync(d.counts, 0, sizeof(int32_t) * n, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(d.offsets, 0, sizeof(int32_t) * (n + 1), stream);
    return e;
  }
  const int nblk = dispatch_blocks(d.T);
  dp::hist_kernel<<<nblk, dp::TPB, sizeof(int32_t) * d.E, stream>>>(d.topk_idx, d.T, d.k, d.E, d.scratch, d.status);
  const int cap = d.capacity > 0 ? d.capacity : 0x7fffffff;
  dp::scan_kernel<<<1, 1024, 0, stream>>>(d.scratch, nblk, d.E, cap, d.counts, d.offsets, d.n_slots, d.slot_expert,
                                          d.slot_replica, d.replicas, d.expert_counts);
  const size_t rank_smem = sizeof(uint32_t) * 2 * dp::WARPS * d.E;
  // the dynamic shared-memory opt-in (up to E = 1024) is a per-device function attribute
  static PerDevice<bool> attr;
  bool attr_set = false;
  cudaError_t ae = per_device<bool>(
      attr,
      [](bool& v) {
        const cudaError_t r = cudaFuncSetAttribute(dp::rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)(sizeof(uint32_t) * 2 * dp::WARPS * 1024));
        v = r == cudaSuccess;
        return r;
      },
      &attr_set);
  if (ae != cudaSuccess) return ae;
  dp::rank_kernel<<<nblk, dp::TPB, rank_smem, stream>>>(d.topk_idx, d.topk_w, d.scratch, d.offsets, d.T, d.k, d.E,
                                                         cap, d.inv_pos, d.row_token, d.row_weight, d.n_slots,
                                                         d.max_replicas, d.replicas, d.replica_slot);
  const int64_t items = (int64_t)d.T * (d.fp8 ? dp::fp8_items_per_row(d.h) : dp::bf16_items_per_row(d.h));
  int64_t blocks = cdiv(items, 8);
  if (blocks > (int64_t)num_sms() * 16) blocks = (int64_t)num_sms() * 16;
  const int R = d.T * d.k;
  if (d.fp8)
    dp::gather_fp8_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(d.x), d.inv_pos,
                                                                reinterpret_cast<uint8_t*>(d.xd), d.xd_scales, d.T,
                                                                d.h, d.k, R, d.shared);
  else
    dp::gather_bf16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(d.x), d.inv_pos,
                                                                 reinterpret_cast<uint4*>(d.xd), d.T, d.h, d.k, R,
                                                                 d.shared);
  return cudaGetLastError();
}

}  // namespace moe
