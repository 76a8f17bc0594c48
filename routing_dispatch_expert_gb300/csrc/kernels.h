// Internal launchers of the sm_103a kernels (host side). Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/moe.h"
#include "device_state.h"

namespace moe {

// SM count of the current device (per device; set up on first use there).
int num_sms();

// The current device and the driver context current on this thread (nullptr if none yet).
cudaError_t current_device(int* dev, const void** ctx);

// table's value for the current device and context, set up by init(T&) -> cudaError_t on first use.
template <class T, class Init>
cudaError_t per_device(PerDevice<T>& table, Init&& init, T* out) {
  int dev = 0;
  const void* ctx = nullptr;
  cudaError_t e = current_device(&dev, &ctx);
  if (e != cudaSuccess) return e;
  const int rc = table.get(dev, ctx, [&](T& v) { return static_cast<int>(init(v)); }, out);
  return rc == -1 ? cudaErrorInvalidDevice : static_cast<cudaError_t>(rc);
}

// EPLB placement plan on the host (eplb.cu).
int eplb_plan(const int64_t* load, int E, int n_cards, int n_redundant, int32_t* replicas, int32_t* slot_expert,
              int32_t* slot_replica, int32_t* replica_slot, double* card_load, std::string* err);

// Step 1: router GEMM, logits[T, E] = x[T, h] (bf16) . w_r[E, h]^T (fp32), fp32 accumulation.
cudaError_t launch_router_gemm(const void* x, const float* w_r, float* logits, int T, int h, int E,
                               cudaStream_t stream);

// Step 1: the fp32 router weight as three bf16 terms hi + mid + lo (w3 [3, E, h]) for the tensor-core
// router GEMM (grouped GEMM mode 2).
cudaError_t launch_split_router_weight(const float* w, void* w3, int64_t n, cudaStream_t stream);

// Step 1: top-k selection and route weights from fp32 logits, one warp per token.
struct TopkDesc {
  const float* logits;
  const float* bias;
  int32_t* topk_idx;
  float* topk_w;
  int T, E, k, n_group, topk_group, score, renorm;
  float routed_scale;
  // a router GEMM whose K range was split over CTAs leaves `splits` partial sums [splits, T, E]; the
  // top-k adds them in split order and writes the sums to `logits` (nullptr: logits are given)
  const float* partials = nullptr;
  int splits = 1;
};
cudaError_t launch_topk(const TopkDesc& d, cudaStream_t stream);

// Steps 2-3: per-block histogram, scan, stable ranks, and the dispatch copy.
int dispatch_blocks(int T);  // token blocks of the histogram / rank kernels
size_t dispatch_scratch_ints(int T, int E);
struct DispatchDesc {
  const void* x;
  const int32_t* topk_idx;
  const float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* inv_pos;
  int32_t* row_token;
  float* row_weight;
  void* xd;
  float* xd_scales;
  int32_t* scratch;  // dispatch_scratch_ints(T, E) ints
  int* status;
  int T, h, E, k;
  int shared;  // also write the T token rows for the shared expert
  int fp8;
  int capacity = 0;  // > 0: keep at most this many rows per expert (earliest tokens)
  // placement (all null: one slot per expert)
  int n_slots = 0;
  int max_replicas = 0;
  const int32_t* slot_expert = nullptr;
  const int32_t* slot_replica = nullptr;
  const int32_t* replicas = nullptr;
  const int32_t* replica_slot = nullptr;
  int32_t* expert_counts = nullptr;  // scratch [E]: kept rows per logical expert
};
cudaError_t launch_dispatch(const DispatchDesc& d, cudaStream_t stream);
// Steps 1-3 of a small batch as one cooperative launch (fused.cu): the router GEMM on the CUDA cores
// (E < 128, or E not a multiple of 32), top-k, counts, offsets, rows and the dispatch copy. Dropless,
// one slot per expert, T <= kFusedMaxT, E <= 256.
constexpr int kFusedMaxT = 4096;
bool fused_route_dispatch_supported(int T, int E);
struct FusedRouteDispatchDesc {
  const void* x;
  const float* w_router;
  TopkDesc tk;  // logits (out), bias, topk_idx, topk_w and the routing shape
  int32_t* counts;
  int32_t* offsets;
  int32_t* inv_pos;
  int32_t* row_token;
  float* row_weight;
  void* xd;
  float* xd_scales;
  int h, shared, fp8;
  unsigned int* barrier;  // zeroed before the launch
  int* status;
};
cudaError_t launch_fused_route_dispatch(const FusedRouteDispatchDesc& d, cudaStream_t stream);

// Load balance of a step from its counts [S] and offsets [S + 1] (S <= 1024).
cudaError_t launch_balance(const int32_t* counts, const int32_t* offsets, int S, int64_t assignments,
                           moe_balance_stats* out, cudaStream_t stream);

// Step 3: grouped GEMM (tcgen05) of one projection.
struct GroupedGemmDesc {
  const void* A;  // [a_rows, K]
  int64_t a_rows;
  const void* B;   // [E, b_rows, K]
  const void* Bs;  // [b_rows, K] shared expert or nullptr
  int64_t b_rows;
  const int32_t* offsets;  // nullptr: a single group of rows [0, T) (router)
  const int32_t* slot_expert = nullptr;  // group -> logical expert (weights), nullptr: identity
  int n_experts = 0;                     // logical experts in B (0: E)
  int E, R, T, K, N, I;
  int mode;  // 0 gate/up -> H, 1 down -> yd, 2 router logits (fp32)
  int ksplit = 1;  // mode 2: B holds 3 bf16 terms of the fp32 weight, [3, N, K]
  int csplit = 1;  // mode 2: CTAs per output tile over disjoint K ranges; out = [csplit, T, ldo] partials
  void* out;
  int ldo;
  const float* row_weight;
  int* status;
  // CTA-pair kernel: a zeroed int from which the persistent pairs take tiles in index order
  // (nullptr: each pair walks a fixed stride). The single-CTA kernel ignores it.
  int* tile_ctr = nullptr;
};
cudaError_t launch_grouped_gemm_bf16(const GroupedGemmDesc& d, cudaStream_t stream, std::string* err);
// one bounded mbarrier wait that nothing completes: records MOE_STATUS_WAIT_TIMEOUT in *status
cudaError_t launch_wait_timeout_selftest(int* status, long long limit_cycles, cudaStream_t stream);
// The expert FFN projections (modes 0 and 1) on CTA pairs: 256 x 256 tiles, tcgen05.mma.cta_group::2.
cudaError_t launch_grouped_gemm_bf16_pair(const GroupedGemmDesc& d, cudaStream_t stream, std::string* err);

// Step 3, FP8 layer: block-scaled grouped GEMM (e4m3 operands, fp32 128x128 weight scales, 1x128
// activation scales). mode 0: H codes + 1x128 scales; mode 1: yd bf16 x row_weight.
struct GroupedGemmFp8Desc {
  const void* A;  // [a_rows, K] e4m3
  const float* a_scales;  // [a_rows, K/128]
  int64_t a_rows;
  const void* B;  // [E, b_rows, K] e4m3
  const float* b_scales;  // [E, b_rows/128, K/128]
  const void* Bs;  // [b_rows, K] shared expert or nullptr
  const float* bs_scales;
  int64_t b_rows;
  const int32_t* offsets;
  const int32_t* slot_expert = nullptr;
  int n_experts = 0;
  int E, R, T, K, N, I;
  int mode;
  void* out;
  float* out_scales;
  int ldo;
  const float* row_weight;
  int* status;
};
cudaError_t launch_grouped_gemm_fp8(const GroupedGemmFp8Desc& d, cudaStream_t stream, std::string* err);

// Step 3, NVFP4-weight layer: bf16 activations, expert weights as e2m1 codes [E, N, K/2], e4m3 block
// scales [E, N, K/16] (one per 16 elements along K) and fp32 matrix scales [E]; expanded to bf16 in
// shared memory and multiplied on the bf16 tensor cores. Modes 0 and 1 as the bf16 kernel.
struct GroupedGemmFp4Desc {
  const void* A;  // [a_rows, K] bf16
  int64_t a_rows;
  const void* Bq;        // [E, b_rows, K/2] codes
  const void* Bs;        // [E, b_rows, K/16] e4m3 block scales
  const float* Bg;       // [E] matrix scales
  const void* Bq_shared; // [b_rows, K/2] shared expert or nullptr
  const void* Bs_shared;
  const float* Bg_shared;
  int64_t b_rows;
  const int32_t* offsets;
  const int32_t* slot_expert = nullptr;
  int n_experts = 0;
  int E, R, T, K, N, I;
  int mode;
  void* out;
  int ldo;
  const float* row_weight;
  int* status;
};
cudaError_t launch_grouped_gemm_nvfp4(const GroupedGemmFp4Desc& d, cudaStream_t stream, std::string* err);
// NVFP4 quantisation of `batch` bf16 matrices [rows, cols] (cols % 256 == 0): the matrix amax is
// gathered in g itself, the blocks are quantised, then g is turned into the matrix scales.
cudaError_t launch_quantize_weights_nvfp4(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, void* s,
                                          float* g, cudaStream_t stream);

// Step 4: combine.
cudaError_t launch_combine(const void* yd, const int32_t* inv_pos, void* y, int T, int h, int k, int shared,
                           cudaStream_t stream);

// Static weight quantisation, 128x128 tiles.
cudaError_t launch_quantize_weights(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, float* s,
                                    cudaStream_t stream);

}  // namespace moe
