// Step 1 of the layer: router scores and top-k selection.
//
// Ultralytics glossary "Expert Parallelism", "How tokens move across GPUs", step 1: the router
// scores every token against every expert and keeps the k best. TensorRT-LLM "DeepSeek R1
// throughput on Blackwell", "RouterGEMM mixed I/O": bf16 activations in, fp32 logits out, no cast
// kernel; "Top-K kernel fusion": groups first, then the top experts inside them, with a bias and a
// scaling factor, as one fused kernel. Perplexity "MoE Router": Mixtral routing is the special case
// top-k-group = all groups; the sparse kernels consume indices and scores directly.
//
// Readings where the pages are silent: the group score is the sum of the two largest biased scores
// of the group; ties go to the lower expert (and group) index; the sigmoid is evaluated in fp64 and
// rounded once to fp32, and the selection key is that fp32 value plus the bias in fp32, so the
// selection is a deterministic function of the fp32 logits (the kernel decides on fp32-evaluated keys
// and re-decides on the exact ones whenever a gap is too small to be certain); softmax layers select
// on the logits.
#include "route_impl.cuh"

namespace moe {

namespace rg {
template <int EMAX, int TPW>
__global__ void __launch_bounds__(THREADS) router_small_e_kernel(const __nv_bfloat16* __restrict__ x,
                                                                 const float* __restrict__ w, float* __restrict__ out,
                                                                 int T, int h, int E, int kw) {
  __shared__ float part[WARPS][TPW][EMAX];
  router_unit<EMAX, TPW>(x, w, out, T, h, E, kw, blockIdx.x, blockIdx.y, threadIdx.x, part, 0);
}
}  // namespace rg

cudaError_t launch_router_gemm(const void* x, const float* w_r, float* logits, int T, int h, int E,
                               cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  const int chunks = h / 256;
  const int kw = chunks >= rg::WARPS ? rg::WARPS : chunks >= 4 ? 4 : chunks >= 2 ? 2 : 1;
  const int groups = rg::WARPS / kw;
#define RG_LAUNCH(EM, TP)                                                                                     \
  rg::router_small_e_kernel<EM, TP><<<dim3((unsigned)cdiv(T, (int64_t)TP * groups), (unsigned)cdiv(E, EM)), \
                                      rg::THREADS, 0, stream>>>(xb, w_r, logits, T, h, E, kw)
  if (E <= 8)
    RG_LAUNCH(8, 4);
  else if (E <= 16)
    RG_LAUNCH(16, 2);
  else if (E <= 32)
    RG_LAUNCH(32, 1);
  else
    RG_LAUNCH(64, 1);
#undef RG_LAUNCH
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// The fp32 router weight as three bf16 terms for the tensor-core router GEMM: hi = bf16(w),
// mid = bf16(w - hi), lo = bf16(w - hi - mid). Each difference is exact in fp32, so hi + mid + lo
// carries 24 significant bits of w (the fp32 significand).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) split_router_weight_kernel(const float* __restrict__ w,
                                                                  __nv_bfloat16* __restrict__ w3, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = __fsub_rn(v, __bfloat162float(hi));
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    w3[i] = hi;
    w3[n + i] = mid;
    w3[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

cudaError_t launch_split_router_weight(const float* w, void* w3, int64_t n, cudaStream_t stream) {
  int64_t blocks = cdiv(n, 256);
  if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
  split_router_weight_kernel<<<(unsigned)blocks, 256, 0, stream>>>(w, reinterpret_cast<__nv_bfloat16*>(w3), n);
  return cudaGetLastError();
}

namespace tk {
template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const TopkDesc d) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const Slots<EPL> sl = make_slots<EPL>(d, lane);
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < d.T; t += warps) topk_token<EPL>(d, sl, lane, t);
}
}  // namespace tk

cudaError_t launch_topk(const TopkDesc& d, cudaStream_t stream) {
  if (d.T == 0) return cudaSuccess;
  // a token's selection is a long chain of dependent warp operations: a small batch spreads its tokens
  // over the SMs two warps per CTA (few warps per SM, each issuing at a full sub-partition's rate), a
  // large one packs eight warps per CTA
  const int threads = d.T <= 8192 ? 64 : 256;
  int64_t blocks = cdiv(d.T, threads / 32);
  if (blocks > (int64_t)num_sms() * 16) blocks = (int64_t)num_sms() * 16;
  const int epl = (d.E + 31) / 32;
  if (epl <= 1)
    tk::topk_kernel<1><<<(unsigned)blocks, threads, 0, stream>>>(d);
  else if (epl <= 2)
    tk::topk_kernel<2><<<(unsigned)blocks, threads, 0, stream>>>(d);
  else if (epl <= 4)
    tk::topk_kernel<4><<<(unsigned)blocks, threads, 0, stream>>>(d);
  else if (epl <= 8)
    tk::topk_kernel<8><<<(unsigned)blocks, threads, 0, stream>>>(d);
  else if (epl <= 16)
    tk::topk_kernel<16><<<(unsigned)blocks, threads, 0, stream>>>(d);
  else
    tk::topk_kernel<32><<<(unsigned)blocks, threads, 0, stream>>>(d);
  return cudaGetLastError();
}

}  // namespace moe
