// Routing and dispatch of a small batch as one persistent kernel.
//
// Perplexity blog "Lower latency and higher throughput with multi-node DeepSeek deployment", "CUDA
// Graph", and TensorRT-LLM "DeepSeek R1 throughput on Blackwell", "Runtime optimizations": a decode
// step is bound by the number of kernel launches, not by its work, so its many small kernels are to be
// merged into few fixed-grid ones. For a batch of at most kFusedMaxT tokens of a layer whose router runs
// on the CUDA cores (E < 128, or E not a multiple of 32), the router GEMM, the top-k selection, the
// per-expert counts and offsets, the stable expert-major row of every (token, slot) and the dispatch
// copy run as one cooperative launch of one CTA per SM, in phases separated by a grid-wide barrier:
//   0  router logits (the same work units as router_small_e_kernel, two per CTA)
//   1  top-k of every token, one warp per token spread over the SMs (the same function as topk_kernel)
//   2  every CTA counts the experts of all T*k assignments, and separately of the tokens before its own
//      range, in shared memory; scans the counts into offsets (CTA 0 stores counts and offsets); and
//      places the assignments of its own tokens: row = offsets[e] + (earlier tokens choosing e), the
//      earlier tokens of its range found from per-warp ballot masks as in rank_kernel
//   3  the dispatch copy, one warp per 1024-element piece of a row (the same functions as the gather
//      kernels)
// Every float result comes from the same device functions as the standalone kernels, and the integer
// results (counts, offsets, rows) have one correct value each, so moe_forward gives bit for bit what the
// step entry points give. The grid barrier counts arrivals on a word that moe_forward zeroes before
// the launch; a CTA that waits longer than a bounded number of clocks records MOE_STATUS_WAIT_TIMEOUT
// and leaves (the others then time out too), so a lost CTA cannot hang the GPU.
#include "dispatch_impl.cuh"
#include "route_impl.cuh"

namespace moe {
namespace fz {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr int PART_FLOATS = 512;  // router partial sums of one 256-thread unit (8 warps x TPW x EMAX)

struct Args {
  const __nv_bfloat16* x;
  const float* w_router;
  int rg_emax, rg_kw;
  TopkDesc tk;
  int32_t* counts;
  int32_t* offsets;
  int32_t* inv_pos;
  int32_t* row_token;
  float* row_weight;
  void* xd;
  float* xd_scales;
  int h, shared, fp8;
  unsigned int* barrier;
  int* status;
  long long wait_limit;
};

// Grid-wide barrier number `n` (0, 1, ...): every CTA adds one arrival to *ctr and waits until
// (n + 1) * gridDim.x have arrived. The fences make the writes of every CTA before the barrier visible
// to every CTA after it. Bounded: returns false (and records the time-out) after `limit` clocks.
__device__ __forceinline__ bool grid_barrier(unsigned int* ctr, int n, int* status, long long limit) {
  __shared__ int ok_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(ctr, 1u);
    const unsigned int target = (unsigned int)(n + 1) * gridDim.x;
    const long long t0 = clock64();
    for (;;) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > limit) {
        atomicOr(status, MOE_STATUS_WAIT_TIMEOUT);
        ok = 0;
        break;
      }
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

template <int EMAX, int TPW>
__device__ __forceinline__ void router_phase(const Args& a, float* part_all) {
  const int unit = threadIdx.x >> 8, tid = threadIdx.x & 255;
  const int groups = rg::WARPS / a.rg_kw;
  const int nbx = (int)cdiv(a.tk.T, (int64_t)TPW * groups), nby = (int)cdiv(a.tk.E, EMAX);
  auto part = reinterpret_cast<float(*)[TPW][EMAX]>(part_all + unit * PART_FLOATS);
  for (int u = blockIdx.x * 2 + unit; u < nbx * nby; u += gridDim.x * 2)
    rg::router_unit<EMAX, TPW>(a.x, a.w_router, const_cast<float*>(a.tk.logits), a.tk.T, a.h, a.tk.E, a.rg_kw,
                               u % nbx, u / nbx, tid, part, 1 + unit);
}

// Exclusive scan of n <= 2 * THREADS values in place (two per thread); returns the total.
__device__ __forceinline__ int block_exclusive_scan(int32_t* v, int n, int32_t* warp_tot) {
  const int i0 = 2 * threadIdx.x;
  const int a = i0 < n ? v[i0] : 0, b = i0 + 1 < n ? v[i0 + 1] : 0;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = a + b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = lane < WARPS ? warp_tot[lane] : 0;
    int ix = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, ix, o);
      if (lane >= o) ix += u;
    }
    if (lane < WARPS) warp_tot[lane] = ix - x;
    if (lane == WARPS - 1) warp_tot[WARPS] = ix;
  }
  __syncthreads();
  const int excl = warp_tot[w] + incl - (a + b);
  if (i0 < n) v[i0] = excl;
  if (i0 + 1 < n) v[i0 + 1] = excl + a;
  const int total = warp_tot[WARPS];
  __syncthreads();
  return total;
}

template <int EPL>
__global__ void __launch_bounds__(THREADS, 1) route_dispatch_kernel(const Args a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.tk.T, E = a.tk.E, k = a.tk.k;
  int nbar = 0;

  // ---- phase 0: router logits
  {
    float* part_all = reinterpret_cast<float*>(smem);
    switch (a.rg_emax) {
      case 8: router_phase<8, 4>(a, part_all); break;
      case 16: router_phase<16, 2>(a, part_all); break;
      case 32: router_phase<32, 1>(a, part_all); break;
      default: router_phase<64, 1>(a, part_all); break;
    }
  }
  if (!grid_barrier(a.barrier, nbar++, a.status, a.wait_limit)) return;

  // ---- phase 1: top-k, one warp per token, consecutive tokens on different SMs (a token's selection is
  // a long chain of dependent warp operations, so a small batch finishes sooner with few warps per SM)
  {
    const tk::Slots<EPL> sl = tk::make_slots<EPL>(a.tk, lane);
    for (int t = warp * gridDim.x + blockIdx.x; t < T; t += gridDim.x * WARPS) tk::topk_token<EPL>(a.tk, sl, lane, t);
  }
  if (!grid_barrier(a.barrier, nbar++, a.status, a.wait_limit)) return;

  // ---- phase 2: counts, offsets and the rows of this CTA's tokens
  int32_t* cnt = reinterpret_cast<int32_t*>(smem);  // [E]: assignments per expert, then offsets
  int32_t* before = cnt + 1024;                      // [E]: assignments of tokens before this CTA's range
  int32_t* warp_tot = before + 1024;                 // [WARPS + 1]
  uint32_t* masks = reinterpret_cast<uint32_t*>(warp_tot + 64);  // [WARPS][E]
  int32_t* wbase = reinterpret_cast<int32_t*>(masks + WARPS * E);  // [WARPS][E]
  const int chunk = (int)cdiv(T, gridDim.x);
  const int t0 = min(T, (int)blockIdx.x * chunk), t1 = min(T, t0 + chunk);
  for (int e = threadIdx.x; e < E; e += THREADS) cnt[e] = before[e] = 0;
  __syncthreads();
  const int32_t* idx = a.tk.topk_idx;
  bool bad = false;
  for (int64_t i = threadIdx.x; i < (int64_t)T * k; i += THREADS) {
    const int e = __ldcg(idx + i);
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
      if (i < (int64_t)t0 * k) atomicAdd(&before[e], 1);
    } else if (i >= (int64_t)t0 * k && i < (int64_t)t1 * k) {
      bad = true;
    }
  }
  if (bad) atomicOr(a.status, MOE_STATUS_BAD_EXPERT_INDEX);
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e < E; e += THREADS) a.counts[e] = cnt[e];
  const int total = block_exclusive_scan(cnt, E, warp_tot);  // cnt now holds the offsets
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += THREADS) a.offsets[e] = cnt[e];
    if (threadIdx.x == 0) a.offsets[E] = total;
  }
  // this CTA's tokens, THREADS at a time: a token's rank inside expert e is the number of earlier
  // tokens choosing e (a token picks an expert at most once)
  for (int base = t0; base < t1; base += THREADS) {
    for (int i = threadIdx.x; i < WARPS * E; i += THREADS) masks[i] = 0;
    __syncthreads();
    const int t = base + threadIdx.x;
    const bool tv = t < t1;
    if (tv)
      for (int j = 0; j < k; ++j) {
        const int e = __ldcg(idx + (int64_t)t * k + j);
        if (e >= 0 && e < E) atomicOr(&masks[warp * E + e], 1u << lane);
      }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += THREADS) {
      int run = before[e];
      for (int ww = 0; ww < WARPS; ++ww) {
        wbase[ww * E + e] = run;
        run += __popc(masks[ww * E + e]);
      }
      before[e] = run;  // the next THREADS tokens start here
    }
    __syncthreads();
    if (tv) {
      const uint32_t lt = (1u << lane) - 1u;
      for (int j = 0; j < k; ++j) {
        const int e = __ldcg(idx + (int64_t)t * k + j);
        int row = -1;
        if (e >= 0 && e < E) {
          row = cnt[e] + wbase[warp * E + e] + __popc(masks[warp * E + e] & lt);
          a.row_token[row] = t;
          a.row_weight[row] = __ldcg(a.tk.topk_w + (int64_t)t * k + j);
        }
        a.inv_pos[(int64_t)t * k + j] = row;
      }
    }
    __syncthreads();
  }
  if (!grid_barrier(a.barrier, nbar++, a.status, a.wait_limit)) return;

  // ---- phase 3: the dispatch copy
  const int64_t warps_all = (int64_t)gridDim.x * WARPS;
  const int R = T * k;
  if (a.fp8) {
    const int64_t items = (int64_t)T * dp::fp8_items_per_row(a.h);
    for (int64_t it = (int64_t)blockIdx.x * WARPS + warp; it < items; it += warps_all)
      dp::gather_fp8_item(reinterpret_cast<const uint4*>(a.x), a.inv_pos, reinterpret_cast<uint8_t*>(a.xd),
                          a.xd_scales, a.h, k, R, a.shared, it, lane);
  } else {
    const int64_t items = (int64_t)T * dp::bf16_items_per_row(a.h);
    for (int64_t it = (int64_t)blockIdx.x * WARPS + warp; it < items; it += warps_all)
      dp::gather_bf16_item(reinterpret_cast<const uint4*>(a.x), a.inv_pos, reinterpret_cast<uint4*>(a.xd), a.h, k,
                           R, a.shared, it, lane);
  }
}

size_t smem_bytes(int E) {
  const size_t phase2 = sizeof(int32_t) * (1024 + 1024 + 64) + sizeof(uint32_t) * 2 * WARPS * (size_t)E;
  const size_t phase0 = sizeof(float) * 2 * PART_FLOATS;
  return phase2 > phase0 ? phase2 : phase0;
}

}  // namespace fz

bool fused_route_dispatch_supported(int T, int E) { return T > 0 && T <= kFusedMaxT && E <= 256; }

cudaError_t launch_fused_route_dispatch(const FusedRouteDispatchDesc& d, cudaStream_t stream) {
  const int epl = (d.tk.E + 31) / 32;
  const void* fn = epl <= 1   ? (const void*)fz::route_dispatch_kernel<1>
                   : epl <= 2 ? (const void*)fz::route_dispatch_kernel<2>
                   : epl <= 4 ? (const void*)fz::route_dispatch_kernel<4>
                              : (const void*)fz::route_dispatch_kernel<8>;
  const size_t smem = fz::smem_bytes(d.tk.E);
  // the shared-memory opt-in (above 48 KB for E > 160) and the co-resident grid, per device
  static PerDevice<int> blocks_table[4];
  const int which = epl <= 1 ? 0 : epl <= 2 ? 1 : epl <= 4 ? 2 : 3;
  int per_sm = 0;
  cudaError_t e = per_device<int>(
      blocks_table[which],
      [fn](int& v) {
        cudaError_t r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)fz::smem_bytes(256));
        if (r != cudaSuccess) return r;
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, fn, fz::THREADS, fz::smem_bytes(256));
        if (r == cudaSuccess && v < 1) r = cudaErrorInvalidConfiguration;
        return r;
      },
      &per_sm);
  if (e != cudaSuccess) return e;
  fz::Args a;
  a.x = reinterpret_cast<const __nv_bfloat16*>(d.x);
  a.w_router = d.w_router;
  const int chunks = d.h / 256;
  a.rg_kw = chunks >= rg::WARPS ? rg::WARPS : chunks >= 4 ? 4 : chunks >= 2 ? 2 : 1;
  a.rg_emax = d.tk.E <= 8 ? 8 : d.tk.E <= 16 ? 16 : d.tk.E <= 32 ? 32 : 64;
  a.tk = d.tk;
  a.counts = d.counts;
  a.offsets = d.offsets;
  a.inv_pos = d.inv_pos;
  a.row_token = d.row_token;
  a.row_weight = d.row_weight;
  a.xd = d.xd;
  a.xd_scales = d.xd_scales;
  a.h = d.h;
  a.shared = d.shared;
  a.fp8 = d.fp8;
  a.barrier = d.barrier;
  a.status = d.status;
  a.wait_limit = 2000000000LL;  // about a second of SM clock
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3((unsigned)num_sms());  // one CTA per SM (at most per_sm are co-resident)
  cfg.blockDim = dim3(fz::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  e = cudaLaunchKernelExC(&cfg, fn, args);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
