// C ABI of the library: argument checks, workspace layout and the launch sequence of each step.
// Declarations and the contract of every entry point are in include/moe.h.
#include <stdio.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <string>

#include "common.cuh"
#include "kernels.h"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_err;
std::atomic<uint64_t> g_launches{0};

void counted(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return MOE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int check_config(const moe_config* c) {
  if (!c) return fail(MOE_ERR_INVALID, "cfg is NULL");
  if (c->T < 0 || c->h <= 0 || c->E <= 0 || c->k <= 0 || c->I <= 0 || c->I_shared < 0)
    return fail(MOE_ERR_INVALID, "T must be >= 0 and h, E, k, I positive, I_shared >= 0");
  if (c->k > c->E || c->k > 32) return fail(MOE_ERR_INVALID, "k must lie in [1, min(E, 32)]");
  if (c->n_group < 1 || c->n_group > 32 || c->E % c->n_group != 0)
    return fail(MOE_ERR_INVALID, "n_group must lie in [1, 32] and divide E");
  if (c->topk_group < 1 || c->topk_group > c->n_group)
    return fail(MOE_ERR_INVALID, "topk_group must lie in [1, n_group]");
  if ((int64_t)c->topk_group * (c->E / c->n_group) < c->k)
    return fail(MOE_ERR_INVALID, "the kept groups hold fewer than k experts");
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return fail(MOE_ERR_INVALID, "unknown score");
  if (c->dtype != MOE_DTYPE_BF16 && c->dtype != MOE_DTYPE_FP8_BLOCK128 && c->dtype != MOE_DTYPE_NVFP4)
    return fail(MOE_ERR_INVALID, "unknown dtype");
  if (c->E > 1024) return fail(MOE_ERR_UNSUPPORTED, "E > 1024");
  if (c->h % 256 != 0) return fail(MOE_ERR_UNSUPPORTED, "h must be a multiple of 256");
  if (c->I % 128 != 0) return fail(MOE_ERR_UNSUPPORTED, "I must be a multiple of 128");
  if (c->dtype == MOE_DTYPE_NVFP4 && c->I % 256 != 0)
    return fail(MOE_ERR_UNSUPPORTED, "NVFP4 weights need I to be a multiple of 256");
  if (c->I_shared != 0 && c->I_shared != c->I) return fail(MOE_ERR_UNSUPPORTED, "I_shared must be 0 or I");
  if ((int64_t)c->T * (c->k + 1) > INT32_MAX) return fail(MOE_ERR_UNSUPPORTED, "T * (k + 1) exceeds int32 rows");
  if (!(c->capacity_factor >= 0.f)) return fail(MOE_ERR_INVALID, "capacity_factor must be >= 0");
  if (c->placement) {
    const moe_placement* p = c->placement;
    if (p->n_slots < c->E || p->n_slots > 1024 || p->max_replicas < 1)
      return fail(MOE_ERR_INVALID, "placement: need E <= n_slots <= 1024 and max_replicas >= 1");
    if (!p->slot_expert || !p->slot_replica || !p->replicas || !p->replica_slot)
      return fail(MOE_ERR_INVALID, "placement: NULL table");
  }
  return MOE_OK;
}

struct Layout {
  moe_ws_layout l;
  int64_t R, R_tot;
};

// expert-major buffers are grouped per physical slot (one per expert without a placement)
int64_t n_groups(const moe_config* c) { return c->placement ? c->placement->n_slots : c->E; }

// The tensor-core router (E >= 128, E a multiple of 32) works on 128 x 128 output tiles; a batch with
// fewer than 64 of them would leave most SMs idle for the whole K loop (T = 256, E = 256: 4 tiles, each
// 336 K steps), so each tile's K range is split over several CTAs (at least 2 K blocks of 64 each, up
// to about 128 CTAs in all) whose fp32 partial sums are added in a fixed order afterwards.
bool tensor_core_router(const moe_config* c) { return c->E >= 128 && c->E % 32 == 0; }
int router_csplit(const moe_config* c) {
  if (!tensor_core_router(c) || c->T <= 0) return 1;
  const int64_t tiles = moe::cdiv(c->T, 128) * moe::cdiv(c->E, 128);
  if (tiles >= 64) return 1;
  const int kpb = c->h / 64;
  const int want = (int)std::min<int64_t>(kpb / 2, moe::cdiv(128, tiles));
  if (want < 2) return 1;
  const int kper = (kpb + want - 1) / want;
  return (kpb + kper - 1) / kper;  // every split gets a non-empty K range
}
// bytes of the scratch region in front of the router's partial sums (status word, histograms)
size_t scratch_core_bytes(const moe_config* c) {
  return align256(256 + sizeof(int32_t) * (moe::dispatch_scratch_ints(c->T, c->E) + c->E));
}

Layout make_layout(const moe_config* c) {
  Layout L;
  const int64_t T = c->T, E = c->E, k = c->k, h = c->h, I = c->I, S = n_groups(c);
  const bool fp8 = c->dtype == MOE_DTYPE_FP8_BLOCK128;
  L.R = T * k;
  L.R_tot = L.R + (c->I_shared > 0 ? T : 0);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  moe_ws_layout& l = L.l;
  l.logits = take(sizeof(float) * T * E);
  l.topk_idx = take(sizeof(int32_t) * T * k);
  l.topk_w = take(sizeof(float) * T * k);
  l.counts = take(sizeof(int32_t) * S);
  l.offsets = take(sizeof(int32_t) * (S + 1));
  l.inv_pos = take(sizeof(int32_t) * T * k);
  l.row_token = take(sizeof(int32_t) * L.R);
  l.row_weight = take(sizeof(float) * L.R);
  l.xd = take((fp8 ? 1 : 2) * L.R_tot * h);
  l.xd_scales = take(fp8 ? sizeof(float) * L.R_tot * (h / 128) : 0);
  l.hbuf = take((fp8 ? 1 : 2) * L.R_tot * I);
  l.h_scales = take(fp8 ? sizeof(float) * L.R_tot * (I / 128) : 0);
  l.yd = take(2 * L.R_tot * h);
  l.router_w3 = take(2 * 3 * E * h);
  const int cs = router_csplit(c);
  l.scratch = take(scratch_core_bytes(c) + (cs > 1 ? sizeof(float) * cs * T * E : 0));
  l.total = o;
  return L;
}

int* status_ptr(void* ws, const moe_ws_layout& l) {
  return reinterpret_cast<int*>(static_cast<char*>(ws) + l.scratch);
}
// tile counters of the CTA-pair grouped GEMM launches, in the scratch header after the status word:
// [0] gate/up and [1] down of the routed launches, [2] and [3] those of the shared expert's launches
// on the second stream. moe_forward zeroes them with the status word; moe_expert_ffn zeroes the
// routed pair on its own stream.
constexpr int kTileCounters = 4;
// then the arrival counter of the fused small-batch kernel's grid barrier, also zeroed by moe_forward
constexpr int kHeaderInts = 16 + kTileCounters + 1;
static_assert(kHeaderInts * sizeof(int) <= 256, "the scratch header holds the status word and the counters");
int* tile_ctr_ptr(void* ws, const moe_ws_layout& l) { return status_ptr(ws, l) + 16; }
unsigned int* grid_barrier_ptr(void* ws, const moe_ws_layout& l) {
  return reinterpret_cast<unsigned int*>(status_ptr(ws, l) + 16 + kTileCounters);
}
int32_t* hist_ptr(void* ws, const moe_ws_layout& l) {
  return reinterpret_cast<int32_t*>(static_cast<char*>(ws) + l.scratch + 256);
}
// kept rows per logical expert (placement only), after the histograms
int32_t* expert_counts_ptr(void* ws, const moe_ws_layout& l, const moe_config* c) {
  return hist_ptr(ws, l) + moe::dispatch_scratch_ints(c->T, c->E);
}

void set_placement(moe::DispatchDesc& d, const moe_config* c, int32_t* expert_counts) {
  if (!c->placement) return;
  const moe_placement* p = c->placement;
  d.n_slots = p->n_slots;
  d.max_replicas = p->max_replicas;
  d.slot_expert = p->slot_expert;
  d.slot_replica = p->slot_replica;
  d.replicas = p->replicas;
  d.replica_slot = p->replica_slot;
  d.expert_counts = expert_counts;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int check_ws(void* ws, size_t ws_bytes, const Layout& L) {
  if (!ws) return fail(MOE_ERR_INVALID, "ws is NULL");
  if (!aligned16(ws)) return fail(MOE_ERR_INVALID, "ws must be 16-byte aligned");
  if (ws_bytes < L.l.total)
    return fail(MOE_ERR_WORKSPACE, "workspace too small: " + std::to_string(ws_bytes) + " < " +
                                       std::to_string(L.l.total) + " bytes");
  return MOE_OK;
}

#define REQUIRE_PTR(p, name)                                                   \
  do {                                                                         \
    if (!(p)) return fail(MOE_ERR_INVALID, std::string(name) + " is NULL");    \
    if (!aligned16(p)) return fail(MOE_ERR_INVALID, std::string(name) + " must be 16-byte aligned"); \
  } while (0)

// Step 1a, the router GEMM: logits = x W_r^T on the tensor cores (E >= 128, E % 32 == 0) or the
// CUDA cores (otherwise).
int do_router_gemm(const moe_config* c, const void* x, const moe_weights* w, float* logits, void* ws,
                   const Layout& L, cudaStream_t stream) {
  cudaError_t e;
  if (c->T > 0) {
    if (tensor_core_router(c)) {
      void* w3 = at<void>(ws, L.l.router_w3);
      e = moe::launch_split_router_weight(w->w_router, w3, (int64_t)c->E * c->h, stream);
      if (e != cudaSuccess) return cuda_fail(e, "router weight split launch");
      std::string err;
      moe::GroupedGemmDesc g;
      g.A = x;
      g.a_rows = c->T;
      g.B = w3;
      g.Bs = nullptr;
      g.b_rows = c->E;
      g.offsets = nullptr;
      g.E = 1;
      g.R = 0;
      g.T = c->T;
      g.K = c->h;
      g.N = c->E;
      g.I = 0;
      g.mode = 2;
      g.ksplit = 3;
      g.csplit = router_csplit(c);
      float* partials = at<float>(ws, L.l.scratch + scratch_core_bytes(c));
      g.out = g.csplit > 1 ? static_cast<void*>(partials) : static_cast<void*>(logits);
      g.ldo = c->E;
      g.row_weight = nullptr;
      g.status = status_ptr(ws, L.l);
      e = moe::launch_grouped_gemm_bf16(g, stream, &err);
      if (e != cudaSuccess) return err.empty() ? cuda_fail(e, "router GEMM launch") : cuda_fail(e, err.c_str());
      counted(2);
      // a split K range leaves partial sums; the top-k adds them (see do_route)
    } else {
      e = moe::launch_router_gemm(x, w->w_router, logits, c->T, c->h, c->E, stream);
      if (e != cudaSuccess) return cuda_fail(e, "router GEMM launch");
      counted(1);
    }
  }
  return MOE_OK;
}

moe::TopkDesc topk_desc(const moe_config* c, const moe_weights* w, const float* logits, int32_t* topk_idx,
                        float* topk_w) {
  moe::TopkDesc d;
  d.logits = const_cast<float*>(logits);
  d.bias = w ? w->bias : nullptr;
  d.topk_idx = topk_idx;
  d.topk_w = topk_w;
  d.T = c->T;
  d.E = c->E;
  d.k = c->k;
  d.n_group = c->n_group;
  d.topk_group = c->topk_group;
  d.score = c->score;
  d.renorm = c->renormalize;
  d.routed_scale = c->routed_scale;
  if (c->score == MOE_SCORE_SOFTMAX) d.bias = nullptr;
  return d;
}

int do_route(const moe_config* c, const void* x, const moe_weights* w, float* logits, int flags, int32_t* topk_idx,
             float* topk_w, void* ws, const Layout& L, cudaStream_t stream) {
  moe::TopkDesc d = topk_desc(c, w, logits, topk_idx, topk_w);
  if (!(flags & MOE_LOGITS_GIVEN)) {
    const int rc = do_router_gemm(c, x, w, logits, ws, L, stream);
    if (rc) return rc;
    // a tensor-core router whose K range was split over CTAs left partial sums in the scratch region:
    // the top-k kernel adds them in split order and writes the logits (one launch fewer)
    const int cs = router_csplit(c);
    if (tensor_core_router(c) && cs > 1) {
      d.partials = at<float>(ws, L.l.scratch + scratch_core_bytes(c));
      d.splits = cs;
    }
  }
  cudaError_t e = moe::launch_topk(d, stream);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  if (c->T > 0) counted(1);
  return MOE_OK;
}

// ceil(capacity_factor * T * k / E) assignments per expert, 0 = no limit
int capacity_of(const moe_config* c) {
  if (c->capacity_factor <= 0.f) return 0;
  const double cap = std::ceil((double)c->capacity_factor * (double)c->T * c->k / c->E);
  return cap >= (double)INT32_MAX ? 0 : (int)cap;
}

int do_dispatch(const moe_config* c, const void* x, const int32_t* topk_idx, const float* topk_w, int32_t* counts,
                int32_t* offsets, int32_t* inv_pos, int32_t* row_token, float* row_weight, void* xd, float* xd_scales,
                void* ws, const Layout& L, cudaStream_t stream, bool shared_rows = true) {
  moe::DispatchDesc d;
  d.x = x;
  d.topk_idx = topk_idx;
  d.topk_w = topk_w;
  d.counts = counts;
  d.offsets = offsets;
  d.inv_pos = inv_pos;
  d.row_token = row_token;
  d.row_weight = row_weight;
  d.xd = xd;
  d.xd_scales = xd_scales;
  d.scratch = hist_ptr(ws, L.l);
  d.status = status_ptr(ws, L.l);
  d.T = c->T;
  d.h = c->h;
  d.E = c->E;
  d.k = c->k;
  d.shared = c->I_shared > 0 && shared_rows;  // false: the shared expert reads x itself
  d.fp8 = c->dtype == MOE_DTYPE_FP8_BLOCK128;
  d.capacity = capacity_of(c);
  set_placement(d, c, expert_counts_ptr(ws, L.l, c));
  cudaError_t e = moe::launch_dispatch(d, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  if (c->T > 0) counted(4);
  return MOE_OK;
}

// Small batches in moe_forward: router, top-k, counts, offsets, rows and the dispatch copy as one
// cooperative kernel instead of six launches (Perplexity "CUDA Graph"; TensorRT-LLM "Runtime
// optimizations": a small step is launch-bound). Used where the router runs on the CUDA cores (E < 128,
// or E not a multiple of 32): with the tensor-core router in front, the fused kernel would replace
// only five short launches, and measured slower than them (a 256-token decode step: about 46 us
// against about 30 us, its phases separated by grid barriers and its top-k latency-bound on the few
// tokens). Dropless layers with one slot per expert only.
// The fused kernel runs on one CTA per SM (16 warps each), so it pays only while the work is small: a
// router of at most 2^25 multiply-adds (the tiny layer's 4096 x 512 x 8 is 2^24) and a dispatch copy of
// at most 2^22 elements per copy of x. Beyond that the standalone kernels, with many more warps to
// hide latency, are faster (a 4096-token layer with h 7168 and 32 experts: 369 us fused under ncu).
constexpr int64_t kFusedMaxRouterMacs = int64_t(1) << 25;
constexpr int64_t kFusedMaxRowElems = int64_t(1) << 22;
bool use_fused(const moe_config* c) {
  const int64_t th = (int64_t)c->T * c->h;
  return moe::fused_route_dispatch_supported(c->T, c->E) && capacity_of(c) == 0 && !c->placement &&
         !tensor_core_router(c) && th * c->E <= kFusedMaxRouterMacs && th <= kFusedMaxRowElems;
}

int do_fused_route_dispatch(const moe_config* c, const void* x, const moe_weights* w, void* ws, const Layout& L,
                            cudaStream_t stream, bool shared_rows) {
  const moe_ws_layout& l = L.l;
  float* logits = at<float>(ws, l.logits);
  moe::FusedRouteDispatchDesc d;
  d.x = x;
  d.w_router = w->w_router;
  d.tk = topk_desc(c, w, logits, at<int32_t>(ws, l.topk_idx), at<float>(ws, l.topk_w));
  d.counts = at<int32_t>(ws, l.counts);
  d.offsets = at<int32_t>(ws, l.offsets);
  d.inv_pos = at<int32_t>(ws, l.inv_pos);
  d.row_token = at<int32_t>(ws, l.row_token);
  d.row_weight = at<float>(ws, l.row_weight);
  d.xd = at<void>(ws, l.xd);
  d.xd_scales = at<float>(ws, l.xd_scales);
  d.h = c->h;
  d.shared = c->I_shared > 0 && shared_rows;
  d.fp8 = c->dtype == MOE_DTYPE_FP8_BLOCK128;
  d.barrier = grid_barrier_ptr(ws, l);
  d.status = status_ptr(ws, l);
  cudaError_t e = moe::launch_fused_route_dispatch(d, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fused route-and-dispatch launch");
  counted(1);
  return MOE_OK;
}

// bf16 expert GEMMs: CTA-pair tiles (256 rows, an expert's tail of at most 128 rows as a 128-row pair
// tile) move less shared memory per MMA than single-CTA tiles, but each CTA stages only half a weight
// tile per K step: a weight-streaming step (a few rows per expert) keeps more weight bytes in flight on
// single CTAs. (The FP8 kernel stays on single CTAs: its per-K-block promotion hand-off would have to
// cross the pair every 128 K elements.) A layer whose full pair tiles of the gate/up launch would not
// exceed one wave of pairs (the tiny layer: 64 tiles for 76 pairs) also stays on single CTAs: twice
// as many tiles for the same SMs, so no pair runs a second tile while the others idle.
constexpr int64_t kPairMinRowsPerGroup = 128;
bool use_pair_tiles(const moe_config* c, int S) {
  if (S <= 0 || (int64_t)c->T * c->k < kPairMinRowsPerGroup * S) return false;
  const int64_t pair_tiles = ((int64_t)c->T * c->k / 256) * (c->I / 128);
  return pair_tiles > moe::num_sms() / 2;
}

int do_expert_ffn(const moe_config* c, const moe_weights* w, const void* xd, const float* xd_scales,
                  const int32_t* offsets, const float* row_weight, void* yd, void* ws, const Layout& L,
                  cudaStream_t stream, bool with_shared = true, bool reset_ctr = true) {
  if (c->T == 0) return MOE_OK;
  const bool shared = c->I_shared > 0 && with_shared;
  std::string err;
  const int S = (int)n_groups(c);
  const int32_t* slot_expert = c->placement ? c->placement->slot_expert : nullptr;
  if (c->dtype == MOE_DTYPE_FP8_BLOCK128) {
    moe::GroupedGemmFp8Desc g;
    g.slot_expert = slot_expert;
    g.n_experts = c->E;
    g.A = xd;
    g.a_scales = xd_scales;
    g.a_rows = L.R_tot;
    g.B = w->w_gu;
    g.b_scales = w->s_gu;
    g.Bs = shared ? w->w_gu_shared : nullptr;
    g.bs_scales = shared ? w->s_gu_shared : nullptr;
    g.b_rows = 2 * (int64_t)c->I;
    g.offsets = offsets;
    g.E = S;
    g.R = (int)L.R;
    g.T = c->T;
    g.K = c->h;
    g.N = 2 * c->I;
    g.I = c->I;
    g.mode = 0;
    g.out = at<void>(ws, L.l.hbuf);
    g.out_scales = at<float>(ws, L.l.h_scales);
    g.ldo = c->I;
    g.row_weight = nullptr;
    g.status = status_ptr(ws, L.l);
    cudaError_t e = moe::launch_grouped_gemm_fp8(g, stream, &err);
    if (e != cudaSuccess) return err.empty() ? cuda_fail(e, "FP8 gate/up grouped GEMM launch") : cuda_fail(e, err.c_str());
    g.A = at<void>(ws, L.l.hbuf);
    g.a_scales = at<float>(ws, L.l.h_scales);
    g.B = w->w_d;
    g.b_scales = w->s_d;
    g.Bs = shared ? w->w_d_shared : nullptr;
    g.bs_scales = shared ? w->s_d_shared : nullptr;
    g.b_rows = c->h;
    g.K = c->I;
    g.N = c->h;
    g.mode = 1;
    g.out = yd;
    g.out_scales = nullptr;
    g.ldo = c->h;
    g.row_weight = row_weight;
    e = moe::launch_grouped_gemm_fp8(g, stream, &err);
    if (e != cudaSuccess) return err.empty() ? cuda_fail(e, "FP8 down grouped GEMM launch") : cuda_fail(e, err.c_str());
    counted(2);
    return MOE_OK;
  }
  if (c->dtype == MOE_DTYPE_NVFP4) {
    moe::GroupedGemmFp4Desc g;
    g.slot_expert = slot_expert;
    g.n_experts = c->E;
    g.A = xd;
    g.a_rows = L.R_tot;
    g.Bq = w->w_gu;
    g.Bs = w->s_gu;
    g.Bg = w->g_gu;
    g.Bq_shared = shared ? w->w_gu_shared : nullptr;
    g.Bs_shared = shared ? w->s_gu_shared : nullptr;
    g.Bg_shared = shared ? w->g_gu_shared : nullptr;
    g.b_rows = 2 * (int64_t)c->I;
    g.offsets = offsets;
    g.E = S;
    g.R = (int)L.R;
    g.T = c->T;
    g.K = c->h;
    g.N = 2 * c->I;
    g.I = c->I;
    g.mode = 0;
    g.out = at<void>(ws, L.l.hbuf);
    g.ldo = c->I;
    g.row_weight = nullptr;
    g.status = status_ptr(ws, L.l);
    cudaError_t e = moe::launch_grouped_gemm_nvfp4(g, stream, &err);
    if (e != cudaSuccess)
      return err.empty() ? cuda_fail(e, "NVFP4 gate/up grouped GEMM launch") : cuda_fail(e, err.c_str());
    g.A = at<void>(ws, L.l.hbuf);
    g.Bq = w->w_d;
    g.Bs = w->s_d;
    g.Bg = w->g_d;
    g.Bq_shared = shared ? w->w_d_shared : nullptr;
    g.Bs_shared = shared ? w->s_d_shared : nullptr;
    g.Bg_shared = shared ? w->g_d_shared : nullptr;
    g.b_rows = c->h;
    g.K = c->I;
    g.N = c->h;
    g.mode = 1;
    g.out = yd;
    g.ldo = c->h;
    g.row_weight = row_weight;
    e = moe::launch_grouped_gemm_nvfp4(g, stream, &err);
    if (e != cudaSuccess) return err.empty() ? cuda_fail(e, "NVFP4 down grouped GEMM launch") : cuda_fail(e, err.c_str());
    counted(2);
    return MOE_OK;
  }
  const bool pairs = use_pair_tiles(c, S);
  auto launch = pairs ? moe::launch_grouped_gemm_bf16_pair : moe::launch_grouped_gemm_bf16;
  int* ctr = tile_ctr_ptr(ws, L.l);
  if (pairs && reset_ctr) {
    cudaError_t e = cudaMemsetAsync(ctr, 0, 2 * sizeof(int), stream);
    if (e != cudaSuccess) return cuda_fail(e, "tile counter reset");
  }
  moe::GroupedGemmDesc g;
  g.slot_expert = slot_expert;
  g.n_experts = c->E;
  g.A = xd;
  g.a_rows = L.R_tot;
  g.B = w->w_gu;
  g.Bs = shared ? w->w_gu_shared : nullptr;
  g.b_rows = 2 * (int64_t)c->I;
  g.offsets = offsets;
  g.E = S;
  g.R = (int)L.R;
  g.T = c->T;
  g.K = c->h;
  g.N = 2 * c->I;
  g.I = c->I;
  g.mode = 0;
  g.out = at<void>(ws, L.l.hbuf);
  g.ldo = c->I;
  g.row_weight = nullptr;
  g.status = status_ptr(ws, L.l);
  g.tile_ctr = pairs ? ctr : nullptr;
  cudaError_t e = launch(g, stream, &err);
  if (e != cudaSuccess) return err.empty() ? cuda_fail(e, "gate/up grouped GEMM launch") : cuda_fail(e, err.c_str());
  g.A = at<void>(ws, L.l.hbuf);
  g.B = w->w_d;
  g.Bs = shared ? w->w_d_shared : nullptr;
  g.b_rows = c->h;
  g.K = c->I;
  g.N = c->h;
  g.mode = 1;
  g.out = yd;
  g.ldo = c->h;
  g.row_weight = row_weight;
  g.tile_ctr = pairs ? ctr + 1 : nullptr;
  e = launch(g, stream, &err);
  if (e != cudaSuccess) return err.empty() ? cuda_fail(e, "down grouped GEMM launch") : cuda_fail(e, err.c_str());
  counted(2);
  return MOE_OK;
}

// The shared expert alone (bf16): a dense SwiGLU MLP over all T tokens (inference guide 6.4 section 7:
// every token uses it, weight 1), as one group whose rows are read straight from x; it writes rows
// [R, R + T) of hbuf and yd, where the combine expects them. moe_forward runs it on a second stream
// while the routed rows are dispatched (TensorRT-LLM "DeepSeek R1 throughput on Blackwell",
// multi-stream: the shared expert does not depend on the routing).
int do_shared_ffn_bf16(const moe_config* c, const moe_weights* w, const void* x, void* ws, const Layout& L,
                       cudaStream_t stream) {
  if (c->T == 0) return MOE_OK;
  std::string err;
  // the kernel the shared group would get inside the routed launch, so that both paths compute its
  // rows with the same tiles (bit-identical outputs)
  const bool pairs = use_pair_tiles(c, (int)n_groups(c));
  auto launch = pairs ? moe::launch_grouped_gemm_bf16_pair : moe::launch_grouped_gemm_bf16;
  int* ctr = tile_ctr_ptr(ws, L.l) + 2;  // zeroed by moe_forward, the only caller
  __nv_bfloat16* hs = at<__nv_bfloat16>(ws, L.l.hbuf) + L.R * (int64_t)c->I;
  __nv_bfloat16* ys = at<__nv_bfloat16>(ws, L.l.yd) + L.R * (int64_t)c->h;
  moe::GroupedGemmDesc g;
  g.slot_expert = nullptr;
  g.n_experts = 1;
  g.A = x;
  g.a_rows = c->T;
  g.B = w->w_gu_shared;
  g.Bs = w->w_gu_shared;
  g.b_rows = 2 * (int64_t)c->I;
  g.offsets = nullptr;  // one group: rows [0, T)
  g.E = 0;
  g.R = 0;
  g.T = c->T;
  g.K = c->h;
  g.N = 2 * c->I;
  g.I = c->I;
  g.mode = 0;
  g.out = hs;
  g.ldo = c->I;
  g.row_weight = nullptr;
  g.status = status_ptr(ws, L.l);
  g.tile_ctr = pairs ? ctr : nullptr;
  cudaError_t e = launch(g, stream, &err);
  if (e != cudaSuccess)
    return err.empty() ? cuda_fail(e, "shared-expert gate/up launch") : cuda_fail(e, err.c_str());
  g.A = hs;
  g.B = w->w_d_shared;
  g.Bs = w->w_d_shared;
  g.b_rows = c->h;
  g.K = c->I;
  g.N = c->h;
  g.mode = 1;
  g.out = ys;
  g.ldo = c->h;
  g.tile_ctr = pairs ? ctr + 1 : nullptr;
  e = launch(g, stream, &err);
  if (e != cudaSuccess) return err.empty() ? cuda_fail(e, "shared-expert down launch") : cuda_fail(e, err.c_str());
  counted(2);
  return MOE_OK;
}

int check_expert_weights(const moe_config* c, const moe_weights* w) {
  if (!w) return fail(MOE_ERR_INVALID, "weights is NULL");
  REQUIRE_PTR(w->w_gu, "weights->w_gu");
  REQUIRE_PTR(w->w_d, "weights->w_d");
  if (c->I_shared > 0) {
    REQUIRE_PTR(w->w_gu_shared, "weights->w_gu_shared");
    REQUIRE_PTR(w->w_d_shared, "weights->w_d_shared");
  }
  if (c->dtype == MOE_DTYPE_FP8_BLOCK128 || c->dtype == MOE_DTYPE_NVFP4) {
    REQUIRE_PTR(w->s_gu, "weights->s_gu");
    REQUIRE_PTR(w->s_d, "weights->s_d");
    if (c->I_shared > 0) {
      REQUIRE_PTR(w->s_gu_shared, "weights->s_gu_shared");
      REQUIRE_PTR(w->s_d_shared, "weights->s_d_shared");
    }
  }
  if (c->dtype == MOE_DTYPE_NVFP4) {
    if (!w->g_gu || !w->g_d) return fail(MOE_ERR_INVALID, "weights->g_gu / g_d is NULL");
    if (c->I_shared > 0 && (!w->g_gu_shared || !w->g_d_shared))
      return fail(MOE_ERR_INVALID, "weights->g_gu_shared / g_d_shared is NULL");
  }
  return MOE_OK;
}

}  // namespace

MOE_EXPORT const char* moe_last_error(void) { return g_err.c_str(); }

MOE_EXPORT uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

MOE_EXPORT int moe_workspace_layout(const moe_config* cfg, moe_ws_layout* layout) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!layout) return fail(MOE_ERR_INVALID, "layout is NULL");
  *layout = make_layout(cfg).l;
  return MOE_OK;
}

MOE_EXPORT int moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!bytes) return fail(MOE_ERR_INVALID, "bytes is NULL");
  *bytes = make_layout(cfg).l.total;
  return MOE_OK;
}

MOE_EXPORT int moe_route(const moe_config* cfg, const void* x, const moe_weights* weights, float* logits, int flags,
                         int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (flags & ~MOE_LOGITS_GIVEN) return fail(MOE_ERR_INVALID, "unknown flags");
  Layout L = make_layout(cfg);
  if (flags & MOE_LOGITS_GIVEN) {
    REQUIRE_PTR(logits, "logits (given)");
  } else {
    REQUIRE_PTR(x, "x");
    if (!weights) return fail(MOE_ERR_INVALID, "weights is NULL");
    REQUIRE_PTR(weights->w_router, "weights->w_router");
    if ((rc = check_ws(ws, ws_bytes, L))) return rc;
    if (!logits)
      logits = at<float>(ws, L.l.logits);
    else if (!aligned16(logits))
      return fail(MOE_ERR_INVALID, "logits must be 16-byte aligned");
  }
  if (cfg->score == MOE_SCORE_SIGMOID && weights && weights->bias && !aligned16(weights->bias))
    return fail(MOE_ERR_INVALID, "weights->bias must be 16-byte aligned");
  REQUIRE_PTR(topk_idx, "topk_idx");
  REQUIRE_PTR(topk_w, "topk_w");
  return do_route(cfg, x, weights, logits, flags, topk_idx, topk_w, ws, L, (cudaStream_t)stream);
}

MOE_EXPORT int moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx, const float* topk_w,
                            int32_t* counts, int32_t* offsets, int32_t* inv_pos, int32_t* row_token,
                            float* row_weight, void* xd, float* xd_scales, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  Layout L = make_layout(cfg);
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  REQUIRE_PTR(x, "x");
  REQUIRE_PTR(topk_idx, "topk_idx");
  REQUIRE_PTR(topk_w, "topk_w");
  REQUIRE_PTR(counts, "counts");
  REQUIRE_PTR(offsets, "offsets");
  REQUIRE_PTR(inv_pos, "inv_pos");
  REQUIRE_PTR(row_token, "row_token");
  REQUIRE_PTR(row_weight, "row_weight");
  REQUIRE_PTR(xd, "xd");
  if (cfg->dtype == MOE_DTYPE_FP8_BLOCK128) REQUIRE_PTR(xd_scales, "xd_scales");
  return do_dispatch(cfg, x, topk_idx, topk_w, counts, offsets, inv_pos, row_token, row_weight, xd, xd_scales, ws, L,
                     (cudaStream_t)stream);
}

MOE_EXPORT int moe_expert_ffn(const moe_config* cfg, const moe_weights* weights, const void* xd,
                              const float* xd_scales, const int32_t* offsets, const float* row_weight, void* yd,
                              void* ws, size_t ws_bytes, moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  Layout L = make_layout(cfg);
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  if ((rc = check_expert_weights(cfg, weights))) return rc;
  REQUIRE_PTR(xd, "xd");
  REQUIRE_PTR(offsets, "offsets");
  REQUIRE_PTR(row_weight, "row_weight");
  REQUIRE_PTR(yd, "yd");
  if (cfg->dtype == MOE_DTYPE_FP8_BLOCK128) REQUIRE_PTR(xd_scales, "xd_scales");
  return do_expert_ffn(cfg, weights, xd, xd_scales, offsets, row_weight, yd, ws, L, (cudaStream_t)stream);
}

MOE_EXPORT int moe_combine(const moe_config* cfg, const void* yd, const int32_t* inv_pos, void* y,
                           moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  REQUIRE_PTR(yd, "yd");
  REQUIRE_PTR(inv_pos, "inv_pos");
  REQUIRE_PTR(y, "y");
  cudaError_t e = moe::launch_combine(yd, inv_pos, y, cfg->T, cfg->h, cfg->k, cfg->I_shared > 0, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  if (cfg->T > 0) counted(1);
  return MOE_OK;
}

namespace {

// A second stream per device for the shared expert, with the fork and join events. Created on first
// use on a device (and again under a new context there, e.g. after cudaDeviceReset) and kept for the
// life of the process; the enqueue of a fork ... join section holds g_side_mu, so calls from several
// host threads cannot interleave their event records.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
moe::PerDevice<SideStream> g_side;

cudaError_t side_stream(SideStream* out) {
  return moe::per_device<SideStream>(
      g_side,
      [](SideStream& sd) {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        return cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming);
      },
      out);
}

}  // namespace

MOE_EXPORT int moe_forward(const moe_config* cfg, const void* x, const moe_weights* weights, void* y, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  Layout L = make_layout(cfg);
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  REQUIRE_PTR(x, "x");
  REQUIRE_PTR(y, "y");
  if (!weights) return fail(MOE_ERR_INVALID, "weights is NULL");
  REQUIRE_PTR(weights->w_router, "weights->w_router");
  if ((rc = check_expert_weights(cfg, weights))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  // the status word, the grouped GEMMs' tile counters and the fused kernel's barrier counter
  cudaError_t e = cudaMemsetAsync(status_ptr(ws, L.l), 0, kHeaderInts * sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  const moe_ws_layout& l = L.l;
  // bf16 layers with a shared expert: the shared expert runs on a second stream (it needs only x),
  // overlapping dispatch and the routed GEMMs; the combine waits for it
  const bool side = cfg->I_shared > 0 && cfg->T > 0 && cfg->dtype == MOE_DTYPE_BF16;
  // small batches: routing and dispatch as one cooperative kernel, before the second stream forks (the
  // fork then overlaps the routed GEMMs, and the cooperative grid never shares the SMs with it)
  const bool fused = use_fused(cfg);
  if (fused) {
    if ((rc = do_fused_route_dispatch(cfg, x, weights, ws, L, s, !side))) return rc;
  } else if ((rc = do_route(cfg, x, weights, at<float>(ws, l.logits), 0, at<int32_t>(ws, l.topk_idx),
                            at<float>(ws, l.topk_w), ws, L, s))) {
    return rc;
  }
  std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
  SideStream side_handles;
  SideStream* sd = &side_handles;
  if (side) {
    side_lock.lock();
    if ((e = side_stream(sd)) != cudaSuccess) return cuda_fail(e, "second stream set-up");
    if ((e = cudaEventRecord(sd->fork, s)) != cudaSuccess) return cuda_fail(e, "fork event record");
    if ((e = cudaStreamWaitEvent(sd->stream, sd->fork, 0)) != cudaSuccess) return cuda_fail(e, "fork wait");
    const int src = do_shared_ffn_bf16(cfg, weights, x, ws, L, sd->stream);
    // the join is recorded even after a failed launch, so that a capture on `s` can still end
    if ((e = cudaEventRecord(sd->join, sd->stream)) != cudaSuccess) return cuda_fail(e, "join event record");
    if (src) {
      cudaStreamWaitEvent(s, sd->join, 0);
      return src;
    }
  }
  if (!fused && (rc = do_dispatch(cfg, x, at<int32_t>(ws, l.topk_idx), at<float>(ws, l.topk_w),
                                  at<int32_t>(ws, l.counts), at<int32_t>(ws, l.offsets), at<int32_t>(ws, l.inv_pos),
                                  at<int32_t>(ws, l.row_token), at<float>(ws, l.row_weight), at<void>(ws, l.xd),
                                  at<float>(ws, l.xd_scales), ws, L, s, !side))) {
    if (side) cudaStreamWaitEvent(s, sd->join, 0);
    return rc;
  }
  if ((rc = do_expert_ffn(cfg, weights, at<void>(ws, l.xd), at<float>(ws, l.xd_scales), at<int32_t>(ws, l.offsets),
                          at<float>(ws, l.row_weight), at<void>(ws, l.yd), ws, L, s, !side, false))) {
    if (side) cudaStreamWaitEvent(s, sd->join, 0);
    return rc;
  }
  if (side) {
    // the join wait is enqueued before the lock is released: it binds the record of this call
    if ((e = cudaStreamWaitEvent(s, sd->join, 0)) != cudaSuccess) return cuda_fail(e, "join wait");
    side_lock.unlock();
  }
  e = moe::launch_combine(at<void>(ws, l.yd), at<int32_t>(ws, l.inv_pos), y, cfg->T, cfg->h, cfg->k,
                          cfg->I_shared > 0, s);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  if (cfg->T > 0) counted(1);
  return MOE_OK;
}

// ------------------------------------------------------------------------------------------
// CUDA graph of the whole layer
// ------------------------------------------------------------------------------------------
struct moe_graph_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int kernels = 0;  // library kernels per launch
};

MOE_EXPORT int moe_graph_create(const moe_config* cfg, const void* x, const moe_weights* weights, void* y, void* ws,
                                size_t ws_bytes, moe_stream_t stream, moe_graph* graph) {
  if (!graph) return fail(MOE_ERR_INVALID, "graph is NULL");
  *graph = nullptr;
  if (!stream) return fail(MOE_ERR_INVALID, "capture needs a created stream, not the legacy default stream");
  cudaStream_t s = (cudaStream_t)stream;
  // eager run: validates the arguments and performs the lazy one-time set-up outside the capture
  int rc = moe_forward(cfg, x, weights, y, ws, ws_bytes, stream);
  if (rc) return rc;
  const uint64_t before = g_launches.load();
  cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
  rc = moe_forward(cfg, x, weights, y, ws, ws_bytes, stream);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(s, &g);
  if (rc) {
    if (g) cudaGraphDestroy(g);
    return rc;
  }
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
  cudaGraphExec_t ex = nullptr;
  e = cudaGraphInstantiate(&ex, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return cuda_fail(e, "cudaGraphInstantiate");
  }
  moe_graph_s* out = new moe_graph_s;
  out->graph = g;
  out->exec = ex;
  out->kernels = (int)(g_launches.load() - before);
  g_launches.fetch_sub((uint64_t)out->kernels);  // captured, not launched
  *graph = out;
  return MOE_OK;
}

MOE_EXPORT int moe_graph_launch(moe_graph graph, moe_stream_t stream) {
  if (!graph) return fail(MOE_ERR_INVALID, "graph is NULL");
  cudaError_t e = cudaGraphLaunch(graph->exec, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  counted(graph->kernels);
  return MOE_OK;
}

MOE_EXPORT int moe_graph_destroy(moe_graph graph) {
  if (!graph) return MOE_OK;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
  return MOE_OK;
}

MOE_EXPORT int moe_quantize_weights_fp8(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, float* s,
                                        moe_stream_t stream) {
  if (batch < 0 || rows < 0 || cols < 0) return fail(MOE_ERR_INVALID, "negative size");
  if (rows % 128 || cols % 128) return fail(MOE_ERR_UNSUPPORTED, "rows and cols must be multiples of 128");
  REQUIRE_PTR(w, "w");
  REQUIRE_PTR(q, "q");
  if (!s) return fail(MOE_ERR_INVALID, "s is NULL");
  cudaError_t e = moe::launch_quantize_weights(w, batch, rows, cols, q, s, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "weight quantisation launch");
  if (batch * (rows / 128) * (cols / 128) > 0) counted(1);
  return MOE_OK;
}

MOE_EXPORT int moe_quantize_weights_nvfp4(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, void* s,
                                          float* g, moe_stream_t stream) {
  if (batch < 0 || rows < 0 || cols < 0) return fail(MOE_ERR_INVALID, "negative size");
  if (cols % 256) return fail(MOE_ERR_UNSUPPORTED, "cols must be a multiple of 256");
  if (batch > 65535) return fail(MOE_ERR_UNSUPPORTED, "batch > 65535");
  REQUIRE_PTR(w, "w");
  REQUIRE_PTR(q, "q");
  if (!s || !g) return fail(MOE_ERR_INVALID, "s or g is NULL");
  cudaError_t e = moe::launch_quantize_weights_nvfp4(w, batch, rows, cols, q, s, g, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 weight quantisation launch");
  if (batch * rows * cols > 0) counted(3);
  return MOE_OK;
}

MOE_EXPORT int moe_eplb_plan(const int64_t* load, int32_t E, int32_t n_cards, int32_t n_redundant, int32_t* replicas,
                             int32_t* slot_expert, int32_t* slot_replica, int32_t* replica_slot, double* card_load) {
  std::string err;
  const int rc = moe::eplb_plan(load, E, n_cards, n_redundant, replicas, slot_expert, slot_replica, replica_slot,
                                card_load, &err);
  if (rc) return fail(rc, err);
  return MOE_OK;
}

MOE_EXPORT int moe_selftest_wait_timeout(const moe_config* cfg, void* ws, size_t ws_bytes, int64_t limit_cycles,
                                         moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  Layout L = make_layout(cfg);
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  if (limit_cycles < 1 || limit_cycles > 4000000000LL) return fail(MOE_ERR_INVALID, "limit_cycles must lie in [1, 4e9]");
  cudaError_t e = moe::launch_wait_timeout_selftest(status_ptr(ws, L.l), (long long)limit_cycles, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  counted(1);
  return MOE_OK;
}

MOE_EXPORT int moe_balance(const moe_config* cfg, const void* ws, moe_balance_stats* stats, moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  REQUIRE_PTR(ws, "ws");
  REQUIRE_PTR(stats, "stats");
  Layout L = make_layout(cfg);
  void* w = const_cast<void*>(ws);
  cudaError_t e = moe::launch_balance(at<int32_t>(w, L.l.counts), at<int32_t>(w, L.l.offsets), (int)n_groups(cfg),
                                      (int64_t)cfg->T * cfg->k, stats, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "balance launch");
  counted(1);
  return MOE_OK;
}

MOE_EXPORT int moe_device_status(const moe_config* cfg, void* ws, int32_t* status, moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!ws || !status) return fail(MOE_ERR_INVALID, "ws and status must not be NULL");
  Layout L = make_layout(cfg);
  int* p = status_ptr(ws, L.l);
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read-back");
  *status = v;
  if (v) return fail(MOE_ERR_DEVICE, "device status bits set: " + std::to_string(v));
  return MOE_OK;
}

// ------------------------------------------------------------------------------------------
// Dispatch without a workspace.
//
// For callers that cannot give the library any device memory of their own: an engine that has
// handed all of device memory to its own pool and permits no other allocation, or a plug-in hook
// whose interface passes only the layer's inputs and outputs (cudaMalloc can also synchronise the
// whole device, which such callers must not do). The dispatch step then takes its scratch (the
// per-block expert histograms and the status word) from an array that lives in the library's own
// global memory. Every GPU that loads the library holds this array until the process exits.
// ------------------------------------------------------------------------------------------
constexpr size_t kNoAllocHistInts = 131072;  // 512 KiB of histograms: ceil(T / 512) * E entries at most
constexpr size_t kNoAllocStatusInts = 64;    // status word, padded to keep the histograms 256-byte aligned

static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocStatusInts + kNoAllocHistInts];

namespace {

moe::PerDevice<int32_t*> g_noalloc_addr;

// Device address of the scratch array on the current device. The name is only a host-side stand-in;
// the address is looked up with the device current, on the first call there, and again when the
// context current on the device has changed since (cudaDeviceReset, or another context made current),
// since the array's address belongs to the module loaded into one context.
int noalloc_scratch(int32_t** out) {
  const cudaError_t e = moe::per_device<int32_t*>(
      g_noalloc_addr,
      [](int32_t*& addr) {
        void* p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        addr = static_cast<int32_t*>(p);
        return r;
      },
      out);
  if (e == cudaErrorInvalidDevice) return fail(MOE_ERR_UNSUPPORTED, "device ordinal beyond 63");
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static dispatch scratch");
  return MOE_OK;
}

}  // namespace

MOE_EXPORT int moe_dispatch_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                    const float* topk_w, int32_t* counts, int32_t* offsets, int32_t* inv_pos,
                                    int32_t* row_token, float* row_weight, void* xd, float* xd_scales,
                                    moe_stream_t stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  const size_t need = moe::dispatch_scratch_ints(cfg->T, cfg->E) + cfg->E;
  if (need > kNoAllocHistInts)
    return fail(MOE_ERR_UNSUPPORTED, "moe_dispatch_noalloc: (ceil(T / 512) + 1) * E = " + std::to_string(need) +
                                         " histogram entries exceed the static scratch of " +
                                         std::to_string(kNoAllocHistInts) + "; use moe_dispatch with a workspace");
  REQUIRE_PTR(x, "x");
  REQUIRE_PTR(topk_idx, "topk_idx");
  REQUIRE_PTR(topk_w, "topk_w");
  REQUIRE_PTR(counts, "counts");
  REQUIRE_PTR(offsets, "offsets");
  REQUIRE_PTR(inv_pos, "inv_pos");
  REQUIRE_PTR(row_token, "row_token");
  REQUIRE_PTR(row_weight, "row_weight");
  REQUIRE_PTR(xd, "xd");
  if (cfg->dtype == MOE_DTYPE_FP8_BLOCK128) REQUIRE_PTR(xd_scales, "xd_scales");
  int32_t* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  // the status word accumulates bits with atomicOr: it must start at zero; the histograms are written
  // in full before they are read, so they need no clearing
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the static dispatch status word");
  moe::DispatchDesc d;
  d.x = x;
  d.topk_idx = topk_idx;
  d.topk_w = topk_w;
  d.counts = counts;
  d.offsets = offsets;
  d.inv_pos = inv_pos;
  d.row_token = row_token;
  d.row_weight = row_weight;
  d.xd = xd;
  d.xd_scales = xd_scales;
  d.scratch = scratch + kNoAllocStatusInts;
  d.status = scratch;
  d.T = cfg->T;
  d.h = cfg->h;
  d.E = cfg->E;
  d.k = cfg->k;
  d.shared = cfg->I_shared > 0;
  d.fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
  d.capacity = capacity_of(cfg);
  set_placement(d, cfg, d.scratch + moe::dispatch_scratch_ints(cfg->T, cfg->E));
  e = moe::launch_dispatch(d, s);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  if (cfg->T > 0) counted(4);
  return MOE_OK;
}
