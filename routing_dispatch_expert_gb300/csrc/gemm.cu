// Grouped GEMM of the expert FFN on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Perplexity blog "Lower latency and higher throughput with multi-node DeepSeek deployment",
// "Roofline model / GroupGEMM": g groups, group i multiplies [m_i, k] x [k, n]. Here the groups are
// the E routed experts (rows [offsets[e], offsets[e+1]) of the expert-major buffer) plus the shared
// expert (the last T rows), and the two projections of the SwiGLU FFN (inference guide 6.4,
// section 2.1: gate, up, down) are two launches:
//   mode 0  H  = silu(A W_gate^T) * (A W_up^T)     A = xd [R_tot, h], W_gu [E, 2I, h]
//   mode 1  yd = (A W_down^T) * row_weight         A = H  [R_tot, I], W_d  [E, h, I]
// and the router GEMM of the same layer as a single group (TensorRT-LLM "DeepSeek R1 throughput on
// Blackwell", "RouterGEMM mixed I/O": bf16 activations in, fp32 logits out):
//   mode 2  logits = x (W_hi + W_mid + W_lo)^T     A = x [T, h], B = the fp32 router weight split into
//           three bf16 terms [3, E, h]; x is exact in bf16 and every bf16 x bf16 product is exact in
//           fp32. The tensor core's accumulator does not round like an IEEE fp32 add over thousands
//           of steps, so the MMAs accumulate chunks of ROUTER_CHUNK K blocks in TMEM (double
//           buffered) and the epilogue sums the chunks in fp32 registers. The router runs a
//           320-thread instantiation: 256-column tiles drained by eight epilogue warps (two per
//           TMEM lane quarter), or 128-column tiles by four when the K range is split. A batch
//           too small to fill the SMs splits each tile's K range over `csplit` CTAs, which write fp32
//           partial sums that the top-k kernel adds in split order.
// Work follows the device-side per-expert counts (Perplexity, "Quantization": kernels read the
// routing information to split the work, instead of sizing it from buffer bounds), so the launch
// needs no host read-back and has a fixed grid.
//
// Design (GB300 / sm_103a):
//   * persistent: one CTA per SM walks tiles blockIdx.x, +gridDim.x, ...; tile order is group-major,
//     then output-column tile, then 128-row tile, so CTAs running together share the weight tile
//     through L2 and an expert's activation rows stay L2-resident across its column tiles;
//   * tile 128 x 256 x 64 (bf16), one tcgen05.mma.cta_group::1 M=128 N=256 K=16 per 32-byte K step;
//   * warp 0 lane 0 issues TMA loads (128-byte swizzle) into a 4-stage shared-memory ring, warp 1
//     lane 0 issues the MMAs, warps 2-5 drain the accumulator (TMEM, 2 x 256 columns, double
//     buffered so the epilogue of one tile overlaps the MMAs of the next);
//   * for mode 0 the B tile holds 128 gate rows and the 128 matching up rows, so the SwiGLU product
//     is formed in the epilogue and only H is written;
//   * every mbarrier wait is bounded; on a time-out the kernel records MOE_STATUS_WAIT_TIMEOUT,
//     drains its own copies and MMAs (again bounded), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {

namespace gg {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // bf16 elements per 128-byte swizzled row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;          // warps 0 TMA, 1 MMA, 2-5 epilogue
constexpr int ROUTER_THREADS = 320;   // the router's instantiation: warps 2-9 drain 256-column tiles
constexpr int TMEM_COLS = 2 * BN;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
constexpr int ROUTER_CHUNK = 8;  // K blocks (512 K elements) per TMEM partial sum in mode 2

struct Args {
  const int32_t* offsets;  // [E + 1]
  int E;
  int shared;  // 1: group E is the shared expert (rows [R, R + T))
  int R;
  int T;
  int K;        // reduction length (multiple of BK)
  int n_tiles;  // output column tiles per group
  const int32_t* slot_expert;  // routed group -> logical expert whose weights it uses (nullptr: identity)
  int mode;     // 0: gate/up + SwiGLU -> H; 1: down * row_weight -> yd; 2: router, fp32 out
  int I;        // mode 0: row offset of the up half inside W_gu
  int ksplit;   // B is split into ksplit K passes over the same A (mode 2: 3), else 1
  int csplit;   // mode 2: CTAs sharing one output tile, each over a contiguous range of K (1: none);
                // split s writes its fp32 partial sums to out + s * T * ldo
  int n_valid;  // mode 2: output columns that exist (E)
  int rbn;      // mode 2: output tile width, 128 or 256 (256 needs the ROUTER_THREADS instantiation)
  int ldo;      // output row stride in elements
  int vec32;    // modes 0 and 1: the output rows and column tiles start on 32-byte boundaries
  void* out;
  const float* row_weight;
  int* status;
  long long wait_limit;
};

struct Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_slot;
  volatile int abort_flag;
  grp::Table tb;
};

using grp::silu;
using grp::Tile;
using grp::wait_or_abort;

template <int NT>
__global__ void __launch_bounds__(NT, 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmBs, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared s;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.E + args.shared;

  // ---- set-up: tile table over groups, barriers, TMEM
  if (warp == 0) {
    grp::build_table(s.tb, args.offsets, args.E, args.shared, args.R, args.T, BM, lane);
    if (lane == 0) {
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(&s.full[i], 1);
        mbar_init(&s.empty[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.tfull[i], 1);
        mbar_init(&s.tempty[i], args.mode == 2 && args.rbn == BN ? 8 : 4);
      }
      mbar_init(&s.mma_done, 1);
      s.abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmBs);
    }
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_slot;
  const int csplit = args.mode == 2 ? args.csplit : 1;
  const int total = s.tb.gtile[G] * args.n_tiles * csplit;
  const int kpb = args.K / BK;  // K blocks per pass over A
  const int kper = (kpb + csplit - 1) / csplit;  // K blocks of A per split
  // the K blocks (in units of the ksplit-interleaved loop) of work unit `tile`; an output tile is
  // tile / csplit, its split tile % csplit
  auto krange = [&](int tile, int& k0, int& k1) {
    const int sp = tile % csplit;
    k0 = min(kpb, sp * kper) * args.ksplit;
    k1 = min(kpb, (sp + 1) * kper) * args.ksplit;
  };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      Tile t = grp::decode(s.tb, G, args.n_tiles, tile / csplit, BM, args.mode == 2);
      int kb0, kb1;
      krange(tile, kb0, kb1);
      const CUtensorMap* mb = t.g < args.E ? &tmB : &tmBs;
      const int zg = t.g < args.E ? (args.slot_expert ? args.slot_expert[t.g] : t.g) : 0;
      int n0, n1;
      if (args.mode == 0) {
        n0 = t.n_tile * (BN / 2);
        n1 = args.I + t.n_tile * (BN / 2);
      } else if (args.mode == 2) {
        n0 = t.n_tile * args.rbn;  // 128-wide tiles: one B box; 256-wide: two (rows past E read as zero)
        n1 = args.rbn == BN ? n0 + BN / 2 : -1;
      } else {
        n0 = t.n_tile * BN;
        n1 = n0 + BN / 2;
      }
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_or_abort(&s.empty[stage], phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        uint8_t* a = smem + stage * STAGE_BYTES;
        uint8_t* b = a + A_BYTES;
        // router: the three weight terms of one K block are consecutive stages, so the A tile is
        // re-read from L2 right away instead of once per full pass over K
        const int pass = args.ksplit > 1 ? kb % args.ksplit : 0;
        const int ka = (args.ksplit > 1 ? kb / args.ksplit : kb) * BK;
        const int z = args.ksplit > 1 ? pass : zg;
        mbar_arrive_expect_tx(&s.full[stage], n1 >= 0 ? STAGE_BYTES : A_BYTES + B_BYTES / 2);
        tma_load_2d(a, &tmA, &s.full[stage], ka, t.a_row);
        tma_load_3d(b, mb, &s.full[stage], ka, n0, z);
        if (n1 >= 0) tma_load_3d(b + B_BYTES / 2, mb, &s.full[stage], ka, n1, z);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // drain: the last fills of every stage must have landed before the CTA may exit
    long long first = issued > STAGES ? issued - STAGES : 0;
    for (long long i = first; i < issued; ++i) {
      int st = (int)(i % STAGES);
      uint32_t ph = (uint32_t)((i / STAGES) & 1);
      long long t0 = clock64();
      while (!mbar_try_wait(&s.full[st], ph) && clock64() - t0 < args.wait_limit) {
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    // The accumulator holds one chunk of K blocks: the whole tile (modes 0, 1) or ROUTER_CHUNK
    // blocks (mode 2, whose epilogue adds the chunks in fp32).
    const uint32_t idesc = args.mode == 2 ? idesc_bf16(BM, args.rbn) : idesc_bf16(BM, BN);
    const int ch_len = args.mode == 2 ? ROUTER_CHUNK : kpb * args.ksplit;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      uint32_t d = 0;
      int kb0, kb1;
      krange(tile, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        const int kc = (kb - kb0) % ch_len;
        if (kc == 0) {
          if (!wait_or_abort(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          d = tmem_base + (uint32_t)(acc * BN);
        }
        if (!wait_or_abort(&s.full[stage], phase, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t b = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_f16(d, sw128_kmajor_desc(a + kk * 32), sw128_kmajor_desc(b + kk * 32), idesc, (kc | kk) != 0);
        umma_commit(&s.empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (kc == ch_len - 1 || kb == kb1 - 1) {
          umma_commit(&s.tfull[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
      }
    }
    // all MMAs issued by this thread complete before TMEM / shared memory go away
    umma_commit(&s.mma_done);
    long long t0 = clock64();
    while (!mbar_try_wait(&s.mma_done, 0) && clock64() - t0 < args.wait_limit) {
    }
  } else if (warp >= 2 && (warp < 6 || (args.mode == 2 && args.rbn == BN))) {
    // ---------------- epilogue: TMEM -> registers -> global
    const int quarter = warp & 3;  // TMEM lanes [32 * quarter, 32 * quarter + 32)
    const int chalf = (warp - 2) >> 2;  // mode 2 with 256-wide tiles: which 128 of the tile's columns
    const int r = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      Tile t = grp::decode(s.tb, G, args.n_tiles, tile / csplit, BM, args.mode == 2);
      if (args.mode == 2) {
        // router: sum the TMEM chunk partials of this tile in fp32 registers, then store
        float run[BN / 2];
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) run[i] = 0.f;
        int kb0, kb1;
        krange(tile, kb0, kb1);
        const int nch = (kb1 - kb0 + ROUTER_CHUNK - 1) / ROUTER_CHUNK;
        bool fine = true;
        for (int ch = 0; ch < nch; ++ch) {
          int ok = 1;
          if (lane == 0) ok = wait_or_abort(&s.tfull[acc], acc_phase, &s.abort_flag, args.status, args.wait_limit);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            fine = false;
            break;
          }
          __syncwarp();
          tc_fence_after();
          const uint32_t taddr =
              tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + chalf * (BN / 2));
#pragma unroll
          for (int c = 0; c < BN / 2; c += 32) {
            uint32_t v[32];
            tmem_ld32(taddr + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) run[c + i] = __fadd_rn(run[c + i], __uint_as_float(v[i]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.tempty[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (!fine) break;
        const int col0 = t.n_tile * args.rbn + chalf * (BN / 2);
        const int ncols = min(BN / 2, args.n_valid - col0);  // a multiple of 32 (may be <= 0)
        if (r < t.rows) {
          float* out = reinterpret_cast<float*>(args.out) + (int64_t)(tile % csplit) * args.T * args.ldo +
                       ((int64_t)t.a_row + r) * args.ldo + col0;
#pragma unroll
          for (int c = 0; c < BN / 2; c += 32)
            if (c < ncols) {
              float4* dst = reinterpret_cast<float4*>(out + c);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(run[c + 4 * i], run[c + 4 * i + 1], run[c + 4 * i + 2], run[c + 4 * i + 3]);
            }
        }
        continue;
      }
      // one lane waits, the warp follows: the tcgen05.ld below is warp-collective
      int ok = 1;
      if (lane == 0) ok = wait_or_abort(&s.tfull[acc], acc_phase, &s.abort_flag, args.status, args.wait_limit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      const bool valid = r < t.rows;
      const int64_t orow = (int64_t)t.a_row + r;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (args.mode == 0) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out) + orow * args.ldo + t.n_tile * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c, g);
          tmem_ld32(taddr + BN / 2 + c, u);
          tmem_ld_wait();
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
            float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
            p[i] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            if (args.vec32) {  // one full L2 sector per store
              st_global_v8(out + c, p);
              st_global_v8(out + c + 16, p + 8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
            }
          }
        }
      } else {
        const float w = (valid && t.g < args.E) ? args.row_weight[orow] : 1.0f;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out) + orow * args.ldo + t.n_tile * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * w, __uint_as_float(v[2 * i + 1]) * w);
          if (valid) {
            if (args.vec32) {  // one full L2 sector per store
              st_global_v8(out + c, p);
              st_global_v8(out + c + 16, p + 8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace gg

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

cudaError_t tma_encoder_ready() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

bool tma_encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int64_t rows, int64_t K,
                   int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K * elem)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_encode_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int64_t G, int64_t rows,
                   int64_t K, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)(K * elem), (cuuint64_t)(rows * K * elem)};
  cuuint32_t box[3] = {(cuuint32_t)(128 / elem), (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_encode_3d_plain(CUtensorMap* m, const void* base, int64_t G, int64_t rows, int64_t K, int box_k, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)G};
  cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)(rows * K)};
  cuuint32_t box[3] = {(cuuint32_t)box_k, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
using PFN_ctx_get_current = CUresult (*)(CUcontext*);
PFN_ctx_get_current g_ctx_get_current = nullptr;
std::once_flag g_ctx_once;
}  // namespace

cudaError_t current_device(int* dev, const void** ctx) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PFN_ctx_get_current>(fn);
  });
  CUcontext c = nullptr;
  if (!g_ctx_get_current || g_ctx_get_current(&c) != CUDA_SUCCESS) c = nullptr;
  *ctx = c;
  return cudaSuccess;
}

int num_sms() {
  static PerDevice<int> table;
  int n = 0;
  const cudaError_t e = per_device<int>(
      table,
      [](int& v) {
        int dev = 0;
        cudaError_t r = cudaGetDevice(&dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess && v <= 0) r = cudaErrorInvalidValue;
        return r;
      },
      &n);
  return e == cudaSuccess ? n : kNumSMsHint;
}

cudaError_t launch_grouped_gemm_bf16(const GroupedGemmDesc& d, cudaStream_t stream, std::string* err) {
  cudaError_t e = tma_encoder_ready();
  if (e != cudaSuccess) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return e;
  }
  // the dynamic shared-memory opt-in is a per-device function attribute
  static PerDevice<bool> attr;
  bool attr_set = false;
  e = per_device<bool>(
      attr,
      [](bool& v) {
        cudaError_t r = cudaFuncSetAttribute(gg::grouped_gemm_bf16_kernel<gg::THREADS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, gg::SMEM_BYTES);
        if (r == cudaSuccess)
          r = cudaFuncSetAttribute(gg::grouped_gemm_bf16_kernel<gg::ROUTER_THREADS>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, gg::SMEM_BYTES);
        v = r == cudaSuccess;
        return r;
      },
      &attr_set);
  if (e != cudaSuccess) {
    *err = "cudaFuncSetAttribute failed";
    return e;
  }
  CUtensorMap tA, tB, tBs;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int ksplit = d.ksplit > 1 ? d.ksplit : 1;
  bool ok = tma_encode_2d(&tA, d.A, BF, 2, d.a_rows, d.K, gg::BM) &&
            tma_encode_3d(&tB, d.B, BF, 2, ksplit > 1 ? ksplit : (d.n_experts > 0 ? d.n_experts : d.E), d.b_rows,
                          d.K, gg::BN / 2) &&
            tma_encode_3d(&tBs, d.Bs ? d.Bs : d.B, BF, 2, 1, d.b_rows, d.K, gg::BN / 2);
  if (!ok) {
    *err = "cuTensorMapEncodeTiled rejected a grouped-GEMM operand";
    return cudaErrorInvalidValue;
  }
  gg::Args a;
  a.offsets = d.offsets;
  a.E = d.E;
  a.shared = d.Bs != nullptr;
  a.R = d.R;
  a.T = d.T;
  a.K = d.K;
  a.mode = d.mode;
  a.slot_expert = d.slot_expert;
  a.I = d.I;
  // the router: 256-wide tiles (one pass over each activation tile for 256 experts) unless its K range is
  // split over CTAs (a small batch), where 128-wide tiles keep the partial sums small
  a.rbn = d.mode == 2 && d.csplit <= 1 ? gg::BN : gg::BN / 2;
  a.n_tiles = d.mode == 0 ? d.I / (gg::BN / 2) : (int)cdiv(d.N, d.mode == 2 ? a.rbn : gg::BN);
  a.ksplit = ksplit;
  a.csplit = d.mode == 2 && d.csplit > 1 ? d.csplit : 1;
  a.n_valid = d.N;
  a.ldo = d.ldo;
  a.vec32 = (reinterpret_cast<uintptr_t>(d.out) & 31) == 0 && ((int64_t)d.ldo * 2) % 32 == 0;
  a.out = d.out;
  a.row_weight = d.row_weight;
  a.status = d.status;
  a.wait_limit = 4000000000LL;  // about two seconds of SM clock
  if (d.mode == 2)
    gg::grouped_gemm_bf16_kernel<gg::ROUTER_THREADS>
        <<<num_sms(), gg::ROUTER_THREADS, gg::SMEM_BYTES, stream>>>(tA, tB, tBs, a);
  else
    gg::grouped_gemm_bf16_kernel<gg::THREADS><<<num_sms(), gg::THREADS, gg::SMEM_BYTES, stream>>>(tA, tB, tBs, a);
  return cudaGetLastError();
}

// Failure-detection self-test: one thread waits, through the bounded wait every pipeline stage of
// the grouped GEMMs uses, on an mbarrier that nothing arrives on. After `limit` SM clocks the wait
// records MOE_STATUS_WAIT_TIMEOUT in *status and returns, so the kernel ends and the context stays
// usable.
__global__ void wait_timeout_selftest_kernel(int* status, long long limit) {
  __shared__ uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) grp::wait_or_abort(&bar, 0, &abort_flag, status, limit);  // phase 0 never completes
}

cudaError_t launch_wait_timeout_selftest(int* status, long long limit_cycles, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_cycles);
  return cudaGetLastError();
}

}  // namespace moe
