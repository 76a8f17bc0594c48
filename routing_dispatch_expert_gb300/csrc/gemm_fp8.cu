// FP8 block-scaled grouped GEMM of the expert FFN (tcgen05 kind::f8f6f4, TMEM, TMA).
//
// Perplexity blog "Lower latency and higher throughput with multi-node DeepSeek deployment",
// "Quantization": weights are quantised statically per 128x128 tile, activations at run time per
// 1x128 vector along K, so a product [M, K] x [K, N] needs the scales (M x K/128) and
// (K/128 x N/128); the activation scales vary only along K. The SiLU output is itself block
// quantised with a 128-element amax before the down projection. Same grouping as the bf16 kernel:
//   mode 0  H (e4m3, 1x128 scales) = quant( silu(A W_gate^T) * (A W_up^T) )
//   mode 1  yd (bf16)              = (A W_down^T) * row_weight
// with A = e4m3 rows [R_tot, K] and per-row scales [R_tot, K/128].
//
// One 128-deep K block is exactly one scale block, so the tensor core computes each K block's
// product in a fresh TMEM partial (2 x 256 columns, double buffered) and sixteen epilogue warps
// promote it: acc += partial * sa[row, kb] * sb[n_block, kb], in fp32 registers (64 per thread; four
// warps share each TMEM lane quarter, one per quarter of the columns; two accumulators per packed
// IEEE fma of a float2). The MMA of block kb+1 overlaps the promotion of block kb; four promotion
// warps per SM sub-partition hide the TMEM-load latency. The scales reach the promotion warps through
// shared memory: a loader warp fetches them 8 K blocks at a time into a 16-slot ring ahead of use,
// because a global load in the promotion loop waits for DRAM (the activation scales of a large batch
// are evicted from L2 by the streaming weights) on every K block. The partial is read 8 columns at a time so
// that 64 accumulators plus the loaded values fit the 96 registers a 576-thread CTA allows without
// spilling (spilled values compete with the 192 KB TMA ring for the SM's L1), and the TMEM buffer is
// handed back as soon as its last columns are in registers.
//   * mode 0: each thread holds 32 gate and the 32 matching up columns of its row, so SwiGLU is local;
//     the 128-column amax of H is shared by the four warps of a row through shared memory and a
//     bounded mbarrier (never a blocking bar.sync, so a timed-out warp cannot hang the others).
//   * persistent, one CTA per SM, 4-stage TMA ring of 48 KB (A 128 x 128 B, B 256 x 128 B), every
//     wait bounded, the same exit path as the bf16 kernel; warps: 0 TMA, 1 MMA, 2-17 promotion and
//     epilogue, 18 scale loader.
#include <cuda.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {
namespace g8 {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // e4m3 elements per 128-byte swizzled row = one scale block along K
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 16;
constexpr int PARTS = EPI_WARPS / 4;  // column parts per TMEM lane quarter
constexpr int SCALE_WARP = 2 + EPI_WARPS;  // stages the scales of each K block into shared memory
constexpr int THREADS = 64 + 32 * EPI_WARPS + 32;
constexpr int SRING = 16;  // K blocks of scales in the shared-memory ring
constexpr int SCHUNK = 8;  // K blocks the scale loader fetches at once
constexpr int TMEM_COLS = 2 * BN;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;

struct Args {
  const int32_t* offsets;
  const int32_t* slot_expert;  // routed group -> logical expert (nullptr: identity)
  int E, shared, R, T, K, n_tiles, mode, I, ldo;
  void* out;               // mode 0: H codes [R_tot, I]; mode 1: yd bf16 [R_tot, ldo]
  float* out_scales;       // mode 0: H scales [R_tot, I / 128]
  const float* a_scales;   // [R_tot, K / 128]
  const float* b_scales;   // routed weights [E, nb, K / 128]
  const float* bs_scales;  // shared expert [nb, K / 128]
  int nb;                  // 128-row blocks of the weight
  const float* row_weight;
  int* status;
  long long wait_limit;
};

// The scales of one K block of a tile: the A scale of each of its 128 rows and the B scale of each
// of its two 128-column blocks (mode 0: the gate block, the up block; mode 1: columns [0, 128) and
// [128, 256)).
struct ScaleSlot {
  float a[BM];
  float b[2];
  float pad[2];
};

struct Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t sfull[SRING];
  uint64_t sempty[SRING];
  uint64_t pfull[2];
  uint64_t pempty[2];
  uint64_t xchg;
  uint64_t mma_done;
  uint32_t tmem_slot;
  volatile int abort_flag;
  float amax[2][PARTS][BM];  // [tile parity][column part][row]
  ScaleSlot sc[SRING];
  grp::Table tb;
};

using grp::wait_or_abort;

__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmBs, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared s;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.E + args.shared;

  if (warp == 0) {
    grp::build_table(s.tb, args.offsets, args.E, args.shared, args.R, args.T, BM, lane);
    if (lane == 0) {
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(&s.full[i], 1);
        mbar_init(&s.empty[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.pfull[i], 1);
        mbar_init(&s.pempty[i], 32 * EPI_WARPS);
      }
      mbar_init(&s.xchg, EPI_WARPS);
      for (int i = 0; i < SRING; ++i) {
        mbar_init(&s.sfull[i], 32);
        mbar_init(&s.sempty[i], 32 * EPI_WARPS);
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
  const int total = s.tb.gtile[G] * args.n_tiles;
  const int kblocks = args.K / BK;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const grp::Tile t = grp::decode(s.tb, G, args.n_tiles, tile, BM);
      const CUtensorMap* mb = t.g < args.E ? &tmB : &tmBs;
      const int z = t.g < args.E ? (args.slot_expert ? args.slot_expert[t.g] : t.g) : 0;
      int n0, n1;
      if (args.mode == 0) {
        n0 = t.n_tile * (BN / 2);
        n1 = args.I + t.n_tile * (BN / 2);
      } else {
        n0 = t.n_tile * BN;
        n1 = n0 + BN / 2;
      }
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&s.empty[stage], phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        uint8_t* a = smem + stage * STAGE_BYTES;
        uint8_t* b = a + A_BYTES;
        mbar_arrive_expect_tx(&s.full[stage], STAGE_BYTES);
        tma_load_2d(a, &tmA, &s.full[stage], kb * BK, t.a_row);
        tma_load_3d(b, mb, &s.full[stage], kb * BK, n0, z);
        tma_load_3d(b + B_BYTES / 2, mb, &s.full[stage], kb * BK, n1, z);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    const long long first = issued > STAGES ? issued - STAGES : 0;
    for (long long i = first; i < issued; ++i)
      grp::drain_wait(&s.full[i % STAGES], (uint32_t)((i / STAGES) & 1), args.wait_limit);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: one K block per TMEM partial
    constexpr uint32_t IDESC = idesc_e4m3(BM, BN);
    int stage = 0, p = 0;
    uint32_t phase = 0, pphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&s.pempty[p], pphase ^ 1, &s.abort_flag, args.status, args.wait_limit) ||
            !wait_or_abort(&s.full[stage], phase, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(p * BN);
        const uint32_t a = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t b = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk)
          umma_f8(d, sw128_kmajor_desc(a + kk * 32), sw128_kmajor_desc(b + kk * 32), IDESC, kk != 0);
        umma_commit(&s.empty[stage]);
        umma_commit(&s.pfull[p]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
        p ^= 1;
        if (p == 0) pphase ^= 1;
      }
    }
    umma_commit(&s.mma_done);
    grp::drain_wait(&s.mma_done, 0, args.wait_limit);
  } else if (warp == SCALE_WARP) {
    // ---------------- scale loader: the scales of SCHUNK K blocks at a time into the ring, so that
    // the promotion warps read them from shared memory instead of waiting on global loads (the
    // activation scales of a large batch do not stay in L2 next to the streaming weights)
    const int KB = kblocks;
    const int R_tot = args.R + (args.shared ? args.T : 0);
    const bool vec = (KB & 3) == 0 && (reinterpret_cast<uintptr_t>(args.a_scales) & 15) == 0;
    int q = 0;
    uint32_t qphase = 0;
    bool fine = true;
    for (int tile = blockIdx.x; tile < total && fine; tile += gridDim.x) {
      const grp::Tile t = grp::decode(s.tb, G, args.n_tiles, tile, BM);
      const float* bsc = t.g < args.E ? args.b_scales : args.bs_scales;
      const int gbase = t.g < args.E ? (args.slot_expert ? args.slot_expert[t.g] : t.g) * args.nb * KB : 0;
      const int nb0 = args.mode == 0 ? t.n_tile : t.n_tile * 2;
      const int nb1 = args.mode == 0 ? args.I / 128 + t.n_tile : t.n_tile * 2 + 1;
      const float* bl = bsc + gbase + (lane == 0 ? nb0 : nb1) * KB;
      const float* ar[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) ar[i] = args.a_scales + (int64_t)min(t.a_row + lane + 32 * i, R_tot - 1) * KB;
      for (int kc = 0; kc < KB && fine; kc += SCHUNK) {
        const int n = min(SCHUNK, KB - kc);
        float av[4][SCHUNK], bv[SCHUNK];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (vec && n == SCHUNK) {
            const float4 u = *reinterpret_cast<const float4*>(ar[i] + kc);
            const float4 w = *reinterpret_cast<const float4*>(ar[i] + kc + 4);
            av[i][0] = u.x, av[i][1] = u.y, av[i][2] = u.z, av[i][3] = u.w;
            av[i][4] = w.x, av[i][5] = w.y, av[i][6] = w.z, av[i][7] = w.w;
          } else {
#pragma unroll
            for (int j = 0; j < SCHUNK; ++j) av[i][j] = j < n ? ar[i][kc + j] : 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < SCHUNK; ++j) bv[j] = (lane < 2 && j < n) ? bl[kc + j] : 0.f;
#pragma unroll
        for (int j = 0; j < SCHUNK; ++j) {
          if (j >= n) break;
          int ok = 1;
          if (lane == 0) ok = wait_or_abort(&s.sempty[q], qphase ^ 1, &s.abort_flag, args.status, args.wait_limit);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            fine = false;
            break;
          }
          __syncwarp();  // the slot is free for every lane, not only the one that waited
#pragma unroll
          for (int i = 0; i < 4; ++i) s.sc[q].a[lane + 32 * i] = av[i][j];
          if (lane < 2) s.sc[q].b[lane] = bv[j];
          mbar_arrive(&s.sfull[q]);
          if (++q == SRING) {
            q = 0;
            qphase ^= 1;
          }
        }
      }
    }
  } else if (warp >= 2) {
    // ---------------- promotion + epilogue (16 warps)
    const int quarter = warp & 3;
    const int part = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    // mode 0: gate columns [32 part, +32) and the matching up columns; mode 1: columns [64 part, +64)
    const int col_a = args.mode == 0 ? part * 32 : part * 64;
    const int col_b = args.mode == 0 ? BN / 2 + part * 32 : part * 64 + 32;
    const uint32_t tq = tmem_base + ((uint32_t)(quarter * 32) << 16);  // this warp's TMEM lane quarter
    const uint32_t tqa = tq + (uint32_t)col_a, tqb = tq + (uint32_t)col_b;
    const int KB = kblocks;
    int p = 0, tpar = 0;
    uint32_t pphase = 0, xphase = 0;
    bool fine = true;
    // column block of this thread's scales: mode 0 gate (block 0) and up (block 1); mode 1 the block
    // holding its 64 columns
    const int blo = args.mode == 0 ? 0 : part >> 1;
    const int bhi = args.mode == 0 ? 1 : part >> 1;
    int q = 0;
    uint32_t qphase = 0;
    for (int tile = blockIdx.x; tile < total && fine; tile += gridDim.x) {
      // acc[i] holds columns (2i, 2i+1) of this thread's 64: [0, 16) the col_a block, [16, 32) col_b
      float2 acc[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.f, 0.f);
      for (int kb = 0; kb < KB; ++kb) {
        // every lane polls the barrier itself: a lane-0 wait followed by a broadcast costs ~7% of the
        // FFN on this per-K-block hand-off
        int ok = wait_or_abort(&s.sfull[q], qphase, &s.abort_flag, args.status, args.wait_limit);
        if (__any_sync(0xffffffffu, !ok)) {
          fine = false;
          break;
        }
        __syncwarp();
        // the scales of this K block (rows past the buffer carry the last row's scale and are never
        // stored); the slot is handed back once they are in registers
        const float sa = s.sc[q].a[r];
        const float s_lo = sa * s.sc[q].b[blo], s_hi = sa * s.sc[q].b[bhi];
        mbar_arrive(&s.sempty[q]);
        if (++q == SRING) {
          q = 0;
          qphase ^= 1;
        }
        const float2 slo = make_float2(s_lo, s_lo), shi = make_float2(s_hi, s_hi);
        ok = wait_or_abort(&s.pfull[p], pphase, &s.abort_flag, args.status, args.wait_limit);
        if (__any_sync(0xffffffffu, !ok)) {
          fine = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
        const uint32_t pofs = (uint32_t)(p * BN);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint32_t v[8];
          tmem_ld8((g < 4 ? tqa : tqb) + pofs + (g & 3) * 8, v);
          tmem_ld_wait_regs(v);
          if (g == 7) {
            // the partial is in registers: hand the TMEM buffer back before the last multiply-adds
            tc_fence_before();
            mbar_arrive(&s.pempty[p]);  // every lane arrives (the barrier counts 32 per warp)
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            acc[4 * g + i] = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                        g < 4 ? slo : shi, acc[4 * g + i]);
        }
        p ^= 1;
        if (p == 0) pphase ^= 1;
      }
      if (!fine) break;

      const grp::Tile t = grp::decode(s.tb, G, args.n_tiles, tile, BM);
      const bool valid = r < t.rows;
      const int64_t row = (int64_t)t.a_row + r;
      if (args.mode == 1) {
        const float w = (valid && t.g < args.E) ? args.row_weight[row] : 1.0f;
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(args.out) + row * args.ldo +
                                                t.n_tile * BN + part * 64);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_uint4(pack_bf16x2(acc[4 * i].x * w, acc[4 * i].y * w),
                                pack_bf16x2(acc[4 * i + 1].x * w, acc[4 * i + 1].y * w),
                                pack_bf16x2(acc[4 * i + 2].x * w, acc[4 * i + 2].y * w),
                                pack_bf16x2(acc[4 * i + 3].x * w, acc[4 * i + 3].y * w));
        }
      } else {
        // SwiGLU on this thread's 32 columns, then the row's 128-column amax shared by the four parts
        float h[32];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          h[2 * i] = grp::silu(acc[i].x) * acc[16 + i].x;
          h[2 * i + 1] = grp::silu(acc[i].y) * acc[16 + i].y;
          amax = fmaxf(amax, fmaxf(fabsf(h[2 * i]), fabsf(h[2 * i + 1])));
        }
        s.amax[tpar][part][r] = amax;
        __syncwarp();
        int ok = 1;
        if (lane == 0) {
          mbar_arrive(&s.xchg);
          ok = wait_or_abort(&s.xchg, xphase, &s.abort_flag, args.status, args.wait_limit);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        xphase ^= 1;
        if (!ok) break;
        float row_amax = s.amax[tpar][0][r];
#pragma unroll
        for (int q = 1; q < PARTS; ++q) row_amax = fmaxf(row_amax, s.amax[tpar][q][r]);
        tpar ^= 1;
        const float scale = row_amax > 0.f ? __fdiv_rn(row_amax, 448.0f) : 1.0f;
        if (valid) {
          uint32_t q[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t w4 = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              w4 |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(h[4 * i + j], scale), __NV_SATFINITE, __NV_E4M3)
                    << (8 * j);
            q[i] = w4;
          }
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(args.out) + row * args.ldo +
                                                t.n_tile * (BN / 2) + part * 32);
          dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
          dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
          if (part == 0) args.out_scales[row * (args.I / 128) + t.n_tile] = scale;
        }
      }
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

}  // namespace g8

cudaError_t launch_grouped_gemm_fp8(const GroupedGemmFp8Desc& d, cudaStream_t stream, std::string* err) {
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
        const cudaError_t r =
            cudaFuncSetAttribute(g8::grouped_gemm_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, g8::SMEM_BYTES);
        v = r == cudaSuccess;
        return r;
      },
      &attr_set);
  if (e != cudaSuccess) {
    *err = "cudaFuncSetAttribute failed";
    return e;
  }
  CUtensorMap tA, tB, tBs;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  bool ok = tma_encode_2d(&tA, d.A, U8, 1, d.a_rows, d.K, g8::BM) &&
            tma_encode_3d(&tB, d.B, U8, 1, d.n_experts > 0 ? d.n_experts : d.E, d.b_rows, d.K, g8::BN / 2) &&
            tma_encode_3d(&tBs, d.Bs ? d.Bs : d.B, U8, 1, 1, d.b_rows, d.K, g8::BN / 2);
  if (!ok) {
    *err = "cuTensorMapEncodeTiled rejected an FP8 grouped-GEMM operand";
    return cudaErrorInvalidValue;
  }
  g8::Args a;
  a.offsets = d.offsets;
  a.slot_expert = d.slot_expert;
  a.E = d.E;
  a.shared = d.Bs != nullptr;
  a.R = d.R;
  a.T = d.T;
  a.K = d.K;
  a.mode = d.mode;
  a.I = d.I;
  a.n_tiles = d.mode == 0 ? d.I / (g8::BN / 2) : d.N / g8::BN;
  a.ldo = d.ldo;
  a.out = d.out;
  a.out_scales = d.out_scales;
  a.a_scales = d.a_scales;
  a.b_scales = d.b_scales;
  a.bs_scales = d.Bs ? d.bs_scales : d.b_scales;
  a.nb = (int)(d.b_rows / 128);
  a.row_weight = d.row_weight;
  a.status = d.status;
  a.wait_limit = 4000000000LL;
  g8::grouped_gemm_fp8_kernel<<<num_sms(), g8::THREADS, g8::SMEM_BYTES, stream>>>(tA, tB, tBs, a);
  return cudaGetLastError();
}

}  // namespace moe
