// Expert-FFN grouped GEMM with NVFP4 expert weights and bf16 activations (tcgen05, TMEM, TMA).
//
// TensorRT-LLM "DeepSeek R1 throughput on Blackwell", "Precision strategy": the MoE weights of the
// Blackwell deployment are FP4, which halves the weight bytes a memory-bound decode step streams.
// The page does not fix the format; the layout here is NVFP4: e2m1 codes (two per byte), one e4m3
// scale per 16 consecutive elements along K, one fp32 scale per matrix. The activations stay bf16.
// Same two launches and grouping as the bf16 kernel (gemm.cu):
//   mode 0  H  = silu(A W_gate^T) * (A W_up^T)     A = xd [R_tot, h], W_gu [E, 2I, h]
//   mode 1  yd = (A W_down^T) * row_weight         A = H  [R_tot, I], W_d  [E, h, I]
//
// The weight tile travels in FP4 (9 KB of codes and scales per 256 x 64 tile instead of 32 KB of
// bf16) and is expanded in shared memory: e2m1 x e4m3 has at most 6 significant bits, so the product
// is exact in bf16, and the bf16 tensor-core MMA then runs unchanged; the fp32 matrix scale
// multiplies the accumulator in the epilogue. (The block-scaled FP4 MMA would need FP4 activations as
// well.)
//
// Roles, 736 threads: warp 0 lane 0 TMA producer of the weight codes and scales, warp 6 lane 0 TMA
// producer of the activation tiles, warp 1 lane 0 MMA issuer, warps 2-5 epilogue, warps 7-22 expand
// the weight tile in two groups of eight that take alternate K blocks (within a group two half rows
// per thread: 16 bytes of codes and 2 scale bytes -> 32 bf16 each, written in the 128-byte-swizzled
// K-major layout the MMA reads). Rings: activations 3 x 16 KB, FP4 tiles 6 x 12 KB, bf16 weight tiles
// 3 x 32 KB. The FP4 ring waits only on the converters, so the weight stream runs ahead of the MMA
// (with one producer for both rings, an FP4 load waited for the MMA to free the activation stage it
// shared). Every wait is bounded; a time-out records MOE_STATUS_WAIT_TIMEOUT and every role returns.
#include <cuda.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {
namespace g4 {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
// K block i uses activation stage i % STAGES and expanded-weight stage i % STAGES, released together
constexpr int STAGES = 3;   // activation and expanded bf16 weight rings
constexpr int QSTAGES = 6;  // FP4 weight ring (codes and scales)
constexpr int A_BYTES = BM * BK * 2;
constexpr int QC_BYTES = BN * BK / 2;  // codes: 256 rows x 32 bytes
constexpr int QS_BYTES = BN * 16;      // scales: 256 rows x 16 bytes (the scales of 4 K blocks)
constexpr int Q_BYTES = QC_BYTES + QS_BYTES;
constexpr int B_BYTES = BN * BK * 2;
constexpr int CONV_GROUP_WARPS = 8;  // one converter group: one weight row per thread (256 rows)
constexpr int CONV_GROUPS = 2;       // groups take alternate K blocks, so two stages expand at once
constexpr int CONV_WARPS = CONV_GROUP_WARPS * CONV_GROUPS;
constexpr int CONV_WARP0 = 7;  // warps 0-6: FP4 producer, MMA, four epilogue warps, activation producer
constexpr int THREADS = 32 * (CONV_WARP0 + CONV_WARPS);
constexpr int TMEM_COLS = 2 * BN;
constexpr int SMEM_BYTES = STAGES * (A_BYTES + B_BYTES) + QSTAGES * Q_BYTES + 1024;

struct Args {
  const int32_t* offsets;
  const int32_t* slot_expert;
  int E, shared, R, T, K, n_tiles, mode, I, ldo;
  const float* g;         // routed matrix scales [n_experts]
  const float* g_shared;  // [1]
  void* out;
  const float* row_weight;
  int* status;
  long long wait_limit;
};

struct Shared {
  // full[i]: the activation tile landed and eight converter warps wrote the weight tile; empty[i]:
  // the MMAs of the K block that read both finished
  uint64_t full[STAGES], empty[STAGES];
  uint64_t qfull[QSTAGES], qempty[QSTAGES];
  uint64_t tfull[2], tempty[2];
  uint64_t mma_done;
  uint32_t tmem_slot;
  volatile int abort_flag;
  grp::Table tb;
};

using grp::silu;
using grp::Tile;
using grp::wait_or_abort;

// e2m1 pair (low nibble -> low half) times an e4m3 scale, as two exact bf16 values: the hardware
// converts the pair to f16x2, the product with the scale (at most 6 significant bits) is exact in f16
// and in bf16.
__device__ __forceinline__ uint32_t expand2(uint32_t byte, __half2 s2) {
  const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)byte, __NV_E2M1);
  const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&r), s2);
  const __nv_bfloat162 b = __float22bfloat162_rn(__half22float2(v));
  return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA64,
                              const __grid_constant__ CUtensorMap tmQ,
                              const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmQs,
                              const __grid_constant__ CUtensorMap tmSs, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared s;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_a = smem;
  uint8_t* ring_q = ring_a + STAGES * A_BYTES;
  uint8_t* ring_b = ring_q + QSTAGES * Q_BYTES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.E + args.shared;

  if (warp == 0) {
    grp::build_table(s.tb, args.offsets, args.E, args.shared, args.R, args.T, BM, lane);
    if (lane == 0) {
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(&s.full[i], CONV_GROUP_WARPS + 1);  // the converter warps + the activation producer
        mbar_init(&s.empty[i], 1);
      }
      for (int i = 0; i < QSTAGES; ++i) {
        mbar_init(&s.qfull[i], 1);
        mbar_init(&s.qempty[i], CONV_GROUP_WARPS);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.tfull[i], 1);
        mbar_init(&s.tempty[i], 4);
      }
      mbar_init(&s.mma_done, 1);
      s.abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA64);
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmS);
      tma_prefetch_desc(&tmQs);
      tma_prefetch_desc(&tmSs);
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
    // ---------------- TMA producer of the FP4 weight tiles (codes and scales). Its ring is deeper than
    // the activation ring and waits only on the converters, so the weight stream runs ahead of the MMA.
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = grp::decode(s.tb, G, args.n_tiles, tile, BM);
      const bool routed = t.g < args.E;
      const CUtensorMap* mq = routed ? &tmQ : &tmQs;
      const CUtensorMap* ms = routed ? &tmS : &tmSs;
      const int z = routed ? (args.slot_expert ? args.slot_expert[t.g] : t.g) : 0;
      // weight rows of the two 128-row halves: mode 0 the gate block and its up block
      const int r0 = args.mode == 0 ? t.n_tile * (BN / 2) : t.n_tile * BN;
      const int r1 = args.mode == 0 ? args.I + t.n_tile * (BN / 2) : r0 + BN / 2;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&s.qempty[stage], phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        uint8_t* q = ring_q + stage * Q_BYTES;
        mbar_arrive_expect_tx(&s.qfull[stage], Q_BYTES);
        tma_load_3d(q, mq, &s.qfull[stage], kb * (BK / 2), r0, z);
        tma_load_3d(q + QC_BYTES / 2, mq, &s.qfull[stage], kb * (BK / 2), r1, z);
        tma_load_3d(q + QC_BYTES, ms, &s.qfull[stage], (kb / 4) * 16, r0, z);
        tma_load_3d(q + QC_BYTES + QS_BYTES / 2, ms, &s.qfull[stage], (kb / 4) * 16, r1, z);
        ++issued;
        if (++stage == QSTAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    const long long first = issued > QSTAGES ? issued - QSTAGES : 0;
    for (long long i = first; i < issued; ++i)
      grp::drain_wait(&s.qfull[i % QSTAGES], (uint32_t)((i / QSTAGES) & 1), args.wait_limit);
  } else if (warp == CONV_WARP0 - 1 && lane == 0) {
    // ---------------- TMA producer of the activation tiles
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = grp::decode(s.tb, G, args.n_tiles, tile, BM);
      const bool half = t.rows <= BM / 2;  // 64 rows or fewer: a 64-row activation box, an M = 64 MMA
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&s.empty[stage], phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        uint8_t* a = ring_a + stage * A_BYTES;
        mbar_arrive_expect_tx(&s.full[stage], half ? A_BYTES / 2 : A_BYTES);
        tma_load_2d(a, half ? &tmA64 : &tmA, &s.full[stage], kb * BK, t.a_row);
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
    // ---------------- MMA issuer
    const uint32_t idesc_full = idesc_bf16(BM, BN), idesc_half = idesc_bf16(BM / 2, BN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const uint32_t idesc =
          grp::decode(s.tb, G, args.n_tiles, tile, BM).rows <= BM / 2 ? idesc_half : idesc_full;
      if (!wait_or_abort(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) break;
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&s.full[stage], phase, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // one descriptor per operand tile: the K step kk starts 32 bytes further, 2 in the descriptor's
        // 16-byte address field (a shared-memory address >> 4 stays below 2^14, so nothing carries).
        // The issuing thread shares its SM sub-partition with converter warps: every instruction
        // taken out of this loop shortens the K block.
        const uint64_t da = sw128_kmajor_desc(smem_u32(ring_a + stage * A_BYTES));
        const uint64_t db = sw128_kmajor_desc(smem_u32(ring_b + stage * B_BYTES));
        umma_f16(d, da, db, idesc, kb != 0);
        umma_f16(d, da + 2, db + 2, idesc, 1);
        umma_f16(d, da + 4, db + 4, idesc, 1);
        umma_f16(d, da + 6, db + 6, idesc, 1);
        umma_commit(&s.empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      umma_commit(&s.tfull[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    umma_commit(&s.mma_done);
    grp::drain_wait(&s.mma_done, 0, args.wait_limit);
  } else if (warp >= CONV_WARP0) {
    // ---------------- weight expansion: FP4 row -> 64 bf16 in the swizzled operand layout. Each group
    // of eight warps expands every other K block (group g the blocks i with i % 2 == g), so one
    // group's loads, conversions, stores and proxy fence of a stage overlap the other group's.
    const int cw = warp - CONV_WARP0;
    const int cgroup = cw / CONV_GROUP_WARPS;
    // thread j of the group takes the half rows (j / 2 + 128 p, half j % 2), p = 0, 1: a warp's code
    // loads are then 512 consecutive bytes (no bank conflicts on the 32-byte rows of the FP4 tile)
    const int j = (cw % CONV_GROUP_WARPS) * 32 + lane;
    const int hh = j & 1;
    int stage = 0, bst = 0;
    uint32_t phase = 0, bphase = 0;
    bool fine = true;
    long long seen = 0;  // K blocks of this CTA so far
    for (int tile = blockIdx.x; tile < total && fine; tile += gridDim.x) {
      for (int kb = 0; kb < kblocks; ++kb, ++seen) {
        if ((int)(seen % CONV_GROUPS) != cgroup) {
          if (++stage == QSTAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (++bst == STAGES) {
            bst = 0;
            bphase ^= 1;
          }
          continue;
        }
        // every lane polls the barriers itself (cheaper than a lane-0 wait and a broadcast)
        const int ok = wait_or_abort(&s.qfull[stage], phase, &s.abort_flag, args.status, args.wait_limit) &&
                       wait_or_abort(&s.empty[bst], bphase ^ 1, &s.abort_flag, args.status, args.wait_limit);
        if (__any_sync(0xffffffffu, !ok)) {
          fine = false;
          break;
        }
        __syncwarp();
        const uint8_t* q = ring_q + stage * Q_BYTES;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const int n = (j >> 1) + 128 * p;  // weight-tile row
          const uint4 cv = *reinterpret_cast<const uint4*>(q + n * 32 + hh * 16);
          const uint32_t sc2 = *reinterpret_cast<const uint16_t*>(q + QC_BYTES + n * 16 + (kb & 3) * 4 + hh * 2);
          const uint32_t words[4] = {cv.x, cv.y, cv.z, cv.w};
          uint8_t* brow = ring_b + bst * B_BYTES + n * 128;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const __half_raw sr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)((sc2 >> (8 * b)) & 0xFF), __NV_E4M3);
            const __half sh = *reinterpret_cast<const __half*>(&sr);
            const __half2 s2 = __halves2half2(sh, sh);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = 4 * hh + 2 * b + h;  // 16-byte chunk of the row: 8 elements
              const uint32_t w = words[2 * b + h];
              const uint4 o = make_uint4(expand2(w & 0xFF, s2), expand2((w >> 8) & 0xFF, s2),
                                         expand2((w >> 16) & 0xFF, s2), expand2(w >> 24, s2));
              *reinterpret_cast<uint4*>(brow + ((c ^ (n & 7)) << 4)) = o;
            }
          }
        }
        fence_proxy_async_smem();  // the tensor core reads this tile through the async proxy
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s.full[bst]);
          mbar_arrive(&s.qempty[stage]);
        }
        if (++stage == QSTAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (++bst == STAGES) {
          bst = 0;
          bphase ^= 1;
        }
      }
    }
  } else if (warp >= 2 && warp < CONV_WARP0 - 1) {
    // ---------------- epilogue: TMEM -> registers -> global, times the matrix scale
    const int quarter = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = grp::decode(s.tb, G, args.n_tiles, tile, BM);
      // an M = 128 tile keeps row r in TMEM lane r; an M = 64 tile keeps rows 16q .. 16q + 15 in lanes
      // 32q .. 32q + 15 (lanes 32q + 16 .. 32q + 31 hold nothing)
      const bool half = t.rows <= BM / 2;
      const int r = half ? quarter * 16 + (lane & 15) : quarter * 32 + lane;
      int ok = 1;
      if (lane == 0) ok = wait_or_abort(&s.tfull[acc], acc_phase, &s.abort_flag, args.status, args.wait_limit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      const bool valid = (!half || lane < 16) && r < t.rows;
      const int64_t orow = (int64_t)t.a_row + r;
      const float gs = t.g < args.E ? args.g[args.slot_expert ? args.slot_expert[t.g] : t.g] : args.g_shared[0];
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (args.mode == 0) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out) + orow * args.ldo + t.n_tile * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c, g);
          tmem_ld32(taddr + BN / 2 + c, u);
          tmem_ld_wait_regs(g);
          tmem_ld_wait_regs(u);
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = silu(__uint_as_float(g[2 * i]) * gs) * (__uint_as_float(u[2 * i]) * gs);
            const float h1 = silu(__uint_as_float(g[2 * i + 1]) * gs) * (__uint_as_float(u[2 * i + 1]) * gs);
            p[i] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
          }
        }
      } else {
        const float w = ((valid && t.g < args.E) ? args.row_weight[orow] : 1.0f) * gs;
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out) + orow * args.ldo + t.n_tile * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_ld_wait_regs(v);
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * w, __uint_as_float(v[2 * i + 1]) * w);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
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

// ------------------------------------------------------------------------------------------
// NVFP4 weight quantisation: matrix amax (gathered as float bits in g), blocks, matrix scale.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint4* __restrict__ w, int64_t per_mat,
                                                         uint32_t* __restrict__ amax_bits) {
  __shared__ float red[8];
  const int64_t b = blockIdx.y;
  const uint4* m = w + b * per_mat;
  float amax = 0.f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < per_mat; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = m[i];
    const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(a[j])), fabsf(bf16_hi(a[j]))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    atomicMax(amax_bits + b, __float_as_uint(fmaxf(amax, red[0])));  // non-negative floats order as integers
  }
}

__device__ __forceinline__ float nvfp4_matrix_scale(uint32_t amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  return amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;  // 6 (largest e2m1) x 448 (largest e4m3)
}

// one thread per 16-element block of a row
__global__ void __launch_bounds__(256) nvfp4_quant_kernel(const uint4* __restrict__ w, int64_t blocks_per_mat,
                                                          int64_t n_blocks, const uint32_t* __restrict__ amax_bits,
                                                          uint2* __restrict__ q, uint8_t* __restrict__ s) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_blocks; i += (int64_t)gridDim.x * blockDim.x) {
    const float gs = nvfp4_matrix_scale(amax_bits[i / blocks_per_mat]);
    const uint4 v0 = w[2 * i], v1 = w[2 * i + 1];
    const uint32_t a[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float x[16];
    float bmax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x[2 * j] = bf16_lo(a[j]);
      x[2 * j + 1] = bf16_hi(a[j]);
      bmax = fmaxf(bmax, fmaxf(fabsf(x[2 * j]), fabsf(x[2 * j + 1])));
    }
    const __nv_fp8_storage_t sc =
        __nv_cvt_float_to_fp8(__fdiv_rn(bmax, __fmul_rn(6.0f, gs)), __NV_SATFINITE, __NV_E4M3);
    const __half_raw sr = __nv_cvt_fp8_to_halfraw(sc, __NV_E4M3);
    const float p = __fmul_rn(__half2float(*reinterpret_cast<const __half*>(&sr)), gs);
    uint32_t out[2] = {0, 0};
    if (p != 0.f) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t c = __nv_cvt_float_to_fp4(__fdiv_rn(x[j], p), __NV_E2M1, cudaRoundNearest) & 0xF;
        out[j / 8] |= c << (4 * (j % 8));
      }
    }
    q[i] = make_uint2(out[0], out[1]);
    s[i] = (uint8_t)sc;
  }
}

__global__ void nvfp4_scale_kernel(uint32_t* g, int64_t batch) {
  const int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (b < batch) g[b] = __float_as_uint(nvfp4_matrix_scale(g[b]));
}

}  // namespace g4

cudaError_t launch_grouped_gemm_nvfp4(const GroupedGemmFp4Desc& d, cudaStream_t stream, std::string* err) {
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
            cudaFuncSetAttribute(g4::grouped_gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, g4::SMEM_BYTES);
        v = r == cudaSuccess;
        return r;
      },
      &attr_set);
  if (e != cudaSuccess) {
    *err = "cudaFuncSetAttribute failed";
    return e;
  }
  const int64_t G = d.n_experts > 0 ? d.n_experts : d.E;
  CUtensorMap tA, tA64, tQ, tS, tQs, tSs;
  bool ok = tma_encode_2d(&tA, d.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d.a_rows, d.K, g4::BM) &&
            tma_encode_2d(&tA64, d.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d.a_rows, d.K, g4::BM / 2) &&
            tma_encode_3d_plain(&tQ, d.Bq, G, d.b_rows, d.K / 2, g4::BK / 2, g4::BN / 2) &&
            tma_encode_3d_plain(&tS, d.Bs, G, d.b_rows, d.K / 16, 16, g4::BN / 2) &&
            tma_encode_3d_plain(&tQs, d.Bq_shared ? d.Bq_shared : d.Bq, 1, d.b_rows, d.K / 2, g4::BK / 2, g4::BN / 2) &&
            tma_encode_3d_plain(&tSs, d.Bs_shared ? d.Bs_shared : d.Bs, 1, d.b_rows, d.K / 16, 16, g4::BN / 2);
  if (!ok) {
    *err = "cuTensorMapEncodeTiled rejected an NVFP4 grouped-GEMM operand";
    return cudaErrorInvalidValue;
  }
  g4::Args a;
  a.offsets = d.offsets;
  a.slot_expert = d.slot_expert;
  a.E = d.E;
  a.shared = d.Bq_shared != nullptr;
  a.R = d.R;
  a.T = d.T;
  a.K = d.K;
  a.mode = d.mode;
  a.I = d.I;
  a.n_tiles = d.mode == 0 ? d.I / (g4::BN / 2) : (int)cdiv(d.N, g4::BN);
  a.ldo = d.ldo;
  a.g = d.Bg;
  a.g_shared = d.Bg_shared ? d.Bg_shared : d.Bg;
  a.out = d.out;
  a.row_weight = d.row_weight;
  a.status = d.status;
  a.wait_limit = 4000000000LL;  // about two seconds of SM clock
  g4::grouped_gemm_nvfp4_kernel<<<num_sms(), g4::THREADS, g4::SMEM_BYTES, stream>>>(tA, tA64, tQ, tS, tQs, tSs, a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weights_nvfp4(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, void* s,
                                          float* g, cudaStream_t stream) {
  if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
  uint32_t* bits = reinterpret_cast<uint32_t*>(g);
  cudaError_t e = cudaMemsetAsync(bits, 0, sizeof(uint32_t) * batch, stream);
  if (e != cudaSuccess) return e;
  const int64_t per_mat = rows * cols / 8;  // uint4 per matrix
  int64_t bx = cdiv(per_mat, 256);
  if (bx > num_sms() * 4) bx = num_sms() * 4;
  g4::nvfp4_amax_kernel<<<dim3((unsigned)bx, (unsigned)batch), 256, 0, stream>>>(reinterpret_cast<const uint4*>(w),
                                                                                  per_mat, bits);
  const int64_t n_blocks = batch * rows * (cols / 16);
  int64_t qb = cdiv(n_blocks, 256);
  if (qb > (int64_t)num_sms() * 32) qb = (int64_t)num_sms() * 32;
  g4::nvfp4_quant_kernel<<<(unsigned)qb, 256, 0, stream>>>(reinterpret_cast<const uint4*>(w), rows * (cols / 16),
                                                           n_blocks, bits, reinterpret_cast<uint2*>(q),
                                                           reinterpret_cast<uint8_t*>(s));
  g4::nvfp4_scale_kernel<<<(unsigned)cdiv(batch, 256), 256, 0, stream>>>(bits, batch);
  return cudaGetLastError();
}

}  // namespace moe
