// Expert-FFN grouped GEMM (bf16) on CTA pairs: tcgen05.mma.cta_group::2 with 256 x 256 tiles.
//
// The same two launches as the single-CTA kernel of gemm.cu (Perplexity blog "Lower latency and
// higher throughput with multi-node DeepSeek deployment", "Roofline model / GroupGEMM"; inference
// guide 6.4, section 2.1, the SwiGLU FFN):
//   mode 0  H  = silu(A W_gate^T) * (A W_up^T)     A = xd [R_tot, h], W_gu [E, 2I, h]
//   mode 1  yd = (A W_down^T) * row_weight         A = H  [R_tot, I], W_d  [E, h, I]
// with the groups (routed experts, then the shared expert) walked in tiles of 256 rows.
//
// Why pairs. A single CTA's 128 x 256 tile needs 48 KB of operands per 64-deep K step. The copy of a
// step takes about 1.1 us from TMA issue to arrival under the load of a full GPU (weights stream from
// HBM, shared tiles come from the far L2), so keeping the tensor pipe busy takes more than 4 stages
// in flight: 6 stages x 48 KB do not fit in 227 KB of shared memory. A CTA pair computes a 256 x 256
// tile with one MMA stream: each CTA stages its own 128 rows of A and its own 128 columns of B, 32 KB
// per step, so 6 stages (192 KB) cover the latency, and the weight tile is read from L2 once per 256
// rows instead of once per 128. An expert's last tile, when it holds at most 128 rows, is a half tile:
// an M = 128 pair MMA (64 rows from each CTA), which runs at the same rate per SM, so the row padding
// stays at the 128-row granularity of single-CTA tiles. Its accumulator lands differently: in each CTA,
// lanes 0-63 hold the CTA's 64 rows for output columns [0, 128) and lanes 64-127 the same rows for
// columns [128, 256), in 128 TMEM columns. For the gate/up launch the B rows of a half tile are
// interleaved (leader: gate 0-63 and up 0-63 of the column tile; follower: gate 64-127 and up
// 64-127), so each lane still holds the gate and up value of its outputs.
//
// Schedule: persistent pairs take tiles in index order from a tile counter in global memory (one
// atomic per tile). Every pair starts on tile `pair`; the next tile is the counter's value plus the
// number of pairs. Pairs that run at the same time thus hold neighbouring tiles, which share a weight
// tile (row tiles of one column tile are neighbours) or a row tile, however unequal the tiles are
// (half tiles, short groups); a fixed stride per pair lets the pairs drift apart, after which those
// tiles are read from DRAM again. Without a counter the pair walks tiles pair, pair + pairs, ...
//
// Roles (192 threads per CTA; CTA rank 0 of the cluster is the leader):
//   * warp 0 lane 0 of each CTA: TMA producer into its own 6-stage ring; completions are counted on
//     the leader's `full` barrier (the leader posts the expected bytes of both CTAs). The leader's
//     producer is also the scheduler: it takes the tiles from the counter and posts each one, a
//     tile ahead, in a ring of slots in both CTAs (`tnext`), which the other roles read and release
//     (`tfree`);
//   * warp 1 lane 0 of the leader: issues the pair MMAs (M 256, N 256, K 16) into the accumulator
//     (TMEM, 2 x 256 columns in each CTA, double buffered) and commits to both CTAs' `empty` and
//     `tfull` barriers at once (multicast);
//   * warps 2-5 of each CTA: drain its own 128 accumulator rows (SwiGLU or route weight, bf16) and
//     arrive on the leader's `tempty` barrier (8 arrivals: 4 warps x 2 CTAs).
// Every mbarrier wait is bounded; a time-out records MOE_STATUS_WAIT_TIMEOUT and every role runs to
// the final cluster barrier, so neither CTA leaves while its peer may still touch its memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {

namespace g2 {

constexpr int BM = 128;                 // rows per CTA
constexpr int PM = 2 * BM;              // rows per pair tile
constexpr int BN = 256;                 // output columns per pair tile
constexpr int BNH = BN / 2;             // B rows (output columns) staged by each CTA
constexpr int BK = 64;                  // bf16 elements per 128-byte swizzled row
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BYTES = BNH * BK * 2;   // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int TRING = 4;                // schedule slots (tile indices handed from the scheduler to the roles)
constexpr int TREADERS = 10;            // readers of a slot: leader MMA + 4 epilogue warps, follower producer + 4
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;

struct Args {
  const int32_t* offsets;
  const int32_t* slot_expert;
  int E, shared, R, T, K, n_tiles, mode, I, ldo;
  void* out;
  const float* row_weight;
  int* status;
  int* tile_ctr;  // tile counter (zero before the launch), or nullptr: fixed stride
  int vec32;      // the output rows and their column tiles start on 32-byte boundaries
  long long wait_limit;
};

struct Shared {
  uint64_t full[STAGES];    // leader only: both CTAs' copies of a stage have landed
  uint64_t empty[STAGES];   // each CTA: the pair MMAs reading this CTA's stage are done
  uint64_t tfull[2];        // each CTA: accumulator buffer complete
  uint64_t tempty[2];       // leader only: both CTAs drained the accumulator buffer
  uint64_t mma_done;
  uint64_t tnext[TRING];    // each CTA: the slot holds the next tile (the leader's scheduler arrives)
  uint64_t tfree[TRING];    // leader only: every reader of the slot has taken the tile
  int next_tile[TRING];
  uint32_t tmem_slot;
  volatile int abort_flag;
  grp::Table tb;
};

using grp::silu;
using grp::Tile;
using grp::wait_or_abort;

__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                  const __grid_constant__ CUtensorMap tmBs, const __grid_constant__ CUtensorMap tmB64,
                                  const __grid_constant__ CUtensorMap tmBs64, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared s;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int G = args.E + args.shared;

  if (warp == 0) {
    grp::build_table(s.tb, args.offsets, args.E, args.shared, args.R, args.T, PM, lane);
    if (lane == 0) {
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(&s.full[i], 1);
        mbar_init(&s.empty[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.tfull[i], 1);
        mbar_init(&s.tempty[i], 8);
      }
      mbar_init(&s.mma_done, 1);
      for (int i = 0; i < TRING; ++i) {
        mbar_init(&s.tnext[i], 1);
        mbar_init(&s.tfree[i], TREADERS);
      }
      s.abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmBs);
      tma_prefetch_desc(&tmB64);
      tma_prefetch_desc(&tmBs64);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&s.tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before anything signals them
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_slot;
  const int total = s.tb.gtile[G] * args.n_tiles;
  const int kblocks = args.K / BK;
  const uint32_t tfree0 = mapa_shared(smem_u32(&s.tfree[0]), 0);  // the leader's tfree[0]
  // the tile in schedule slot `it` (a reader other than the scheduler): wait for it, take it, release
  // the slot; -1 when the wait gave up
  // The leader's readers wait and arrive at CTA scope (the scheduler is a thread of their own CTA);
  // only the follower's readers need cluster scope.
  auto take_tile = [&](int it) -> int {
    const int slot = it % TRING;
    const uint32_t par = (uint32_t)((it / TRING) & 1);
    const bool got = rank == 0
                         ? wait_or_abort(&s.tnext[slot], par, &s.abort_flag, args.status, args.wait_limit)
                         : wait_or_abort<true>(&s.tnext[slot], par, &s.abort_flag, args.status, args.wait_limit);
    if (!got) return -1;
    const int t = *reinterpret_cast<volatile int*>(&s.next_tile[slot]);
    if (rank == 0)
      mbar_arrive(&s.tfree[slot]);
    else
      mbar_arrive_cluster(tfree0 + (uint32_t)(slot * sizeof(uint64_t)));
    return t;
  };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs)
    const uint32_t full0 = mapa_shared(smem_u32(&s.full[0]), 0);  // the leader's full[0]
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool ok = true;
    const uint32_t peer_next0 = mapa_shared(smem_u32(&s.next_tile[0]), 1);
    const uint32_t peer_tnext0 = mapa_shared(smem_u32(&s.tnext[0]), 1);
    // scheduler (leader): post tile `t` in slot `j` of both CTAs once every reader has released the
    // slot's previous tile (false when that wait gave up); take the tile that follows `t`
    auto post = [&](int j, int t) -> bool {
      const int slot = j % TRING;
      if (!wait_or_abort<true>(&s.tfree[slot], (uint32_t)(((j / TRING) & 1) ^ 1), &s.abort_flag, args.status,
                               args.wait_limit))
        return false;
      st_shared_cluster_u32(peer_next0 + (uint32_t)(slot * sizeof(int)), (uint32_t)t);
      mbar_arrive_cluster(peer_tnext0 + (uint32_t)(slot * sizeof(uint64_t)));
      *reinterpret_cast<volatile int*>(&s.next_tile[slot]) = t;
      mbar_arrive(&s.tnext[slot]);
      return true;
    };
    auto fetch = [&](int t) -> int { return args.tile_ctr ? npairs + atomicAdd(args.tile_ctr, 1) : t + npairs; };
    // The leader posts each tile one whole tile ahead of its copies, so that no reader (the follower's
    // copies above all) waits for it at a tile boundary, and takes the tile after it at the same time
    // (the atomic's latency hides behind a tile's copies).
    int tile = pair, next = 0;
    if (rank == 0) {
      ok = post(0, tile);
      next = tile < total ? fetch(tile) : tile;
    }
    for (int it = 0; ok; ++it) {
      int after = 0;  // leader: the tile after `next`
      if (rank == 0) {
        if (tile >= total) break;
        if (!post(it + 1, next)) break;
        after = next < total ? fetch(next) : next;
      } else {
        tile = take_tile(it);
        if (tile < 0 || tile >= total) break;
      }
      const Tile t = grp::decode(s.tb, G, args.n_tiles, tile, PM);
      const bool half = t.rows <= BM;  // the M = 128 pair tile: 64 rows per CTA
      const bool gu_half = half && args.mode == 0;
      const CUtensorMap* mb = t.g < args.E ? (gu_half ? &tmB64 : &tmB) : (gu_half ? &tmBs64 : &tmBs);
      const int z = t.g < args.E ? (args.slot_expert ? args.slot_expert[t.g] : t.g) : 0;
      const int a_row = t.a_row + (int)rank * (half ? BM / 2 : BM);
      // mode 0: the leader stages the 128 gate rows, the follower the matching up rows (half tiles:
      // each CTA stages 64 gate rows and the 64 matching up rows)
      const int n0 = gu_half ? t.n_tile * BNH + (int)rank * (BNH / 2)
                     : args.mode == 0 ? (int)rank * args.I + t.n_tile * BNH : t.n_tile * BN + (int)rank * BNH;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&s.empty[stage], phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        uint8_t* a = smem + stage * STAGE_BYTES;
        uint8_t* b = a + A_BYTES;
        const uint32_t fb = full0 + (uint32_t)(stage * sizeof(uint64_t));
        if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 2 * STAGE_BYTES);
        tma_load_2d_pair(a, &tmA, fb, kb * BK, a_row);
        if (gu_half) {
          tma_load_3d_pair(b, mb, fb, kb * BK, n0, z);
          tma_load_3d_pair(b + B_BYTES / 2, mb, fb, kb * BK, args.I + n0, z);
        } else {
          tma_load_3d_pair(b, mb, fb, kb * BK, n0, z);
        }
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (rank == 0) {
        tile = next;
        next = after;
      }
    }
    // the leader's last fills of every stage (both CTAs' bytes) must land before either CTA exits;
    // the follower is held by the final cluster barrier until the leader has seen them
    if (rank == 0) {
      const long long first = issued > STAGES ? issued - STAGES : 0;
      for (long long i = first; i < issued; ++i)
        grp::drain_wait(&s.full[i % STAGES], (uint32_t)((i / STAGES) & 1), args.wait_limit);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (leader)
    const uint32_t idesc_full = idesc_bf16(PM, BN), idesc_half = idesc_bf16(PM / 2, BN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      const int tile = take_tile(it);
      if (tile < 0 || tile >= total) break;
      const uint32_t idesc = grp::decode(s.tb, G, args.n_tiles, tile, PM).rows <= BM ? idesc_half : idesc_full;
      if (!wait_or_abort(&s.tempty[acc], acc_phase ^ 1, &s.abort_flag, args.status, args.wait_limit)) break;
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!wait_or_abort(&s.full[stage], phase, &s.abort_flag, args.status, args.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t b = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_f16_pair(d, sw128_kmajor_desc(a + kk * 32), sw128_kmajor_desc(b + kk * 32), idesc, (kb | kk) != 0);
        umma_commit_pair(&s.empty[stage], 0x3);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      umma_commit_pair(&s.tfull[acc], 0x3);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    umma_commit_pair(&s.mma_done, 0x1);
    grp::drain_wait(&s.mma_done, 0, args.wait_limit);
  } else if (warp >= 2) {
    // ---------------- epilogue: this CTA's 128 accumulator rows -> registers -> global
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t tempty0 = mapa_shared(smem_u32(&s.tempty[0]), 0);  // the leader's tempty[0]
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0;; ++it) {
      int tile = 0;
      if (lane == 0) tile = take_tile(it);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (tile < 0 || tile >= total) break;
      const Tile t = grp::decode(s.tb, G, args.n_tiles, tile, PM);
      int ok = 1;
      if (lane == 0) ok = wait_or_abort(&s.tfull[acc], acc_phase, &s.abort_flag, args.status, args.wait_limit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      const bool half = t.rows <= BM;
      // full tile: lane r of this CTA = row 128 rank + r, all 256 columns. Half tile: lanes 0-63 and
      // 64-127 both hold rows 64 rank + (r mod 64), for output columns [0, 128) and [128, 256)
      const int lr = half ? (int)rank * (BM / 2) + (r & 63) : (int)rank * BM + r;  // row within the pair tile
      const int ch = half ? r >> 6 : 0;  // half tiles: which 128 output columns this lane holds
      const bool valid = lr < t.rows;
      const int64_t orow = (int64_t)t.a_row + lr;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (args.mode == 0) {
        // full: gate columns [0, 128), up [128, 256) -> H columns [0, 128) of the tile; half: gate
        // columns [0, 64), up [64, 128) -> H columns [64 ch, 64 ch + 64)
        const int ncol = half ? BNH / 2 : BNH;
        const int up = half ? BNH / 2 : BNH;
        __nv_bfloat16* out =
            reinterpret_cast<__nv_bfloat16*>(args.out) + orow * args.ldo + t.n_tile * BNH + ch * (BNH / 2);
#pragma unroll 1
        for (int c = 0; c < ncol; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c, g);
          tmem_ld32(taddr + up + c, u);
          tmem_ld_wait_regs(g);
          tmem_ld_wait_regs(u);
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
            const float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
            p[i] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            if (args.vec32) {
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
        const int ncol = half ? BN / 2 : BN;
        __nv_bfloat16* out =
            reinterpret_cast<__nv_bfloat16*>(args.out) + orow * args.ldo + t.n_tile * BN + ch * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < ncol; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_ld_wait_regs(v);
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * w, __uint_as_float(v[2 * i + 1]) * w);
          if (valid) {
            if (args.vec32) {
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
      if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)(acc * sizeof(uint64_t)));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  // Neither CTA may leave (or free TMEM) while the pair MMAs, the peer's copies or the peer's
  // arrivals can still touch it.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace g2

cudaError_t launch_grouped_gemm_bf16_pair(const GroupedGemmDesc& d, cudaStream_t stream, std::string* err) {
  cudaError_t e = tma_encoder_ready();
  if (e != cudaSuccess) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(g2::THREADS);
  cfg.dynamicSmemBytes = g2::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the shared-memory opt-in and the resident-cluster count are per device
  static PerDevice<int> pairs_table;
  int max_pairs = 0;
  e = per_device<int>(
      pairs_table,
      [&cfg](int& v) {
        cudaError_t r = cudaFuncSetAttribute(g2::grouped_gemm_bf16_pair_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, g2::SMEM_BYTES);
        if (r != cudaSuccess) return r;
        // as many pairs as can be resident at once (SMs of a GPC pair up; an odd one stays out)
        cudaLaunchConfig_t probe = cfg;
        probe.gridDim = dim3(2 * (num_sms() / 2));
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, g2::grouped_gemm_bf16_pair_kernel, &probe);
        if (r != cudaSuccess) return r;
        if (n <= 0) return cudaErrorInvalidConfiguration;
        v = n < num_sms() / 2 ? n : num_sms() / 2;
        return cudaSuccess;
      },
      &max_pairs);
  if (e != cudaSuccess) {
    *err = "cudaFuncSetAttribute / cudaOccupancyMaxActiveClusters failed for the CTA-pair grouped GEMM";
    return e;
  }
  CUtensorMap tA, tB, tBs, tB64, tBs64;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t G = d.n_experts > 0 ? d.n_experts : d.E;
  bool ok = tma_encode_2d(&tA, d.A, BF, 2, d.a_rows, d.K, g2::BM) &&
            tma_encode_3d(&tB, d.B, BF, 2, G, d.b_rows, d.K, g2::BNH) &&
            tma_encode_3d(&tBs, d.Bs ? d.Bs : d.B, BF, 2, 1, d.b_rows, d.K, g2::BNH) &&
            tma_encode_3d(&tB64, d.B, BF, 2, G, d.b_rows, d.K, g2::BNH / 2) &&
            tma_encode_3d(&tBs64, d.Bs ? d.Bs : d.B, BF, 2, 1, d.b_rows, d.K, g2::BNH / 2);
  if (!ok) {
    *err = "cuTensorMapEncodeTiled rejected a grouped-GEMM operand";
    return cudaErrorInvalidValue;
  }
  g2::Args a;
  a.offsets = d.offsets;
  a.slot_expert = d.slot_expert;
  a.E = d.E;
  a.shared = d.Bs != nullptr;
  a.R = d.R;
  a.T = d.T;
  a.K = d.K;
  a.mode = d.mode;
  a.I = d.I;
  a.n_tiles = d.mode == 0 ? d.I / g2::BNH : (int)cdiv(d.N, g2::BN);
  a.ldo = d.ldo;
  a.out = d.out;
  a.row_weight = d.row_weight;
  a.status = d.status;
  a.tile_ctr = d.tile_ctr;
  a.vec32 = (reinterpret_cast<uintptr_t>(d.out) & 31) == 0 && ((int64_t)d.ldo * 2) % 32 == 0;
  a.wait_limit = 4000000000LL;  // about two seconds of SM clock
  cfg.gridDim = dim3(2 * max_pairs);
  e = cudaLaunchKernelEx(&cfg, g2::grouped_gemm_bf16_pair_kernel, tA, tB, tBs, tB64, tBs64, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
