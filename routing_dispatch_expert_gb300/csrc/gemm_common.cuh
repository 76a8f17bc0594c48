// Pieces shared by the grouped-GEMM kernels (bf16 and FP8): the per-group tile table built from the
// device-side expert offsets, the tile decoder of the persistent schedule, the bounded mbarrier wait,
// and the host-side TMA descriptor encoders.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace grp {

constexpr int MAX_GROUPS = 1025;  // E <= 1024 routed experts + the shared expert

// gtile[g]: exclusive prefix of 128-row tiles over groups; grow[g]: first row of group g; gend:
// one past the last row of the last routed group (offsets[E]; with a capacity limit it can lie below
// R, the shared expert's first row). Groups: the E routed experts (rows [offsets[e], offsets[e+1]))
// and, with a shared expert, group E = rows [R, R + T). offsets == nullptr means one group of rows
// [0, T).
struct Table {
  int gtile[MAX_GROUPS + 1];
  int grow[MAX_GROUPS + 1];
  int n_routed;  // groups whose rows come from offsets (E, or 0 when offsets == nullptr)
  int gend;
};

struct Tile {
  int g, m_tile, n_tile, a_row, rows;
};

// Called by one full warp.
__device__ __forceinline__ void build_table(Table& tb, const int32_t* offsets, int E, int shared, int R, int T,
                                            int BM, int lane) {
  const int G = E + shared;
  int carry = 0;
  for (int base = 0; base < G; base += 32) {
    const int g = base + lane;
    int row0 = 0, m = 0;
    if (g < G) {
      if (offsets == nullptr) {
        row0 = 0;
        m = T;
      } else if (g < E) {
        row0 = offsets[g];
        m = offsets[g + 1] - row0;
      } else {
        row0 = R;
        m = T;
      }
    }
    const int mt = (m + BM - 1) / BM;
    int incl = mt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (g < G) {
      tb.gtile[g] = carry + incl - mt;
      tb.grow[g] = row0;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    tb.gtile[G] = carry;
    tb.grow[G] = offsets == nullptr ? T : (shared ? R + T : offsets[E]);
    tb.n_routed = offsets == nullptr ? 0 : E;
    tb.gend = offsets == nullptr ? T : offsets[E];
  }
}

// Tile order: group-major; inside a group, bands of up to kBand row tiles, and inside a band the
// output-column tile, then the row tile (so the CTAs running together share one weight tile through
// L2, and a group with many rows -- the shared expert over a whole batch, a hot expert -- streams its
// activation rows from DRAM once per band instead of once per column tile). A group of at most kBand
// row tiles is one band. n_inner makes the column tile the innermost index (the router: the
// activation rows are the large operand).
constexpr int kBand = 8;
__device__ __forceinline__ Tile decode(const Table& tb, int G, int n_tiles, int tile, int BM, bool n_inner = false) {
  const int q = tile / n_tiles;
  int lo = 0, hi = G - 1;  // last g with gtile[g] <= q
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb.gtile[mid] <= q)
      lo = mid;
    else
      hi = mid - 1;
  }
  Tile t;
  t.g = lo;
  const int local = tile - tb.gtile[lo] * n_tiles;
  const int mtc = tb.gtile[lo + 1] - tb.gtile[lo];
  if (n_inner) {
    t.m_tile = local / n_tiles;
    t.n_tile = local - t.m_tile * n_tiles;
  } else {
    const int band = local / (kBand * n_tiles);
    const int rem = local - band * kBand * n_tiles;
    const int bw = min(kBand, mtc - band * kBand);  // row tiles in this band
    t.n_tile = rem / bw;
    t.m_tile = band * kBand + (rem - t.n_tile * bw);
  }
  t.a_row = tb.grow[lo] + t.m_tile * BM;
  const int end = lo + 1 == tb.n_routed ? tb.gend : tb.grow[lo + 1];
  t.rows = min(BM, end - t.a_row);
  return t;
}

constexpr uint32_t kWaitSleepNs = 20000;  // one suspension of a waiting thread: at most 20 us

// Bounded wait on an mbarrier phase. Gives up when another role of the CTA has aborted, or after
// `limit` SM clocks (then it raises the CTA's abort flag and records MOE_STATUS_WAIT_TIMEOUT).
// With kCluster the wait acquires at cluster scope (a phase completed from the other CTA of a pair).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                              long long limit) {
  auto poll = [&]() {
    return kCluster ? mbar_try_wait_sleep_cluster(bar, parity, kWaitSleepNs)
                    : mbar_try_wait_sleep(bar, parity, kWaitSleepNs);
  };
  if (!kCluster && mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!poll()) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(status, MOE_STATUS_WAIT_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Bounded drain used on the way out (normal or aborted): wait for a phase, give up after `limit`.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kWaitSleepNs) && clock64() - t0 < limit) {
  }
}

// SiLU in fp32 with the fast reciprocal (a few ulp, far below the bf16 / e4m3 rounding of H that
// follows): the IEEE division's longer instruction sequence made the gate/up epilogue of a small layer
// latency-bound.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

}  // namespace grp

// host: TMA descriptors (gemm.cu)
cudaError_t tma_encoder_ready();
// [rows, K] row-major, `elem`-byte elements; box = box_rows x 128 bytes of K, 128-byte swizzle.
bool tma_encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int64_t rows, int64_t K,
                   int box_rows);
// [G, rows, K] row-major stack; box = 1 x box_rows x 128 bytes of K, 128-byte swizzle.
// [G, rows, K] bytes, no swizzle, box = box_k bytes x box_rows rows (box_k * elem a multiple of 16).
bool tma_encode_3d_plain(CUtensorMap* m, const void* base, int64_t G, int64_t rows, int64_t K, int box_k, int box_rows);
bool tma_encode_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int64_t G, int64_t rows,
                   int64_t K, int box_rows);

}  // namespace moe
