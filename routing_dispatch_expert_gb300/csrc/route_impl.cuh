// Device code of step 1 (router GEMM for small E, top-k selection) shared by the standalone kernels
// (route.cu) and the fused small-batch route-and-dispatch kernel (fused.cu). Both call the same
// functions, so a logit, a selection and a route weight are bit-for-bit the same on either path.
#pragma once

#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------------------------------------------
// router GEMM for small E (E < 128, or E not a multiple of 32): logits[T, E] = x[T, h] . w_r[E, h]^T
// on the CUDA cores in fp32. The output is only E columns wide, so the work is split over tokens and K
// instead of output tiles: a CTA of 8 warps takes EMAX experts (blockIdx.y selects the expert block
// when E > 64) and `groups` x TPW tokens. The warps form `groups` groups of kw = 8 / groups warps
// (kw = 8 when h has at least 8 chunks of 256, else the largest power of two not above the chunk
// count, so that no warp idles on a short row); warp j of a group takes that group's TPW tokens and
// the 256-element K chunks j, j + kw, ... (each lane 8 consecutive elements of a chunk: one 16-byte
// load of x per token, two 16-byte loads of each expert's weight row, L1-resident); lanes are summed
// by a butterfly, the kw warps' partial sums in warp order through shared memory (the same order on
// every run).
// ------------------------------------------------------------------------------------------
namespace rg {
constexpr int WARPS = 8, THREADS = 32 * WARPS;

// Named barrier over the `n` threads of one (virtual) CTA: barrier 0 with n = blockDim.x is
// __syncthreads; a fused kernel running two 256-thread units side by side gives each its own id.
__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// One work unit of the small-E router: the CTA (blockIdx.x, blockIdx.y) = (bx, by) of the standalone
// launch, run by THREADS threads whose index in the unit is tid, with shared partial sums `part` and
// named barrier `bar_id`. The arithmetic of every logit depends only on (token, expert), h and kw, not
// on which CTA runs the unit.
template <int EMAX, int TPW>
__device__ __forceinline__ void router_unit(const __nv_bfloat16* __restrict__ x, const float* __restrict__ w,
                                            float* __restrict__ out, int T, int h, int E, int kw, int bx, int by,
                                            int tid, float (*part)[TPW][EMAX], int bar_id) {
  const int warp = tid >> 5, lane = tid & 31;
  const int groups = WARPS / kw;
  const int grp = warp / kw, kj = warp - grp * kw;
  const int t0 = (bx * groups + grp) * TPW;
  const int e0 = by * EMAX;
  const int ne = min(EMAX, E - e0);  // experts of this block
  float acc[TPW][EMAX];
#pragma unroll
  for (int t = 0; t < TPW; ++t)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[t][e] = 0.f;
  const int chunks = h / 256;
  for (int c = kj; c < chunks; c += kw) {
    const int k = c * 256 + lane * 8;
    float xv[TPW][8];
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
      const uint4 v = t0 + t < T ? *reinterpret_cast<const uint4*>(x + (int64_t)(t0 + t) * h + k)
                                 : make_uint4(0, 0, 0, 0);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[t][2 * i] = bf16_lo(u[i]);
        xv[t][2 * i + 1] = bf16_hi(u[i]);
      }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e < ne) {
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(w + (int64_t)(e0 + e) * h + k));
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + (int64_t)(e0 + e) * h + k + 4));
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[t][e] = fmaf(xv[t][i], wv[i], acc[t][e]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TPW; ++t)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      float v = acc[t][e];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) part[warp][t][e] = v;
    }
  bar_sync(bar_id, THREADS);
  for (int i = tid; i < groups * TPW * EMAX; i += THREADS) {
    const int g = i / (TPW * EMAX), t = (i / EMAX) % TPW, e = i % EMAX;
    const int tok = (bx * groups + g) * TPW + t;
    if (e < ne && tok < T) {
      float v = part[g * kw][t][e];
      for (int q = 1; q < kw; ++q) v += part[g * kw + q][t][e];
      out[(int64_t)tok * E + e0 + e] = v;
    }
  }
  bar_sync(bar_id, THREADS);  // part[] is free for the unit's next use
}
}  // namespace rg

// ------------------------------------------------------------------------------------------
// top-k: one warp per token; lane l holds experts [l * EPL, l * EPL + EPL).
// ------------------------------------------------------------------------------------------
namespace tk {

// Keys as order-preserving unsigned integers: a > b as floats <=> ord(a) > ord(b) (-0 is taken as +0;
// NaN keys are replaced by -inf before). Every key maps above 0, so 0 marks "no candidate". A warp
// argmax is then one redux.sync max plus a ballot: the lowest lane holding the maximum, and inside a
// lane the lowest slot, is the lowest expert index among equal keys.
__device__ __forceinline__ uint32_t ord(float f) {
  const uint32_t b = __float_as_uint(__fadd_rn(f, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord(uint32_t u) {
  if (u == 0) return -INFINITY;
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// The selection key of the sigmoid layers is fp32(sigmoid(l)) + bias with the sigmoid evaluated in
// fp64 and rounded once. The fast pass evaluates it in fp32 (expf, at most 2 ulp, then two correctly
// rounded operations): |key_fast - key| < 4e-7. A decision taken on the fast keys is the decision on
// the exact keys whenever every deciding gap exceeds twice the error (a group score, a sum of two
// keys, four times it); the thresholds below leave a further margin. A token with a smaller gap is
// selected again on the exact fp64 keys.
constexpr float kKeyGap = 1e-6f;    // between two expert keys
constexpr float kGroupGap = 2e-6f;  // between two group scores (sums of two keys)

__device__ __forceinline__ float sigmoid_exact(float l) { return __double2float_rn(1.0 / (1.0 + exp(-(double)l))); }
__device__ __forceinline__ float sigmoid_fast(float l) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l))); }

// Per-lane constants of the expert slots: group index and validity, the same for every token.
template <int EPL>
struct Slots {
  int grp[EPL];
  bool valid[EPL];
  float bias[EPL];
  int lpg;  // lanes per group when every group is a whole number of lanes (else 0)
};

// Group stage and expert stage on the keys of one token. Returns in sel_e / sel_l (lanes < k) the
// chosen experts in descending key order and their logits. *clear is false when a deciding gap is
// below the thresholds (only tracked when track_gaps); *groups_clear is false when the group stage's
// gap is, and *cut is the best key left out of the selection (the (k+1)-th, when track_gaps).
template <int EPL>
__device__ __forceinline__ void select_experts(const TopkDesc& d, const Slots<EPL>& sl, const float (&key)[EPL],
                                               const float (&lv)[EPL], int lane, bool track_gaps, int& sel_e,
                                               float& sel_l, bool& clear, bool& groups_clear, float& cut) {
  clear = true;
  groups_clear = true;
  cut = -INFINITY;
  uint32_t kept = 0xffffffffu;
  if (d.n_group > 1) {
    // the score of group g (sum of its two best keys) ends in every lane of the group (lane-aligned
    // groups) or in lane g
    float my_gscore = -INFINITY;
    int my_group = -1;
    if (sl.lpg) {
      float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const float v = key[i];
        if (v > t1) {
          t2 = t1;
          t1 = v;
        } else if (v > t2) {
          t2 = v;
        }
      }
      for (int o = 1; o < sl.lpg; o <<= 1) {
        const float o1 = __shfl_xor_sync(0xffffffffu, t1, o);
        const float o2 = __shfl_xor_sync(0xffffffffu, t2, o);
        const float n1 = fmaxf(t1, o1);
        t2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
        t1 = n1;
      }
      my_gscore = EPL * sl.lpg >= 2 ? __fadd_rn(t1, t2) : t1;
      my_group = sl.grp[0];
    } else {
      const int gs = d.E / d.n_group;
      for (int g = 0; g < d.n_group; ++g) {
        float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          if (sl.valid[i] && sl.grp[i] == g) {
            const float v = key[i];
            if (v > t1) {
              t2 = t1;
              t1 = v;
            } else if (v > t2) {
              t2 = v;
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float o1 = __shfl_xor_sync(0xffffffffu, t1, o);
          const float o2 = __shfl_xor_sync(0xffffffffu, t2, o);
          const float n1 = fmaxf(t1, o1);
          t2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
          t1 = n1;
        }
        const float sc = gs >= 2 ? __fadd_rn(t1, t2) : t1;
        if (lane == g) my_gscore = sc;
      }
      my_group = lane < d.n_group ? lane : -1;
    }
    // the topk_group best groups, ties to the lower group index (lanes are in group order)
    const uint32_t gu = my_group >= 0 ? ord(my_gscore) : 0u;
    kept = 0;
    for (int r = 0; r < d.topk_group; ++r) {
      const bool cand = my_group >= 0 && !((kept >> my_group) & 1u);
      const uint32_t u = cand ? gu : 0u;
      const uint32_t m = __reduce_max_sync(0xffffffffu, u);
      const uint32_t b = __ballot_sync(0xffffffffu, cand && u == m);
      const int wl = __ffs(b) - 1;
      kept |= 1u << __shfl_sync(0xffffffffu, my_group, wl);
    }
    if (track_gaps && d.topk_group < d.n_group) {
      const bool in = my_group >= 0 && ((kept >> my_group) & 1u);
      const bool out = my_group >= 0 && !((kept >> my_group) & 1u);
      const float kept_min = unord(__reduce_min_sync(0xffffffffu, in ? gu : 0xffffffffu));
      const float rest_max = unord(__reduce_max_sync(0xffffffffu, out ? gu : 0u));
      if (!(kept_min - rest_max > kGroupGap)) clear = groups_clear = false;
    }
  }
  uint32_t uk[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) uk[i] = (sl.valid[i] && ((kept >> sl.grp[i]) & 1u)) ? ord(key[i]) : 0u;
  sel_e = 0;
  sel_l = 0.f;
  float prev = 0.f;
  const int rounds = track_gaps ? d.k + 1 : d.k;  // one more round finds the best key left out
  for (int j = 0; j < rounds; ++j) {
    uint32_t lb = 0;
    int li = 0;
    float ll = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (uk[i] > lb) {
        lb = uk[i];
        li = i;
        ll = lv[i];
      }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, lb);
    const float bv = unord(m);
    if (track_gaps && j > 0 && !(prev - bv > kKeyGap)) clear = false;
    prev = bv;
    if (j == d.k) {  // the (k+1)-th key only checks the gap
      cut = bv;
      break;
    }
    const uint32_t b = __ballot_sync(0xffffffffu, m != 0 && lb == m);
    const int wl = b ? __ffs(b) - 1 : 0;
    const int wi = __shfl_sync(0xffffffffu, li, wl);
    const float wlv = __shfl_sync(0xffffffffu, ll, wl);
    if (lane == wl && b) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == li) uk[i] = 0u;
    }
    if (lane == j) {
      sel_e = b ? wl * EPL + wi : 0x7fffffff;
      sel_l = wlv;
    }
  }
}

// Per-lane slot constants of the layer (the same for every token).
template <int EPL>
__device__ __forceinline__ Slots<EPL> make_slots(const TopkDesc& d, int lane) {
  const bool sigmoid = d.score == MOE_SCORE_SIGMOID;
  const int gs = d.E / d.n_group;
  Slots<EPL> sl;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane * EPL + i;
    sl.valid[i] = e < d.E;
    sl.grp[i] = sl.valid[i] ? e / gs : 0;
    sl.bias[i] = (sigmoid && d.bias && sl.valid[i]) ? d.bias[e] : 0.f;
  }
  // groups made of whole lanes: every slot of a lane in one group, a power-of-two lane count per group
  const int lpg_c = gs / EPL;
  sl.lpg = (d.E == 32 * EPL && gs % EPL == 0 && lpg_c >= 1 && (lpg_c & (lpg_c - 1)) == 0) ? lpg_c : 0;
  return sl;
}

// Selection and route weights of token t by one warp: topk_idx[t, :] and topk_w[t, :]. The result
// depends only on the token's logits (and the layer's bias and shape), not on which warp runs it.
template <int EPL>
__device__ __forceinline__ void topk_token(const TopkDesc& d, const Slots<EPL>& sl, int lane, int t) {
  const bool sigmoid = d.score == MOE_SCORE_SIGMOID;
  const bool vec = EPL % 4 == 0 && d.E == 32 * EPL && (reinterpret_cast<uintptr_t>(d.logits) & 15) == 0;
  const float* lrow = d.logits + (int64_t)t * d.E;
  float key[EPL], lv[EPL];
  if (d.partials) {
    // the router's split-K partial sums, added in split order and stored as the logits; the loads of
    // one split for all of a lane's experts (and, unrolled, of the next splits) are independent, so
    // they are in flight together
    const int64_t n = (int64_t)d.T * d.E;
    const float* p = d.partials + (int64_t)t * d.E + lane * EPL;
#pragma unroll
    for (int i = 0; i < EPL; ++i) lv[i] = sl.valid[i] ? p[i] : 0.f;
#pragma unroll 4
    for (int q = 1; q < d.splits; ++q) {
      float vq[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) vq[i] = sl.valid[i] ? p[(int64_t)q * n + i] : 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) lv[i] = __fadd_rn(lv[i], vq[i]);
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (sl.valid[i]) const_cast<float*>(d.logits)[(int64_t)t * d.E + lane * EPL + i] = lv[i];
  } else if (vec) {
#pragma unroll
    for (int i = 0; i < EPL; i += 4) {
      const float4 q = *reinterpret_cast<const float4*>(lrow + lane * EPL + i);
      lv[i] = q.x;
      lv[i + 1] = q.y;
      lv[i + 2] = q.z;
      lv[i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) lv[i] = sl.valid[i] ? lrow[lane * EPL + i] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    float kv = sigmoid ? __fadd_rn(sigmoid_fast(lv[i]), sl.bias[i]) : lv[i];
    if (kv != kv) kv = -INFINITY;  // NaN never wins
    key[i] = sl.valid[i] ? kv : -INFINITY;
  }
  int sel_e;
  float sel_l;
  bool clear, groups_clear;
  float cut;
  select_experts<EPL>(d, sl, key, lv, lane, sigmoid, sel_e, sel_l, clear, groups_clear, cut);
  if (sigmoid && !clear) {
    // A near tie: decide on the exact keys (fp64 sigmoid, slow on this part's fp64 pipe). When the
    // group stage is settled (its gap exceeds twice the fast keys' error, so the same groups are kept
    // on exact keys), only an expert whose fast key lies within kCutWindow of the best key left out
    // can enter the selection or change its order: every other key stays more than kCutWindow - 2 x
    // 4e-7 away from each re-evaluated one, so its order against them is the same on exact keys.
    // Those experts keep their fast keys; slot positions no lane needs are skipped. With a group near
    // tie every key is re-evaluated.
    constexpr float kCutWindow = 2e-6f;
    const float lo = groups_clear ? cut - kCutWindow : -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const bool need = sl.valid[i] && key[i] >= lo;
      if (__any_sync(0xffffffffu, need) && need) {
        float kv = __fadd_rn(sigmoid_exact(lv[i]), sl.bias[i]);
        if (kv != kv) kv = -INFINITY;
        key[i] = kv;
      }
    }
    select_experts<EPL>(d, sl, key, lv, lane, false, sel_e, sel_l, clear, groups_clear, cut);
  }

  // route weights. They enter the combine, not a selection, so they are formed in fp32 (this part's
  // fp64 pipe runs at a small fraction of the fp32 rate, and a few fp64 operations per token made the
  // whole top-k fp64-bound), with error bounds well inside the weights' tolerance:
  if (sigmoid) {
    // w_j = s_j * (scale / sum s): s in fp32 (relative error below 4e-7); the k scores summed in slot
    // order by every lane (the same sum on every lane, k - 1 roundings)
    const float sj = lane < d.k ? sigmoid_fast(sel_l) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < d.k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, sj, j));
    const float scale = d.renorm ? __fdiv_rn(d.routed_scale, sum) : d.routed_scale;
    if (lane < d.k) {
      d.topk_idx[(int64_t)t * d.k + lane] = sel_e;
      d.topk_w[(int64_t)t * d.k + lane] = __fmul_rn(sj, scale);
    }
    return;
  }
  // softmax: e_i = exp(l_i - lmax), with the rounding error of the subtraction carried into the
  // exponential (l - lmax = dh + dl exactly, e = expf(dh) * (1 + dl)), so e has expf's 2 ulp plus a
  // few roundings. Renormalised, w_j = e_j / sum_sel e (the normaliser over all experts cancels; k - 1
  // roundings in slot order); otherwise w_j = e_j / z with z = sum over all experts, per lane in slot
  // order and then a butterfly (every lane ends with the same z; EPL + 4 roundings); above 256
  // experts z is summed in fp64 to keep its error small.
  float lmax = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (sl.valid[i]) lmax = fmaxf(lmax, lv[i]);
  lmax = warp_max(lmax);
  auto expd = [lmax](float l) {
    const float b = -lmax;
    const float dh = __fadd_rn(l, b);
    const float e = expf(dh);
    if (!(e > 0.f) || isinf(e)) return e;  // 0, inf or NaN: nothing to correct
    // TwoSum (Knuth): dh + dl == l + b exactly
    const float bb = __fsub_rn(dh, l);
    const float dl = __fadd_rn(__fsub_rn(l, __fsub_rn(dh, bb)), __fsub_rn(b, bb));
    return __fmaf_rn(e, dl, e);  // exp(dh + dl) to first order in dl (|dl| <= 2^-24 |dh|)
  };
  const float e_sel = lane < d.k ? expd(sel_l) : 0.f;
  float w;
  if (d.renorm) {
    float sum = 0.f;
    for (int j = 0; j < d.k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, e_sel, j));
    w = __fdiv_rn(e_sel, sum);
  } else if (EPL <= 8) {
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (sl.valid[i]) z = __fadd_rn(z, expd(lv[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, o));
    w = __fdiv_rn(e_sel, z);
  } else {
    double z = 0.0;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (sl.valid[i]) z += (double)expd(lv[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    w = (float)((double)e_sel / z);
  }
  if (lane < d.k) {
    d.topk_idx[(int64_t)t * d.k + lane] = sel_e;
    d.topk_w[(int64_t)t * d.k + lane] = __fmul_rn(w, d.routed_scale);
  }
}

}  // namespace tk

}  // namespace moe
