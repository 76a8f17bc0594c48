/*
 * CPU oracle of the single-GPU MoE layer: route -> dispatch -> SwiGLU experts -> combine.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the bench's CPU-baseline /
 * reference arm load this library. The product (the CUDA library and its Python binding)
 * never calls it, and it shares no code, header, table or helper with the product.
 *
 * Style: plain scalar loops, fp64 arithmetic, no blocking, fusion or reordering beyond what
 * the definition states. Every function names the passage it follows.
 *
 * Sources (web pages on expert-parallel MoE inference):
 *   [ULTRA]  Ultralytics glossary "Expert Parallelism", section "How tokens move across GPUs"
 *            (the four steps: route, dispatch, compute, combine) and "Load balancing and
 *            capacity" (per-expert bias that only affects which experts are selected).
 *   [INFRA]  Inference guide 6.4 "Data parallelism and expert parallelism": section 2.1 (an
 *            expert is three matrices gate, up, down), section 3.1 (data flow of one MoE
 *            layer: each token's hidden state is copied k times, results are summed with the
 *            route weights), section 7 (the shared expert acts like a routed expert every
 *            token must pick).
 *   [PPLX]   Perplexity blog "Lower latency and higher throughput with multi-node DeepSeek
 *            deployment": "MoE Router" (Mixtral routing is DeepSeek routing with top-k-group =
 *            all groups; dense dispatch needs per-expert aggregation), "Quantization" (FP8
 *            block scheme: 1x128 activation vectors scaled at run time, 128x128 weight tiles;
 *            SiLU output block-quantised with a 128-element amax).
 *   [TRTLLM] NVIDIA TensorRT-LLM "DeepSeek R1 throughput on Blackwell", "MoE layer
 *            optimizations / Top-K kernel fusion" (two-stage selection: groups first, then the
 *            top-8 experts inside them, plus a bias and a scaling factor).
 *
 * Readings where the pages leave a step open (each is also listed in the design notes):
 *   R1 group score = sum of the two largest biased scores in the group;
 *   R2 ties break to the lower expert index, and among groups to the lower group index;
 *   R3 sigmoid computed in fp64 and rounded once to fp32; key = fp32(s) + bias in fp32;
 *   R4 softmax configurations select on the raw logits (softmax is monotone); weights are the
 *      full-softmax probabilities, optionally renormalised over the selected experts;
 *   R6 the scaling factor multiplies the (renormalised) routed weights;
 *   R7 the shared expert is added with weight 1;
 *   R8 storage points: the SwiGLU product is stored in bf16 (FP8 1x128 in the FP8 layer);
 *   R10 FP8 scale = amax / 448 in fp32, all-zero block -> scale 1, round-to-nearest-even with
 *       saturation to +-448.
 *   R19 FP4 expert weights ([TRTLLM] "Precision strategy": the MoE weights of the Blackwell
 *       deployment are FP4, halving the weight bytes a memory-bound decode step streams) use
 *       the NVFP4 layout: e2m1 elements, one e4m3 scale per 16 consecutive elements of a row,
 *       one fp32 scale per weight matrix; activations stay bf16 (weight-only FP4);
 *   R20 NVFP4 quantisation: global g = amax(W) / (6 * 448) in fp32 (all-zero matrix -> 1);
 *       block code s = e4m3(fp32(amax_block / fp32(6 * g))); element code e2m1(fp32(w /
 *       fp32(s * g))), nearest with ties to the even code, saturating at +-6; a block whose
 *       scale code is zero has all element codes zero. Value = e2m1 * s * g.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------------------------
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits; same range as fp32.
 * ---------------------------------------------------------------------------------------- */

ORC_API double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even, directly from the double (no
 * intermediate float rounding). Written from the format: 8 significant bits for normal
 * numbers, a fixed quantum of 2^-133 below 2^-126. */
ORC_API uint16_t orc_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
  double a = fabs(v);
  double q; /* quantum of the bf16 grid around a */
  if (a < ldexp(1.0, -126)) {
    q = ldexp(1.0, -133);
  } else {
    int e;
    frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1 */
    q = ldexp(1.0, e - 8);
  }
  double r = nearbyint(a / q) * q; /* default rounding mode: to nearest, ties to even */
  if (r >= ldexp(1.0, 128)) r = INFINITY;
  float f = (float)r; /* exact: r is on the bf16 grid */
  if (v < 0) f = -f;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------------------------
 * FP8 e4m3 (OCP 8-bit floating point): 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent field 0 is subnormal; no infinities; S.1111.111 is NaN; max finite 448.
 * ---------------------------------------------------------------------------------------- */

ORC_API double orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, E = (c >> 3) & 15, M = c & 7;
  double v;
  if (E == 15 && M == 7) return NAN;
  if (E == 0)
    v = ldexp((double)M / 8.0, 1 - 7);
  else
    v = ldexp(1.0 + (double)M / 8.0, E - 7);
  return s ? -v : v;
}

/* Nearest e4m3 value to f, ties to the even code (mantissa LSB 0), magnitudes above 448
 * saturate to 448. Positive codes 0x00..0x7E are monotone in value, so a binary search for
 * the last code whose value is <= |f| and a comparison with the next code is enough. */
ORC_API uint8_t orc_e4m3_encode(float f) {
  if (isnan(f)) return 0x7F;
  uint8_t sign = signbit(f) ? 0x80 : 0x00;
  double a = fabs((double)f);
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) or hi is 448 */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (orc_e4m3_decode((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  double vlo = orc_e4m3_decode((uint8_t)lo), vhi = orc_e4m3_decode((uint8_t)hi);
  int code;
  if (a - vlo < vhi - a)
    code = lo;
  else if (a - vlo > vhi - a)
    code = hi;
  else
    code = (lo & 1) ? hi : lo;
  return sign | (uint8_t)code;
}

/* Block quantisation rule (reading R10): scale = amax / 448 rounded to fp32 (1 if the block
 * is all zero); code = e4m3(fp32(v / scale)). The quotient is rounded to fp32 before the
 * e4m3 rounding, i.e. the code is decided in fp32. */
static float orc_fp8_scale(double amax) {
  if (amax == 0.0) return 1.0f;
  return (float)(amax / 448.0);
}

/* 1x128 activation quantisation ([PPLX] "Quantization": activation scales are computed at
 * run time per 128-element vector along K). v: [m, n] row-major doubles; n % 128 == 0.
 * q: [m, n] codes; s: [m, n/128] fp32 scales. */
ORC_API void orc_quant_1x128(const double* v, int64_t m, int64_t n, uint8_t* q, float* s) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < m; ++r)
    for (int64_t b = 0; b < n / 128; ++b) {
      const double* blk = v + r * n + b * 128;
      double amax = 0.0;
      for (int i = 0; i < 128; ++i)
        if (fabs(blk[i]) > amax) amax = fabs(blk[i]);
      float sc = orc_fp8_scale(amax);
      s[r * (n / 128) + b] = sc;
      for (int i = 0; i < 128; ++i) q[r * n + b * 128 + i] = orc_e4m3_encode((float)(blk[i] / (double)sc));
    }
}

/* 128x128 static weight quantisation ([PPLX] "Quantization": weights scaled per 128x128
 * tile). w: [rows, cols] bf16; rows % 128 == 0, cols % 128 == 0. q: [rows, cols] codes;
 * s: [rows/128, cols/128] fp32 scales. */
ORC_API void orc_quant_weight_128x128(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* q, float* s) {
#pragma omp parallel for schedule(static)
  for (int64_t br = 0; br < rows / 128; ++br)
    for (int64_t bc = 0; bc < cols / 128; ++bc) {
      double amax = 0.0;
      for (int64_t i = 0; i < 128; ++i)
        for (int64_t j = 0; j < 128; ++j) {
          double a = fabs(orc_bf16_to_double(w[(br * 128 + i) * cols + bc * 128 + j]));
          if (a > amax) amax = a;
        }
      float sc = orc_fp8_scale(amax);
      s[br * (cols / 128) + bc] = sc;
      for (int64_t i = 0; i < 128; ++i)
        for (int64_t j = 0; j < 128; ++j) {
          int64_t o = (br * 128 + i) * cols + bc * 128 + j;
          q[o] = orc_e4m3_encode((float)(orc_bf16_to_double(w[o]) / (double)sc));
        }
    }
}

/* ------------------------------------------------------------------------------------------
 * FP4 e2m1 (OCP Microscaling formats, the element type of NVFP4; reading R19): 1 sign, 2
 * exponent bits with bias 1, 1 mantissa bit; exponent field 0 is subnormal; no infinities or
 * NaN. Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. A code is the low nibble of a byte.
 * ---------------------------------------------------------------------------------------- */
ORC_API double orc_e2m1_decode(uint8_t c) {
  int s = (c >> 3) & 1, E = (c >> 1) & 3, M = c & 1;
  double v = E == 0 ? 0.5 * M : ldexp(1.0 + 0.5 * M, E - 1);
  return s ? -v : v;
}

/* Nearest e2m1 value to f, ties to the even code (mantissa bit 0), magnitudes above 6 saturate
 * to 6; the format has no NaN, and NaN maps to +6 like an overflow. Positive codes 0..7 are
 * monotone in value. */
ORC_API uint8_t orc_e2m1_encode(float f) {
  if (isnan(f)) return 0x7;
  uint8_t sign = signbit(f) ? 0x8 : 0x0;
  double a = fabs((double)f);
  if (a >= 6.0) return sign | 0x7;
  int lo = 0;
  while (lo < 7 && orc_e2m1_decode((uint8_t)(lo + 1)) <= a) ++lo;
  int code = lo;
  if (lo < 7) {
    double vlo = orc_e2m1_decode((uint8_t)lo), vhi = orc_e2m1_decode((uint8_t)(lo + 1));
    if (a - vlo > vhi - a || (a - vlo == vhi - a && (lo & 1))) code = lo + 1;
  }
  return sign | (uint8_t)code;
}

/* NVFP4 quantisation of one weight matrix (readings R19, R20). w: [rows, cols] bf16 with
 * cols % 16 == 0. q: [rows, cols / 2] bytes, element 2i in the low nibble of byte i, 2i + 1 in
 * the high nibble; s: [rows, cols / 16] e4m3 block-scale codes; *g: the fp32 matrix scale. */
ORC_API void orc_quant_weight_nvfp4(const uint16_t* w, int64_t rows, int64_t cols, uint8_t* q, uint8_t* s,
                                    float* g) {
  double amax = 0.0;
#pragma omp parallel for schedule(static) reduction(max : amax)
  for (int64_t i = 0; i < rows * cols; ++i) {
    double a = fabs(orc_bf16_to_double(w[i]));
    if (a > amax) amax = a;
  }
  const float gs = amax == 0.0 ? 1.0f : (float)(amax / 2688.0);
  const float d = (float)(6.0 * (double)gs);
  *g = gs;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < cols / 16; ++b) {
      const uint16_t* blk = w + r * cols + b * 16;
      double bmax = 0.0;
      for (int i = 0; i < 16; ++i) {
        double a = fabs(orc_bf16_to_double(blk[i]));
        if (a > bmax) bmax = a;
      }
      const uint8_t sc = orc_e4m3_encode((float)(bmax / (double)d));
      s[r * (cols / 16) + b] = sc;
      const float p = (float)(orc_e4m3_decode(sc) * (double)gs);
      for (int i = 0; i < 16; i += 2) {
        uint8_t c0 = 0, c1 = 0;
        if (p != 0.0f) {
          c0 = orc_e2m1_encode((float)(orc_bf16_to_double(blk[i]) / (double)p));
          c1 = orc_e2m1_encode((float)(orc_bf16_to_double(blk[i + 1]) / (double)p));
        }
        q[r * (cols / 2) + b * 8 + i / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
}

/* Value of element (r, c) of an NVFP4 matrix: e2m1 * e4m3 block scale * matrix scale. */
static double orc_nvfp4_value(const uint8_t* q, const uint8_t* s, float g, int64_t cols, int64_t r, int64_t c) {
  uint8_t byte = q[r * (cols / 2) + c / 2];
  uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
  return orc_e2m1_decode(code) * orc_e4m3_decode(s[r * (cols / 16) + c / 16]) * (double)g;
}

ORC_API void orc_dequant_nvfp4(const uint8_t* q, const uint8_t* s, float g, int64_t rows, int64_t cols, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = orc_nvfp4_value(q, s, g, cols, r, c);
}

/* ------------------------------------------------------------------------------------------
 * Step 1: router scores. logits[t,e] = sum_d x[t,d] * W_r[e,d] in fp64, rounded once to
 * fp32 ([ULTRA] step 1: the router scores every token against every expert). No router
 * bias term (reading R5).
 * ---------------------------------------------------------------------------------------- */
ORC_API void orc_router_logits(const uint16_t* x, const float* w_r, int64_t T, int64_t h, int64_t E,
                               float* logits) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t d = 0; d < h; ++d) acc += orc_bf16_to_double(x[t * h + d]) * (double)w_r[e * h + d];
      logits[t * E + e] = (float)acc;
    }
}

/* ------------------------------------------------------------------------------------------
 * Step 1 (cont.): top-k selection and routed weights.
 *   score 0 (softmax, Mixtral): key = logit; weight = softmax probability over all E experts.
 *   score 1 (sigmoid, DeepSeek-V3): s = sigmoid(logit); key = s + bias (bias selects only,
 *     [ULTRA] "Load balancing and capacity"); group stage first, then top-k inside the kept
 *     groups ([TRTLLM] "Top-K kernel fusion"); weight = s.
 *   renorm: divide the selected weights by their sum; then multiply by routed_scale.
 * Output order within a token: descending key, ties to the lower expert index.
 * ---------------------------------------------------------------------------------------- */

/* index of the largest key among entries with allowed[i] != 0, ties to the lower index */
static int orc_argmax_allowed(const float* key, const unsigned char* allowed, int n) {
  int best = -1;
  for (int i = 0; i < n; ++i) {
    if (!allowed[i]) continue;
    if (best < 0 || key[i] > key[best]) best = i;
  }
  return best;
}

ORC_API int orc_route(const float* logits, const float* bias, int64_t T, int E, int k, int n_group,
                      int topk_group, int score, int renorm, float routed_scale, int32_t* topk_idx,
                      float* topk_w) {
  if (k < 1 || k > E || n_group < 1 || E % n_group != 0 || topk_group < 1 || topk_group > n_group) return -1;
  int gsize = E / n_group;
  if (topk_group * gsize < k) return -1;
  float* key = (float*)malloc(sizeof(float) * E);
  float* s = (float*)malloc(sizeof(float) * E);
  float* gscore = (float*)malloc(sizeof(float) * n_group);
  unsigned char* allowed = (unsigned char*)malloc(E);
  unsigned char* gallowed = (unsigned char*)malloc(n_group);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    for (int e = 0; e < E; ++e) {
      if (score == 0) {
        s[e] = l[e];
        key[e] = l[e];
      } else {
        s[e] = (float)(1.0 / (1.0 + exp(-(double)l[e]))); /* reading R3 */
        key[e] = bias ? s[e] + bias[e] : s[e];           /* fp32 add */
      }
    }
    /* group stage: keep the topk_group groups with the largest group score */
    for (int e = 0; e < E; ++e) allowed[e] = 1;
    if (n_group > 1) {
      for (int g = 0; g < n_group; ++g) {
        const float* kg = key + g * gsize;
        int i1 = 0;
        for (int i = 1; i < gsize; ++i)
          if (kg[i] > kg[i1]) i1 = i;
        float top2 = kg[i1];
        if (gsize > 1) {
          int i2 = -1;
          for (int i = 0; i < gsize; ++i)
            if (i != i1 && (i2 < 0 || kg[i] > kg[i2])) i2 = i;
          top2 = kg[i1] + kg[i2]; /* reading R1, fp32 add */
        }
        gscore[g] = top2;
      }
      for (int g = 0; g < n_group; ++g) gallowed[g] = 1;
      unsigned char* kept = (unsigned char*)calloc(n_group, 1);
      for (int r = 0; r < topk_group; ++r) {
        int g = orc_argmax_allowed(gscore, gallowed, n_group);
        kept[g] = 1;
        gallowed[g] = 0;
      }
      for (int e = 0; e < E; ++e) allowed[e] = kept[e / gsize];
      free(kept);
    }
    /* expert stage: k largest keys among the allowed experts */
    for (int j = 0; j < k; ++j) {
      int e = orc_argmax_allowed(key, allowed, E);
      topk_idx[t * k + j] = e;
      allowed[e] = 0;
    }
    /* routed weights */
    double wsel[64];
    double denom = 0.0;
    if (score == 0) {
      double mx = -INFINITY, z = 0.0;
      for (int e = 0; e < E; ++e)
        if ((double)l[e] > mx) mx = (double)l[e];
      for (int e = 0; e < E; ++e) z += exp((double)l[e] - mx);
      for (int j = 0; j < k; ++j) wsel[j] = exp((double)l[topk_idx[t * k + j]] - mx) / z;
    } else {
      for (int j = 0; j < k; ++j) wsel[j] = (double)s[topk_idx[t * k + j]];
    }
    for (int j = 0; j < k; ++j) denom += wsel[j];
    for (int j = 0; j < k; ++j) {
      double w = renorm ? wsel[j] / denom : wsel[j];
      topk_w[t * k + j] = (float)(w * (double)routed_scale);
    }
  }
  free(key);
  free(s);
  free(gscore);
  free(allowed);
  free(gallowed);
  return 0;
}

/* ------------------------------------------------------------------------------------------
 * Step 2: dispatch as a local permute. Routing information aggregated per expert ([PPLX]
 * "MoE Router": dense dispatch needs it per expert, not per token): counts, exclusive
 * offsets, and the expert-major row of every (token, slot). Within one expert the rows are
 * in ascending token order. Dropless: no capacity limit.
 * ---------------------------------------------------------------------------------------- */
ORC_API int orc_permute(const int32_t* topk_idx, int64_t T, int k, int E, int32_t* counts, int32_t* offsets,
                        int32_t* inv_pos, int32_t* row_token) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * k; ++i) {
    if (topk_idx[i] < 0 || topk_idx[i] >= E) return -1;
    counts[topk_idx[i]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int e = 0; e < E; ++e) {
    int32_t r = 0;
    for (int64_t t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (topk_idx[t * k + j] == e) {
          int32_t row = offsets[e] + r++;
          row_token[row] = (int32_t)t;
          inv_pos[t * k + j] = row;
        }
  }
  return 0;
}

/* Capacity limit ([ULTRA] "Load balancing and capacity": each expert accepts at most a fixed number
 * of assignments per batch, e.g. 1.25 times the fair share; the rest skip the expert). The expert keeps
 * its earliest `cap` tokens (ascending token order); a dropped (token, slot) gets inv_pos = -1 and no
 * row. cap <= 0 means no limit. */
ORC_API int orc_permute_capacity(const int32_t* topk_idx, int64_t T, int k, int E, int32_t cap, int32_t* counts,
                                 int32_t* offsets, int32_t* inv_pos, int32_t* row_token) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < T * k; ++i) {
    if (topk_idx[i] < 0 || topk_idx[i] >= E) return -1;
    inv_pos[i] = -1;
  }
  for (int e = 0; e < E; ++e) {
    int32_t taken = 0;
    for (int64_t t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (topk_idx[t * k + j] == e && (cap <= 0 || taken < cap)) taken++;
    counts[e] = taken;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int e = 0; e < E; ++e) {
    int32_t r = 0;
    for (int64_t t = 0; t < T && r < counts[e]; ++t)
      for (int j = 0; j < k; ++j)
        if (topk_idx[t * k + j] == e) {
          int32_t row = offsets[e] + r++;
          row_token[row] = (int32_t)t;
          inv_pos[t * k + j] = row;
        }
  }
  return 0;
}

/* Dispatch copy ([INFRA] 3.1 step 2: the hidden state of each token is copied once per
 * chosen expert): xd[row] = x[row_token[row]]. Element type of width `elem` bytes. */
ORC_API void orc_gather_rows(const void* x, int64_t h, int elem, const int32_t* row_token, int64_t R, void* xd) {
  for (int64_t r = 0; r < R; ++r)
    memcpy((char*)xd + r * h * elem, (const char*)x + (int64_t)row_token[r] * h * elem, (size_t)(h * elem));
}

/* ------------------------------------------------------------------------------------------
 * Step 3: one expert's SwiGLU FFN ([INFRA] 2.1: an expert is gate, up and down matrices;
 * [PPLX] "Quantization": SiLU activation).
 *   g = x W_gate^T, u = x W_up^T (fp64);  a = silu(g) * u stored in bf16 (reading R8);
 *   o = a W_down^T (fp64).
 * x: [m, h] bf16; w_gu: [2I, h] bf16, rows [0, I) gate and [I, 2I) up; w_d: [h, I] bf16.
 * out: [m, h] doubles.
 * ---------------------------------------------------------------------------------------- */
static double orc_silu(double g) { return g / (1.0 + exp(-g)); }

ORC_API void orc_expert_ffn_bf16(const uint16_t* x, int64_t m, int64_t h, int64_t I, const uint16_t* w_gu,
                                 const uint16_t* w_d, double* out) {
  double* a = (double*)malloc(sizeof(double) * I);
  for (int64_t r = 0; r < m; ++r) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < I; ++c) {
      double g = 0.0, u = 0.0;
      for (int64_t d = 0; d < h; ++d) {
        double xv = orc_bf16_to_double(x[r * h + d]);
        g += xv * orc_bf16_to_double(w_gu[c * h + d]);
        u += xv * orc_bf16_to_double(w_gu[(I + c) * h + d]);
      }
      a[c] = orc_bf16_to_double(orc_bf16_from_double(orc_silu(g) * u));
    }
#pragma omp parallel for schedule(static)
    for (int64_t d = 0; d < h; ++d) {
      double o = 0.0;
      for (int64_t c = 0; c < I; ++c) o += a[c] * orc_bf16_to_double(w_d[d * I + c]);
      out[r * h + d] = o;
    }
  }
  free(a);
}

/* FP8 block-scaled variant ([PPLX] "Quantization"): operands are e4m3 codes with fp32
 * scales; a value is code * scale. xq: [m, h], xs: [m, h/128]; w_gu_q: [2I, h] with
 * w_gu_s: [2I/128, h/128]; w_d_q: [h, I] with w_d_s: [h/128, I/128]. Every operand is first
 * dequantised to its value (exact in fp64: a 4-bit significand times a 24-bit one), then the
 * FFN runs on the values in fp64 as in the bf16 layer. The SwiGLU product is quantised 1x128
 * along I ([PPLX]: SiLU output block-quantised with a 128-element amax) and dequantised before
 * the down projection. */
ORC_API void orc_expert_ffn_fp8(const uint8_t* xq, const float* xs, int64_t m, int64_t h, int64_t I,
                                const uint8_t* w_gu_q, const float* w_gu_s, const uint8_t* w_d_q,
                                const float* w_d_s, double* out) {
  int64_t hb = h / 128, ib = I / 128;
  double* wgu = (double*)malloc(sizeof(double) * 2 * I * h);
  double* wd = (double*)malloc(sizeof(double) * h * I);
  double* xv = (double*)malloc(sizeof(double) * h);
  double* a = (double*)malloc(sizeof(double) * I);
  double* av = (double*)malloc(sizeof(double) * I);
  uint8_t* aq = (uint8_t*)malloc(I);
  float* as = (float*)malloc(sizeof(float) * ib);
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < 2 * I; ++c)
    for (int64_t d = 0; d < h; ++d)
      wgu[c * h + d] = orc_e4m3_decode(w_gu_q[c * h + d]) * (double)w_gu_s[(c / 128) * hb + d / 128];
#pragma omp parallel for schedule(static)
  for (int64_t d = 0; d < h; ++d)
    for (int64_t c = 0; c < I; ++c)
      wd[d * I + c] = orc_e4m3_decode(w_d_q[d * I + c]) * (double)w_d_s[(d / 128) * ib + c / 128];
  for (int64_t r = 0; r < m; ++r) {
    for (int64_t d = 0; d < h; ++d) xv[d] = orc_e4m3_decode(xq[r * h + d]) * (double)xs[r * hb + d / 128];
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < I; ++c) {
      double g = 0.0, u = 0.0;
      for (int64_t d = 0; d < h; ++d) {
        g += xv[d] * wgu[c * h + d];
        u += xv[d] * wgu[(I + c) * h + d];
      }
      a[c] = orc_silu(g) * u;
    }
    orc_quant_1x128(a, 1, I, aq, as);
    for (int64_t c = 0; c < I; ++c) av[c] = orc_e4m3_decode(aq[c]) * (double)as[c / 128];
#pragma omp parallel for schedule(static)
    for (int64_t d = 0; d < h; ++d) {
      double o = 0.0;
      for (int64_t c = 0; c < I; ++c) o += av[c] * wd[d * I + c];
      out[r * h + d] = o;
    }
  }
  free(wgu);
  free(wd);
  free(xv);
  free(a);
  free(av);
  free(aq);
  free(as);
}

/* NVFP4-weight variant (readings R19, R20): bf16 activations, weights given as NVFP4 matrices
 * w_gu: [2I, h] (codes [2I, h/2], scales [2I, h/16], matrix scale g_gu) and w_d: [h, I]; the
 * weights are dequantised to fp64 first (exact), then the SwiGLU FFN runs as in the bf16 layer,
 * with the product stored in bf16 (R8). */
ORC_API void orc_expert_ffn_nvfp4(const uint16_t* x, int64_t m, int64_t h, int64_t I, const uint8_t* w_gu_q,
                                  const uint8_t* w_gu_s, float g_gu, const uint8_t* w_d_q, const uint8_t* w_d_s,
                                  float g_d, double* out) {
  double* gu = (double*)malloc(sizeof(double) * 2 * I * h);
  double* wd = (double*)malloc(sizeof(double) * h * I);
  double* a = (double*)malloc(sizeof(double) * I);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < 2 * I; ++r)
    for (int64_t c = 0; c < h; ++c) gu[r * h + c] = orc_nvfp4_value(w_gu_q, w_gu_s, g_gu, h, r, c);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < h; ++r)
    for (int64_t c = 0; c < I; ++c) wd[r * I + c] = orc_nvfp4_value(w_d_q, w_d_s, g_d, I, r, c);
  for (int64_t r = 0; r < m; ++r) {
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < I; ++c) {
      double g = 0.0, u = 0.0;
      for (int64_t d = 0; d < h; ++d) {
        double xv = orc_bf16_to_double(x[r * h + d]);
        g += xv * gu[c * h + d];
        u += xv * gu[(I + c) * h + d];
      }
      a[c] = orc_bf16_to_double(orc_bf16_from_double(orc_silu(g) * u));
    }
#pragma omp parallel for schedule(static)
    for (int64_t d = 0; d < h; ++d) {
      double o = 0.0;
      for (int64_t c = 0; c < I; ++c) o += a[c] * wd[d * I + c];
      out[r * h + d] = o;
    }
  }
  free(gu);
  free(wd);
  free(a);
}

/* ------------------------------------------------------------------------------------------
 * Step 4: combine ([ULTRA] step 4 and [INFRA] 3.1 step 4: outputs return to their token and
 * are summed weighted by the route weights; [INFRA] 7: the shared expert is one more expert
 * every token uses, weight 1, reading R7). Rounded once to bf16.
 * o: [n, k, h] expert output of each (token, slot); w: [n, k]; shared: [n, h] or NULL.
 * ---------------------------------------------------------------------------------------- */
ORC_API void orc_combine(const double* o, const float* w, const double* shared, int64_t n, int k, int64_t h,
                         uint16_t* y) {
  for (int64_t t = 0; t < n; ++t)
    for (int64_t d = 0; d < h; ++d) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += (double)w[t * k + j] * o[(t * k + j) * h + d];
      if (shared) acc += shared[t * h + d];
      y[t * h + d] = orc_bf16_from_double(acc);
    }
}

/* ------------------------------------------------------------------------------------------
 * Array forms of the scalar codecs above, for the Python wrapper.
 * ---------------------------------------------------------------------------------------- */
ORC_API void orc_bf16_from_double_n(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_double(v[i]);
}
ORC_API void orc_bf16_to_double_n(const uint16_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_double(b[i]);
}
ORC_API void orc_e4m3_encode_n(const float* f, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(f[i]);
}
ORC_API void orc_e4m3_decode_n(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}
