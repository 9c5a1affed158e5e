/*
 * Plain, slow CPU oracle for the fused Mixture-of-Experts layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The GPU library shares no
 * code, header, table or constant with it.
 *
 * What is computed, and where it comes from ("Amazon SageMaker AI 上的
 * Mixture-of-Experts 内核工程优化", the English original page):
 *   - the fused MoE layer merges token routing, data shuffling (regrouping of
 *     tokens by expert) and the expert network computation into one batched
 *     operation (section "Introduction");
 *   - the FP8 per-tensor-quantised variant applies FP8 tensor scaling, the
 *     matrix multiplications and the expert aggregation in one pass (section
 *     "Backend routing for FP8 tensor quantization");
 *   - the swapped operand order B^T[N,K] x A^T[K,M] = C^T[N,M] changes no
 *     arithmetic (section "Swap-AB for WGMMA utilization"), so the oracle uses
 *     the plain per-expert product.
 * FP8 is E4M3 (4 exponent bits, 3 mantissa bits), as named by the Chinese
 * commentary page ("FP8" background box) and defined by the OCP 8-bit
 * floating point specification.
 *
 * Where the pages are silent the plainest reading is taken:
 *   router  = softmax over all E logits, top-k on the raw fp32 logits with
 *             ties broken towards the lower expert index, optional
 *             renormalisation of the k selected probabilities;
 *   expert  = SwiGLU MLP: rows [0,I) of w13 are the gate, rows [I,2I) the up
 *             projection, h = SiLU(gate) * up, y = w2 h, no bias;
 *   FP8     = one fp32 scale per expert per weight tensor (given as input),
 *             one dynamic fp32 scale per activation tensor: s = amax / 448
 *             (1 when amax == 0), q(v) = E4M3_rne_satfinite(fp32(v) / s)
 *             with an IEEE fp32 division, dequantised value = code * s;
 *   combine = out[t] = sum_j w[t,j] * y[t,j].
 * Everything else is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Scalar formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3 (OCP "E4M3FN"): bias 7, no infinities, S.1111.111 is NaN, largest
 * finite magnitude 1.75 * 2^8 = 448, exponent field 0 holds subnormals
 * m * 2^-9.  Decoding follows the definition field by field. */
double oracle_e4m3_decode(uint8_t code) {
  int sign = code >> 7;
  int ef = (code >> 3) & 0xF;
  int mant = code & 0x7;
  double v;
  if (ef == 0xF && mant == 0x7) return NAN;
  if (ef == 0)
    v = ldexp((double)mant, -9);
  else
    v = ldexp(1.0 + mant / 8.0, ef - 7);
  return sign ? -v : v;
}

/* Round-to-nearest-even to the E4M3 grid, saturating to +-448 (the
 * "satfinite" behaviour: overflow gives the largest finite value, never NaN).
 * Inside one binade [2^e, 2^(e+1)) the grid step is 2^(e-3); below the
 * smallest normal 2^-6 the step is the subnormal step 2^-9. */
uint8_t oracle_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  if (isnan(v)) return 0x7F;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex);              /* a = m * 2^ex, m in [0.5, 1) */
  int e = ex - 1;             /* floor(log2(a)) */
  if (e < -6) e = -6;
  double step = ldexp(1.0, e - 3);
  double r = nearbyint(a / step); /* a/step is exact; default mode is ties-to-even */
  double q = r * step;
  if (q == 0.0) return sign;
  frexp(q, &ex);
  e = ex - 1;
  if (e < -6) {
    int mant = (int)(q / ldexp(1.0, -9));
    return (uint8_t)(sign | mant);
  }
  int mant = (int)((q / ldexp(1.0, e) - 1.0) * 8.0);
  return (uint8_t)(sign | ((e + 7) << 3) | mant);
}

/* Dynamic per-tensor activation scale: amax / 448 in fp32, 1 when amax is 0. */
static float act_scale_from_amax(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  return amax / 448.0f;
}

/* q(v; s) = E4M3(fp32(v) / s), the division done in IEEE fp32. */
static uint8_t quantize(double v, float s) {
  float num = (float)v;
  float qv = num / s;
  return oracle_e4m3_encode(qv);
}

uint8_t oracle_quantize(double v, float s) { return quantize(v, s); }

/* Dynamic per-tensor quantisation of a bf16 tensor: s = amax/448 (1 if the
 * tensor is zero), codes = E4M3(fp32(x) / s). */
void oracle_quantize_act(const uint16_t* x, long n, uint8_t* codes, float* s_out) {
  float amax = 0.0f;
  for (long i = 0; i < n; ++i) {
    float a = fabsf((float)bf16_bits_to_double(x[i]));
    if (a > amax) amax = a;
  }
  float s = act_scale_from_amax(amax);
  for (long i = 0; i < n; ++i) codes[i] = quantize(bf16_bits_to_double(x[i]), s);
  *s_out = s;
}

void oracle_e4m3_encode_n(const float* v, long n, uint8_t* out) {
  for (long i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------ */
/* Router                                                              */
/* ------------------------------------------------------------------ */

/* Per token: softmax over the E logits (fp64, max-subtracted); pick k experts
 * by (logit descending, expert index ascending), comparing the fp32 logits as
 * given; weight_j = p_j, divided by the sum of the k selected p when
 * renormalize is set.  ids/weights are [T, k], slot j in selection order. */
void oracle_route_topk(const float* logits, int T, int E, int k, int renormalize,
                       int32_t* ids, double* weights) {
  char* taken = (char*)malloc((size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)k);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    double m = -INFINITY;
    for (int e = 0; e < E; ++e)
      if ((double)l[e] > m) m = (double)l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp((double)l[e] - m);
    memset(taken, 0, (size_t)E);
    double sel = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: lower index keeps ties */
      }
      taken[best] = 1;
      ids[(size_t)t * k + j] = best;
      p[j] = exp((double)l[best] - m) / z;
      sel += p[j];
    }
    for (int j = 0; j < k; ++j)
      weights[(size_t)t * k + j] = renormalize ? p[j] / sel : p[j];
  }
  free(p);
  free(taken);
}

/* ------------------------------------------------------------------ */
/* Alignment by expert ("data shuffling")                              */
/* ------------------------------------------------------------------ */

/* Pairs p = t*k + j are regrouped by expert.  counts[e] = number of pairs
 * routed to e; each expert's segment is padded to a multiple of block_m;
 * offsets = exclusive prefix sum of the padded sizes (offsets[E] = total);
 * inside a segment the pair ids ascend (stable order), padding slots hold the
 * sentinel P; tile_expert[b] is the expert owning rows [b*block_m, (b+1)*block_m).
 * sorted_ids needs P + E*(block_m-1) entries, tile_expert that divided by
 * block_m. */
void oracle_align(const int32_t* ids, int T, int k, int E, int block_m,
                  int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                  int32_t* tile_expert, int32_t* num_padded) {
  long P = (long)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long p = 0; p < P; ++p) counts[ids[p]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    int padded = (counts[e] + block_m - 1) / block_m * block_m;
    offsets[e + 1] = offsets[e] + padded;
  }
  *num_padded = offsets[E];
  for (int r = 0; r < offsets[E]; ++r) sorted_ids[r] = (int32_t)P;
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (long p = 0; p < P; ++p) {
    int e = ids[p];
    sorted_ids[offsets[e] + fill[e]] = (int32_t)p;
    fill[e] += 1;
  }
  free(fill);
  for (int e = 0; e < E; ++e)
    for (int r = offsets[e]; r < offsets[e + 1]; r += block_m) tile_expert[r / block_m] = e;
}

/* ------------------------------------------------------------------ */
/* Whole layer                                                         */
/* ------------------------------------------------------------------ */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Fused MoE layer forward.
 *   x        bf16 bits [T, H]
 *   logits   fp32 [T, E]
 *   w13      [E, 2I, H]: bf16 bits (is_fp8 = 0) or E4M3 codes (is_fp8 = 1)
 *   w2       [E, H, I]:  same element type as w13
 *   w13_scale, w2_scale  fp32 [E] (FP8 only; the weight value is code * scale)
 *   out      fp64 [n_rows, H]: the output rows of the tokens listed in
 *            `rows` (all T tokens in order when rows == NULL, n_rows = T)
 *   ids, weights, counts   routing results [T,k], [T,k], [E] (may be NULL)
 *   s_x_out, s_h_out       the activation scales used (FP8; may be NULL)
 *   h_amax_in              > 0: the max |h| the scale of h is taken from, in
 *                          place of this call's own (tensor-parallel shards:
 *                          the max over every shard's h); <= 0: this call's
 *   h_amax_out             this call's own max |h| over its routed pairs (FP8;
 *                          may be NULL)
 *   nthreads               OpenMP threads (<= 0: runtime default)
 * The dynamic scale of h spans every routed pair of the call, so in the FP8
 * path h is formed for all pairs even when only some output rows are asked for.
 * Returns 0 on success, nonzero on a bad argument or allocation failure.
 */
int oracle_moe_forward(const uint16_t* x, const float* logits, const void* w13, const void* w2,
                       const float* w13_scale, const float* w2_scale, int is_fp8, int T, int H,
                       int I, int E, int k, int renormalize, const int32_t* rows, int n_rows,
                       double* out, int32_t* ids_out, double* weights_out, int32_t* counts_out,
                       float* s_x_out, float* s_h_out, float h_amax_in, float* h_amax_out,
                       int nthreads) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E) return 1;
  if (rows == NULL) n_rows = T;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  long P = (long)T * k;
  /* value of every E4M3 code, from the field-by-field decoder above */
  double dec[256];
  for (int b = 0; b < 256; ++b) dec[b] = oracle_e4m3_decode((uint8_t)b);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
  double* wts = (double*)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1));
  if (!ids || !wts) return 2;

  /* 1. token routing */
  oracle_route_topk(logits, T, E, k, renormalize, ids, wts);
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)P);
  if (weights_out) memcpy(weights_out, wts, sizeof(double) * (size_t)P);
  if (counts_out) {
    for (int e = 0; e < E; ++e) counts_out[e] = 0;
    for (long p = 0; p < P; ++p) counts_out[ids[p]] += 1;
  }

  /* 2. activation as the expert GEMMs see it: x, or dq(q(x; s_x)) */
  double* xv = (double*)malloc(sizeof(double) * (size_t)T * H + 1);
  float s_x = 1.0f;
  if (is_fp8) {
    float amax = 0.0f;
    for (long i = 0; i < (long)T * H; ++i) {
      float a = fabsf((float)bf16_bits_to_double(x[i]));
      if (a > amax) amax = a;
    }
    s_x = act_scale_from_amax(amax);
    for (long i = 0; i < (long)T * H; ++i)
      xv[i] = dec[quantize(bf16_bits_to_double(x[i]), s_x)] * (double)s_x;
  } else {
    for (long i = 0; i < (long)T * H; ++i) xv[i] = bf16_bits_to_double(x[i]);
  }
  if (s_x_out) *s_x_out = s_x;

  /* which pairs need h: all of them in the FP8 path (global scale of h),
   * otherwise only the pairs of the requested rows */
  char* need = (char*)calloc((size_t)(P > 0 ? P : 1), 1);
  if (is_fp8 || rows == NULL) {
    memset(need, 1, (size_t)P);
  } else {
    for (int r = 0; r < n_rows; ++r)
      for (int j = 0; j < k; ++j) need[(long)rows[r] * k + j] = 1;
  }

  /* 3. expert up-projection and SwiGLU, per routed pair */
  double* h = (double*)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1) * I);
  const uint8_t* w13_8 = (const uint8_t*)w13;
  const uint16_t* w13_16 = (const uint16_t*)w13;
#pragma omp parallel for schedule(dynamic, 1)
  for (long p = 0; p < P; ++p) {
    if (!need[p]) continue;
    long t = p / k;
    int e = ids[p];
    const double* xr = xv + t * H;
    for (int i = 0; i < I; ++i) {
      size_t grow = ((size_t)e * 2 * I + (size_t)i) * H;
      size_t urow = ((size_t)e * 2 * I + (size_t)I + (size_t)i) * H;
      double g = 0.0, u = 0.0;
      if (is_fp8) {
        double s = (double)w13_scale[e];
        for (int c = 0; c < H; ++c) g += dec[w13_8[grow + c]] * s * xr[c];
        for (int c = 0; c < H; ++c) u += dec[w13_8[urow + c]] * s * xr[c];
      } else {
        for (int c = 0; c < H; ++c) g += bf16_bits_to_double(w13_16[grow + c]) * xr[c];
        for (int c = 0; c < H; ++c) u += bf16_bits_to_double(w13_16[urow + c]) * xr[c];
      }
      h[(size_t)p * I + i] = silu(g) * u;
    }
  }

  /* 4. h as the down projection sees it: h, or dq(q(h; s_h)) */
  float s_h = 1.0f;
  if (is_fp8) {
    float amax = 0.0f;
    for (long i = 0; i < P * (long)I; ++i) {
      float a = fabsf((float)h[i]);
      if (a > amax) amax = a;
    }
    if (h_amax_out) *h_amax_out = amax;
    s_h = act_scale_from_amax(h_amax_in > 0.0f ? h_amax_in : amax);
#pragma omp parallel for schedule(static)
    for (long i = 0; i < P * (long)I; ++i)
      h[i] = dec[quantize(h[i], s_h)] * (double)s_h;
  }
  if (s_h_out) *s_h_out = s_h;

  /* 5. down projection and top-k weighted combine */
  const uint8_t* w2_8 = (const uint8_t*)w2;
  const uint16_t* w2_16 = (const uint16_t*)w2;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < n_rows; ++r) {
    long t = rows ? rows[r] : r;
    double* o = out + (size_t)r * H;
    for (int c = 0; c < H; ++c) o[c] = 0.0;
    for (int j = 0; j < k; ++j) {
      long p = t * k + j;
      int e = ids[p];
      const double* hr = h + (size_t)p * I;
      for (int c = 0; c < H; ++c) {
        size_t wrow = ((size_t)e * H + (size_t)c) * I;
        double y = 0.0;
        if (is_fp8) {
          double s = (double)w2_scale[e];
          for (int i = 0; i < I; ++i) y += dec[w2_8[wrow + i]] * s * hr[i];
        } else {
          for (int i = 0; i < I; ++i) y += bf16_bits_to_double(w2_16[wrow + i]) * hr[i];
        }
        o[c] += wts[p] * y;
      }
    }
  }

  free(h);
  free(need);
  free(xv);
  free(wts);
  free(ids);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Inverse rotary position embedding + per-head FP8 quantisation       */
/* ------------------------------------------------------------------ */
/* The pages name one more kernel, _fused_inv_rope_fp8_quant_per_head
 * (section "Triton JIT recompilation elimination": it fuses rotary position
 * embedding with FP8 quantisation and was recompiled for every new number of
 * tokens), and give none of its arithmetic.  Reading taken here:
 *   rotary embedding: the RoFormer rotation of the consecutive pairs
 *     (2i, 2i+1) of each head vector by the angle pos * theta_i; the caller
 *     supplies cos and sin of those angles per position ([max_pos][D/2]
 *     each, fp32), so every implementation rotates with the same values;
 *   inverse: rotation by the negated angle,
 *     y[2i]   = x[2i] c + x[2i+1] s,   y[2i+1] = x[2i+1] c - x[2i] s,
 *     each product rounded to fp32, then the sum or difference;
 *   per-head FP8: one dynamic scale per head over all tokens,
 *     s_h = amax over tokens and dims of |y[., h, .]| / 448 (1 if 0),
 *     code = E4M3(fp32(y) / s_h), the division in IEEE fp32.
 * x: bf16 [T][NH][D]; pos: int32 [T] in [0, max_pos); codes: [T][NH][D];
 * scales: [NH]; y (optional): the rotated values, fp32 [T][NH][D].
 * Returns 0, or -1 for an odd D or a position outside the tables. */
int oracle_inv_rope_quant(const uint16_t* x, const int32_t* pos, const float* cos_tab,
                          const float* sin_tab, int T, int NH, int D, int max_pos,
                          uint8_t* codes, float* scales, float* y) {
  if (D % 2 != 0) return -1;
  for (int t = 0; t < T; ++t)
    if (pos[t] < 0 || pos[t] >= max_pos) return -1;
  const int half = D / 2;
  const long n = (long)T * NH * D;
  float* yy = y ? y : (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  if (!yy) return -1;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < NH; ++h)
      for (int i = 0; i < half; ++i) {
        const long at = ((long)t * NH + h) * D + 2 * i;
        const float x0 = (float)bf16_bits_to_double(x[at]);
        const float x1 = (float)bf16_bits_to_double(x[at + 1]);
        const float c = cos_tab[(long)pos[t] * half + i];
        const float sn = sin_tab[(long)pos[t] * half + i];
        const float a = x0 * c, b = x1 * sn;  /* each product rounded to fp32 */
        const float d = x1 * c, e = x0 * sn;
        yy[at] = a + b;
        yy[at + 1] = d - e;
      }
  for (int h = 0; h < NH; ++h) {
    float amax = 0.0f;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < D; ++j) {
        const float v = fabsf(yy[((long)t * NH + h) * D + j]);
        if (v > amax) amax = v;
      }
    scales[h] = act_scale_from_amax(amax);
  }
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < NH; ++h)
      for (int j = 0; j < D; ++j) {
        const long at = ((long)t * NH + h) * D + j;
        codes[at] = quantize(yy[at], scales[h]);
      }
  if (!y) free(yy);
  return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
