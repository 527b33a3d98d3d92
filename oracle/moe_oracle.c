/*
 * Plain CPU oracle of the fused Mixture-of-Experts layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; both sides only see the same seeded inputs.
 *
 * Every step is written the slow, obvious way, in double precision, one token
 * at a time, in the order the pages describe the layer:
 *
 *   route -> process the token with each of its top-k experts -> weighted sum
 *   ("FusedMoE vs MegaMoE" (zwxr.cn), section 2: the router produces a weight
 *   distribution, the k best experts process the token, their results are
 *   summed with the weights; section 3.1: routing, sorting by expert, index
 *   construction, fused expert computation, reorder + weighted sum).
 *
 * Readings of points the pages leave open (each one is a named choice):
 *   - softmax over all E experts, then top-k; renormalisation optional;
 *   - ranking by probability == ranking by logit (softmax is strictly
 *     monotone); equal logits rank the lower expert index first;
 *   - w13[e] holds the gate rows [0, I) above the up rows [I, 2I);
 *     SiLU(z) = z / (1 + exp(-z)); the routing weight is applied after the
 *     down projection;
 *   - the permutation lists, expert by expert in ascending order, the flat
 *     pair indices f = t*k + j in ascending order, pads each expert to a
 *     multiple of the block size with the sentinel T*k, and gives empty
 *     experts no block;
 *   - FP8 (e4m3, OCP 8-bit floating point spec): one fp32 scale per expert
 *     weight tensor, one dynamic scale for the layer input and one for the
 *     intermediate activation, scale = amax / 448 (1 when amax is 0), codes by
 *     round-to-nearest-even with saturation to +-448.  The code decision is
 *     taken in fp32 (x / scale in fp32), the precision a kernel takes it in.
 *
 * Build: gcc -O2 -fPIC -shared -fopenmp (OpenMP only splits independent
 * tokens across threads; each token's arithmetic is unchanged).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_INT4 = 3 };

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16: the top 16 bits of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t v) {
  uint32_t bits = (uint32_t)v << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* binary32 -> bfloat16, round to nearest, ties to even (NaN stays NaN). */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu)) return (uint16_t)((bits >> 16) | 0x40u);
  uint32_t upper = bits >> 16;
  uint32_t lower = bits & 0xffffu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* E4M3 (OCP FP8): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite magnitude 448.
 * exponent field 0 is subnormal: value = mantissa/8 * 2^-6. */
double oracle_e4m3_to_f64(uint8_t c) {
  int sign = (c >> 7) & 1;
  int ex = (c >> 3) & 0xf;
  int man = c & 0x7;
  double mag;
  if (ex == 0xf && man == 0x7) return NAN;
  if (ex == 0)
    mag = ldexp((double)man / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)man / 8.0, ex - 7);
  return sign ? -mag : mag;
}

/* Decoded value of every e4m3 code, filled from oracle_e4m3_to_f64 before any
 * parallel region (a cache of the decoder above, for speed only). */
static double e4m3_table[256];
static int e4m3_table_ready = 0;
static void e4m3_table_init(void) {
  if (e4m3_table_ready) return;
  for (int c = 0; c < 256; ++c) e4m3_table[c] = oracle_e4m3_to_f64((uint8_t)c);
  e4m3_table_ready = 1;
}

/* float -> E4M3, round to nearest with ties to even, saturating to +-448.
 * The 127 non-negative finite codes are in increasing order of value: find
 * the largest code not above |f| (binary search over the decoded values),
 * then pick the nearer of it and the next code, the even code on a tie. */
uint8_t oracle_f32_to_e4m3_satfinite(float f) {
  if (isnan(f)) return 0x7f;
  e4m3_table_init();
  uint8_t sign = signbit(f) ? 0x80 : 0x00;
  double a = fabs((double)f);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  int lo = 0, hi = 0x7e; /* invariant: table[lo] <= a < table[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (e4m3_table[mid] <= a) lo = mid; else hi = mid;
  }
  double vlo = e4m3_table[lo], vhi = e4m3_table[hi];
  int pick;
  if (a - vlo < vhi - a) pick = lo;
  else if (a - vlo > vhi - a) pick = hi;
  else pick = (lo & 1) ? hi : lo;
  return (uint8_t)(sign | pick);
}

static double load_elem(const void* p, int dtype, size_t i) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)p)[i];
    case ORC_BF16: return oracle_bf16_to_f64(((const uint16_t*)p)[i]);
    case ORC_E4M3: return e4m3_table[((const uint8_t*)p)[i]];
  }
  return NAN;
}

static float load_f32(const void* p, int dtype, size_t i) { return (float)load_elem(p, dtype, i); }

/*
 * INT4 weight-only experts ("FusedMoE vs MegaMoE" (zwxr.cn), section 6.3:
 * quantised expert weights with the fused kernel; the pages give no format).
 * Reading: a code q in [-8, 7] per weight (two's complement nibble) and one
 * bf16 scale s per (weight row, 128 consecutive K elements); the weight is
 * q * s rounded once to bf16 (nearest even).  Packing: each little-endian
 * 32-bit word holds 8 consecutive K elements, element e of the word in nibble
 * (e even ? e / 2 : 4 + e / 2).  K is the row length (H for w13, I for w2).
 * Scales are group-major per expert: [E][K/128][rows of one expert].
 */
static double load_w4(const void* codes, const void* scales, int ex, int r, int rows, int K, int k) {
  const size_t row = (size_t)ex * rows + r;
  const uint8_t* c = (const uint8_t*)codes + (row * (size_t)(K / 8) + (size_t)(k / 8)) * 4;
  const uint32_t word = (uint32_t)c[0] | ((uint32_t)c[1] << 8) | ((uint32_t)c[2] << 16) | ((uint32_t)c[3] << 24);
  const int e = k % 8;
  const int nib = (e % 2 == 0) ? e / 2 : 4 + e / 2;
  int q = (int)((word >> (4 * nib)) & 0xFu);
  if (q >= 8) q -= 16;
  const size_t si = ((size_t)ex * (K / 128) + (size_t)(k / 128)) * rows + r;
  const double s = oracle_bf16_to_f64(((const uint16_t*)scales)[si]);
  return oracle_bf16_to_f64(oracle_f32_to_bf16((float)(q * s)));  /* q * s is exact in fp32 */
}

/* weight w13[e][r][h] / w2[e][h][i] of the stored format */
static double w13_at(const void* W13, int w_dtype, const void* s13, int e, int r, int I, int H, int h) {
  const size_t row = (size_t)e * 2 * I + r;
  return w_dtype == ORC_INT4 ? load_w4(W13, s13, e, r, 2 * I, H, h) : load_elem(W13, w_dtype, row * H + h);
}
static double w2_at(const void* W2, int w_dtype, const void* s2, int e, int h, int H, int I, int i) {
  const size_t row = (size_t)e * H + h;
  return w_dtype == ORC_INT4 ? load_w4(W2, s2, e, h, H, I, i) : load_elem(W2, w_dtype, row * I + i);
}

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------ */
/* Step 1: router gate GEMM, logits[t][e] = sum_h X[t][h] * Wr[e][h]         */
/* ("FusedMoE vs MegaMoE", section 2: the router computes, per token, a      */
/*  weight distribution over the experts.)                                   */
/* ------------------------------------------------------------------------ */
void oracle_router_logits(const void* X, const void* Wr, int dtype, int T, int H, int E, double* logits) {
  e4m3_table_init();
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += load_elem(X, dtype, (size_t)t * H + h) * load_elem(Wr, dtype, (size_t)e * H + h);
      logits[(size_t)t * E + e] = s;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Step 2: softmax over all experts, top-k, optional renormalisation         */
/* ("FusedMoE vs MegaMoE", section 2: the k highest-weight experts are       */
/*  chosen; section 5 names this Top-k gating.)                              */
/* ------------------------------------------------------------------------ */
int oracle_topk(const double* logits, int T, int E, int k, int renorm, int32_t* ids, double* w) {
  if (k < 1 || k > E) return -1;
  char* taken = (char*)malloc((size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  if (!taken || !p) { free(taken); free(p); return -2; }
  for (int t = 0; t < T; ++t) {
    const double* l = logits + (size_t)t * E;
    double m = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - m); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
    memset(taken, 0, (size_t)E);
    /* k rounds of "pick the largest not yet taken"; the strict > keeps the
     * lower index on equal logits.  The ranking uses the logit itself, which
     * orders exactly like p (exp is strictly increasing). */
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;
      }
      taken[best] = 1;
      ids[(size_t)t * k + j] = best;
      w[(size_t)t * k + j] = p[best];
    }
    if (renorm) {
      double s = 0.0;
      for (int j = 0; j < k; ++j) s += w[(size_t)t * k + j];
      for (int j = 0; j < k; ++j) w[(size_t)t * k + j] /= s;
    }
  }
  free(taken);
  free(p);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 3: token-to-expert permutation                                       */
/* ("FusedMoE vs MegaMoE", section 3.1: sort the routed tokens by expert and */
/*  build the index that says which rows belong to which expert; page 1,     */
/*  "Routage backend...": variable token bucketing onto expert tiles.)       */
/* sorted capacity: T*k + min(E, T*k)*(B-1); expert_ids capacity: that / B.  */
/* ------------------------------------------------------------------------ */
int oracle_align(const int32_t* ids, int T, int k, int E, int B, int32_t* sorted, int32_t* expert_ids,
                 int32_t* num_post_pad, int32_t* counts) {
  if (B < 1) return -1;
  const int64_t n = (int64_t)T * k;
  const int32_t sentinel = (int32_t)n;
  int64_t pos = 0, blk = 0;
  for (int e = 0; e < E; ++e) {
    int64_t c = 0;
    for (int64_t f = 0; f < n; ++f) {
      if (ids[f] == e) { sorted[pos++] = (int32_t)f; ++c; }
    }
    if (counts) counts[e] = (int32_t)c;
    if (c == 0) continue;
    int64_t padded = (c + B - 1) / B * B;
    for (int64_t q = c; q < padded; ++q) sorted[pos++] = sentinel;
    for (int64_t b = 0; b < padded / B; ++b) expert_ids[blk++] = e;
  }
  *num_post_pad = (int32_t)pos;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Dynamic per-tensor e4m3 quantisation of one tensor (page 1, "Routage      */
/* backend pour la quantisation des tenseurs FP8": per-tensor FP8 with the   */
/* scale applied where the data is used, read from HBM once).               */
/* ------------------------------------------------------------------------ */
float oracle_e4m3_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

uint8_t oracle_e4m3_quant(float v, float scale) { return oracle_f32_to_e4m3_satfinite(v / scale); }

/* ------------------------------------------------------------------------ */
/* Steps 4-7: per-token expert FFNs and the routing-weighted combine.        */
/* out[i][:] is the output of token tokens[i] (or i when tokens is NULL).    */
/* The router is step 1-2 above, run on the stored inputs.                   */
/* ids_out / w_out (nullable) receive the routing of every one of the T      */
/* tokens.  In FP8 mode the two activation scales are layer-wide: the input  */
/* scale is taken over all T tokens, the intermediate one over every routed  */
/* (token, expert) pair of all T tokens, so the intermediate is formed for   */
/* all T tokens even when only a subset of outputs is asked for.             */
/* Returns 0, or a negative value on bad arguments.                          */
/* ------------------------------------------------------------------------ */
int oracle_moe_forward(const void* X, const void* Wr, const void* W13, const void* W2, int act_dtype, int w_dtype,
                       int T, int H, int I, int E, int k, int renorm, const void* w13_scale_in, const void* w2_scale_in,
                       const int32_t* tokens, int n_tokens, double* out, int32_t* ids_out, double* w_out,
                       float* act_scales_out) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || k > E) return -1;
  if (act_dtype != ORC_F32 && act_dtype != ORC_BF16) return -1;
  /* scales: [E] fp32 for e4m3 weights; bf16 [E][H/128][2I] and [E][I/128][H] for INT4 */
  const float* w13_scale = (const float*)w13_scale_in;
  const float* w2_scale = (const float*)w2_scale_in;
  if (w_dtype == ORC_INT4 && (!w13_scale_in || !w2_scale_in || H % 128 || I % 128 || H % 8 || I % 8)) return -1;
  const int fp8 = (w_dtype == ORC_E4M3);
  if (fp8 && (!w13_scale || !w2_scale || act_dtype != ORC_BF16)) return -1;
  if (!tokens) n_tokens = T;
  if (T == 0) return 0;
  e4m3_table_init();

  double* logits = (double*)malloc(sizeof(double) * (size_t)T * E);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  if (!logits || !ids || !w) { free(logits); free(ids); free(w); return -2; }
  oracle_router_logits(X, Wr, act_dtype, T, H, E, logits);
  oracle_topk(logits, T, E, k, renorm, ids, w);
  free(logits);
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * k);
  if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)T * k);

  if (!fp8) {
#pragma omp parallel
    {
      double* x = (double*)malloc(sizeof(double) * (size_t)H);
      double* a = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
      for (int q = 0; q < n_tokens; ++q) {
        const int t = tokens ? tokens[q] : q;
        double* o = out + (size_t)q * H;
        for (int h = 0; h < H; ++h) { x[h] = load_elem(X, act_dtype, (size_t)t * H + h); o[h] = 0.0; }
        for (int j = 0; j < k; ++j) {
          const int e = ids[(size_t)t * k + j];
          for (int i = 0; i < I; ++i) {
            double g = 0.0, u = 0.0;
            for (int h = 0; h < H; ++h) {
              g += w13_at(W13, w_dtype, w13_scale_in, e, i, I, H, h) * x[h];
              u += w13_at(W13, w_dtype, w13_scale_in, e, I + i, I, H, h) * x[h];
            }
            a[i] = oracle_silu(g) * u;
          }
          const double wj = w[(size_t)t * k + j];
          for (int h = 0; h < H; ++h) {
            double y = 0.0;
            for (int i = 0; i < I; ++i) y += w2_at(W2, w_dtype, w2_scale_in, e, h, H, I, i) * a[i];
            o[h] += wj * y;
          }
        }
      }
      free(x);
      free(a);
    }
    free(ids);
    free(w);
    return 0;
  }

  /* FP8: quantise the layer input with one dynamic scale. */
  float amax_x = 0.0f;
  for (size_t i = 0; i < (size_t)T * H; ++i) {
    float v = fabsf(load_f32(X, act_dtype, i));
    if (v > amax_x) amax_x = v;
  }
  const float s_a1 = oracle_e4m3_scale(amax_x);
  /* Intermediate activation of every routed pair, kept to find its scale. */
  double* A = (double*)malloc(sizeof(double) * (size_t)T * k * I);
  if (!A) { free(ids); free(w); return -2; }
#pragma omp parallel
  {
    double* xq = (double*)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
      for (int h = 0; h < H; ++h)
        xq[h] = e4m3_table[oracle_e4m3_quant(load_f32(X, act_dtype, (size_t)t * H + h), s_a1)];
      for (int j = 0; j < k; ++j) {
        const int e = ids[(size_t)t * k + j];
        const size_t w13_base = (size_t)e * 2 * I * H;
        for (int i = 0; i < I; ++i) {
          double g = 0.0, u = 0.0;
          for (int h = 0; h < H; ++h) {
            g += e4m3_table[((const uint8_t*)W13)[w13_base + (size_t)i * H + h]] * xq[h];
            u += e4m3_table[((const uint8_t*)W13)[w13_base + (size_t)(I + i) * H + h]] * xq[h];
          }
          g = g * (double)s_a1 * (double)w13_scale[e];
          u = u * (double)s_a1 * (double)w13_scale[e];
          A[((size_t)t * k + j) * I + i] = oracle_silu(g) * u;
        }
      }
    }
    free(xq);
  }
  double amax_a = 0.0;
  for (size_t i = 0; i < (size_t)T * k * I; ++i) if (fabs(A[i]) > amax_a) amax_a = fabs(A[i]);
  const float s_a2 = oracle_e4m3_scale((float)amax_a);
  if (act_scales_out) { act_scales_out[0] = s_a1; act_scales_out[1] = s_a2; }
#pragma omp parallel
  {
    double* aq = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
    for (int q = 0; q < n_tokens; ++q) {
      const int t = tokens ? tokens[q] : q;
      double* o = out + (size_t)q * H;
      for (int h = 0; h < H; ++h) o[h] = 0.0;
      for (int j = 0; j < k; ++j) {
        const int e = ids[(size_t)t * k + j];
        for (int i = 0; i < I; ++i)
          aq[i] = e4m3_table[oracle_e4m3_quant((float)A[((size_t)t * k + j) * I + i], s_a2)];
        const size_t w2_base = (size_t)e * H * I;
        const double wj = w[(size_t)t * k + j];
        for (int h = 0; h < H; ++h) {
          double y = 0.0;
          for (int i = 0; i < I; ++i) y += e4m3_table[((const uint8_t*)W2)[w2_base + (size_t)h * I + i]] * aq[i];
          y = y * (double)s_a2 * (double)w2_scale[e];
          o[h] += wj * y;
        }
      }
    }
    free(aq);
  }
  free(A);
  free(ids);
  free(w);
  return 0;
}

/* Thread control for timing the oracle single-threaded and on all cores. */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Inverse rotary position embedding with per-head FP8 quantisation
 * ("Mixture-of-Experts kernel engineering on Amazon SageMaker AI", section on
 * the Triton JIT: the serving stack's _fused_inv_rope_fp8_quant_per_head kernel
 * fuses rotary embedding with FP8 quantisation; the pages give no formula).
 *
 * Readings: the rotate-half pairing (element i with element i + R/2) over the
 * first R = rot_dim elements of each head vector; "inverse" is the rotation by
 * minus the position's angle; the elements from R on pass through; "per head"
 * is one dynamic scale per (token, head) vector, amax / 448 (1 when amax is 0);
 * codes of y * (1 / scale), the reciprocal taken once per vector (the practice
 * of serving stacks' FP8 quantisation kernels), by round-to-nearest-even with
 * saturation.  The cos/sin of each
 * position's R/2 angles are an input table (as a serving stack passes them).
 *
 * Precision: the kernel takes the code decisions in fp32, so this function
 * does the same arithmetic in fp32, one rounding per product, sum and
 * division, in this order (the build disables floating-point contraction).
 *
 *   x:  [T][heads][D] bf16 bit patterns     pos: [T]     cos_sin: [max_pos][R]
 *   y:  [T][heads][D] fp32 rotated values (nullable)
 *   q:  [T][heads][D] e4m3 codes            scale: [T][heads]
 * Returns -1 when a position is outside [0, max_pos).
 */
int oracle_inv_rope_fp8(const uint16_t* x, int T, int heads, int D, int R, const int32_t* pos, const float* cos_sin,
                        int max_pos, float* y, uint8_t* q, float* scale) {
  const int half = R / 2;
  for (int t = 0; t < T; ++t) {
    if (pos[t] < 0 || pos[t] >= max_pos) return -1;
    const float* c = cos_sin + (size_t)pos[t] * R;
    const float* s = c + half;
    for (int h = 0; h < heads; ++h) {
      const size_t base = ((size_t)t * heads + h) * D;
      float* v = (float*)malloc(sizeof(float) * (size_t)D);
      if (!v) return -2;
      for (int i = 0; i < half; ++i) {
        const float x1 = (float)oracle_bf16_to_f64(x[base + i]);
        const float x2 = (float)oracle_bf16_to_f64(x[base + half + i]);
        const float p11 = x1 * c[i], p22 = x2 * s[i];
        const float p21 = x2 * c[i], p12 = x1 * s[i];
        v[i] = p11 + p22;
        v[half + i] = p21 - p12;
      }
      for (int j = R; j < D; ++j) v[j] = (float)oracle_bf16_to_f64(x[base + j]);
      float amax = 0.0f;
      for (int j = 0; j < D; ++j) {
        const float a = fabsf(v[j]);
        if (a > amax) amax = a;
      }
      const float sc = oracle_e4m3_scale(amax);
      const float r = 1.0f / sc;
      scale[(size_t)t * heads + h] = sc;
      for (int j = 0; j < D; ++j) {
        const float z = v[j] * r;
        q[base + j] = oracle_f32_to_e4m3_satfinite(z);
        if (y) y[base + j] = v[j];
      }
      free(v);
    }
  }
  return 0;
}
