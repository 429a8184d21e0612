/*
 * CPU oracle for the NVFP4 W4A16 mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the layer computes, in fp64.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline / reference arm may load it.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (the NVFP4 MoE pages):
 *  - megamoe_rm.cu (sm121 W4A16 NVFP4 MoE forward): header comment (w13 rows
 *    0..I-1 are up and I..2I-1 gate; w2 is [H][I/2]; global scale multiplies the
 *    accumulator), route_prep (a pair's slot is its rank among earlier pairs with
 *    the same expert; expert -1 is skipped), fc1_rm epilogue (SiLU(gate)*up, h
 *    rounded to a 16-bit type; the GLM clamp of gate from above and of up to
 *    [-limit, limit] before the product), fc2_rm epilogue (global scale times routing weight
 *    times accumulator, written per (token, k) pair), combine (sum over k in k
 *    order, skipping pairs without an expert, rounded to bf16).
 *  - tilelang_kernels.py (grouped_gemm_fp4): per-expert dequantize-then-linear
 *    and the routing-weighted sum over the top-k slots.
 *  - cutlass discussion 2855: per-expert row offsets ("total tokens including
 *    expert") as the grouping of the rows.
 *
 * Readings where the pages leave a step open (all listed in the design notes):
 *  - E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}, sign in bit 3; the even K
 *    element sits in the low nibble of its byte.
 *  - E4M3: sign bit 7, exponent bits 6..3 with bias 7, mantissa bits 2..0,
 *    exponent 0 is subnormal (m/8 * 2^-6), 0x7F / 0xFF are NaN (rejected), no
 *    infinities.  Scales may be negative; they are decoded as general E4M3.
 *  - h is rounded to bf16 (round to nearest, ties to even) after SiLU(gate)*up;
 *    every other intermediate stays fp64; the layer output is rounded to bf16.
 *  - SiLU(g) = g / (1 + exp(-g)).
 *  - The SwiGLU limit L (qo_forward_hl; +infinity elsewhere, i.e. no clamp):
 *    gate' = min(gate, L), up' = min(max(up, -L), L), h = bf16(SiLU(gate') * up').
 *  - Expert ids < 0 contribute nothing; ids >= E are invalid: they are skipped
 *    like -1 and the call returns QO_WARN_BAD_ID.
 *  - Routing weights are used as given (no renormalisation); a token may name the
 *    same expert in several slots, each slot is its own pair.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define QO_OK 0
#define QO_ERR_ARG -1
#define QO_ERR_NAN_SCALE -2
#define QO_WARN_BAD_ID 1

/* E2M1: sign bit 3; magnitude code 0..7 -> {0, .5, 1, 1.5, 2, 3, 4, 6}. */
static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double qo_dec_e2m1(int code) {
  double m = kE2M1Mag[code & 7];
  return (code & 8) ? -m : m;
}

/* E4M3 ("fn" variant, the block-scale format): decoded from its bit fields. */
double qo_dec_e4m3(int b) {
  b &= 0xFF;
  int s = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int m = b & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* bf16 <-> double.  Rounding goes straight from double to bf16 (8 significant
 * bits, ties to even), never through fp32. */
double qo_bf16_to_double(uint16_t b) {
  int s = (b >> 15) & 1;
  int e = (b >> 7) & 0xFF;
  int m = b & 0x7F;
  double v;
  if (e == 0xFF) return m ? NAN : (s ? -INFINITY : INFINITY);
  if (e == 0)
    v = ldexp((double)m, -133);
  else
    v = ldexp(1.0 + (double)m / 128.0, e - 127);
  return s ? -v : v;
}

uint16_t qo_bf16_rne(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int ex;
  frexp(a, &ex);      /* a in [2^(ex-1), 2^ex) */
  int e = ex - 1;
  if (e < -126) e = -126; /* subnormal range keeps the quantum 2^-133 */
  double q = ldexp(1.0, e - 7);
  double r = rint(a / q) * q; /* default rounding mode: nearest, ties to even */
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  if (r < ldexp(1.0, -126)) return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -133)));
  int ex2;
  double f = frexp(r, &ex2); /* r = f * 2^ex2, f in [0.5, 1) */
  int E = ex2 - 1;
  uint16_t mant = (uint16_t)((f * 2.0 - 1.0) * 128.0);
  return (uint16_t)(sign | ((E + 127) << 7) | mant);
}

/*
 * Expert grouping (megamoe_rm.cu route_prep; cutlass discussion 2855 offsets).
 * ids[P] with P = M * top_k, pair index i = token * top_k + k.
 *   offsets[e]       = number of valid pairs with expert < e, offsets[E] = total
 *   sorted_pair[pos] = the pair at position pos of the expert-major, stable order
 *                      (a pair's rank within its expert = number of earlier pairs
 *                      with the same expert); entries past offsets[E] are -1
 *   pair_pos[i]      = inverse permutation, -1 for skipped pairs
 *   tiles[t]         = (expert, start position, rows <= tile_n), experts ascending,
 *                      positions ascending within an expert; *n_tiles = count
 * tiles must hold ceil(P / tile_n) + E triples.
 */
int qo_route(const int32_t* ids, int64_t P, int E, int tile_n, int32_t* offsets,
             int32_t* sorted_pair, int32_t* pair_pos, int32_t* tiles, int32_t* n_tiles) {
  if (P < 0 || E < 1 || tile_n < 1) return QO_ERR_ARG;
  int bad = 0;
  int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  int64_t* seen = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  if (!count || !seen) { free(count); free(seen); return QO_ERR_ARG; }
  for (int64_t i = 0; i < P; ++i) {
    int e = ids[i];
    if (e >= E) bad = 1;
    if (e >= 0 && e < E) count[e] += 1;
  }
  int64_t run = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = (int32_t)run;
    run += count[e];
  }
  offsets[E] = (int32_t)run;
  for (int64_t pos = 0; pos < P; ++pos) sorted_pair[pos] = -1;
  for (int64_t i = 0; i < P; ++i) {
    int e = ids[i];
    if (e < 0 || e >= E) {
      pair_pos[i] = -1;
      continue;
    }
    int64_t pos = offsets[e] + seen[e];
    seen[e] += 1;
    sorted_pair[pos] = (int32_t)i;
    pair_pos[i] = (int32_t)pos;
  }
  int32_t t = 0;
  for (int e = 0; e < E; ++e) {
    for (int64_t start = offsets[e]; start < offsets[e + 1]; start += tile_n) {
      int64_t rows = offsets[e + 1] - start;
      if (rows > tile_n) rows = tile_n;
      tiles[3 * t + 0] = e;
      tiles[3 * t + 1] = (int32_t)start;
      tiles[3 * t + 2] = (int32_t)rows;
      t += 1;
    }
  }
  *n_tiles = t;
  free(count);
  free(seen);
  return bad ? QO_WARN_BAD_ID : QO_OK;
}

/* One dequantized weight: code (nibble) times its 16-element block's E4M3 scale. */
static double wq(const uint8_t* w, const uint8_t* s, int64_t K, int64_t n, int64_t k) {
  uint8_t byte = w[n * (K / 2) + k / 2];
  int code = (k & 1) ? (byte >> 4) : (byte & 0xF);
  return qo_dec_e2m1(code) * qo_dec_e4m3(s[n * (K / 16) + k / 16]);
}

/* Adjacent bf16 bit patterns towards +infinity / -infinity (finite inputs). */
static uint16_t bf16_next_up(uint16_t b) {
  if ((b & 0x7FFF) == 0) return 0x0001;
  return (b & 0x8000) ? (uint16_t)(b - 1) : (uint16_t)(b + 1);
}
static uint16_t bf16_next_down(uint16_t b) {
  if ((b & 0x7FFF) == 0) return 0x8001;
  return (b & 0x8000) ? (uint16_t)(b + 1) : (uint16_t)(b - 1);
}

/* The two bf16 values bracketing v (lo <= v <= hi; both equal v when v is a bf16 value). */
static void bf16_bracket(double v, double* lo, double* hi) {
  uint16_t b = qo_bf16_rne(v);
  double r = qo_bf16_to_double(b);
  if (r == v) {
    *lo = *hi = r;
  } else if (r < v) {
    *lo = r;
    *hi = qo_bf16_to_double(bf16_next_up(b));
  } else {
    *hi = r;
    *lo = qo_bf16_to_double(bf16_next_down(b));
  }
}

/*
 * The layer for a subset of tokens (all of them when tokens == NULL):
 *   for each slot k of token m with expert e = ids[m][k] in [0, E):
 *     g[n]  = gs13[e] * sum_h x[m][h] * Wq13[e][n][h]        n < 2I
 *     h[i]  = bf16( silu(g[I + i]) * g[i] )                   i < I (up = rows < I)
 *     y[j]  = gs2[e] * sum_i h[i] * Wq2[e][j][i]              j < H
 *   out[m][j] = bf16( sum over k ascending of topk_w[m][k] * y_k[j] )
 * x is bf16 bits [M][H]; weights are the plain row-major NVFP4 tensors
 * w13 [E][2I][H/2], s13 [E][2I][H/16], w2 [E][H][I/2], s2 [E][H][I/16].
 * out_bf16 / out_f64 are [n_tokens][H] (out_f64 may be NULL).
 *
 * Rounding h to bf16 is a decision taken on a floating-point value; a GPU that
 * accumulates gate and up in fp32 may land on the other side of a rounding midpoint
 * when the exact value is within its rounding noise of one.  qo_forward_h accepts
 * such decisions from the caller: h_given ([n_tokens * top_k][I] bf16 bits, row
 * t * top_k + k for the t-th listed token) replaces the oracle's own rounding, after
 * each given value is checked to be a valid rounding: the bf16 rounding of some value
 * within delta of the exact silu(gate) * up.  delta is the first-order error of an
 * fp32 evaluation in which the dot product is accumulated as a tensor core does it:
 * the products x[h] * Wq[n][h] are exact, each 16-wide K slice sum S_s is rounded to
 * fp32 and added to an fp32 running sum P_s (P_s = S_0 + .. + S_s), every rounding
 * with relative error at most 2u, u = 2^-24 (so both round-to-nearest and truncation
 * are covered):
 *   e_dot  = 2u * (sum_s |S_s| + sum_s |P_s|)
 *   d_up   = |gs13| * e_dot(row i)   + u * |up|       (the global-scale product rounded)
 *   d_gate = |gs13| * e_dot(row I+i) + u * |gate|
 *   delta  = |silu(gate)| * d_up + 1.1 * (|up| + d_up) * d_gate + 8 * u * |silu(gate) * up|
 * since |SiLU(g + e) - SiLU(g)| <= 1.1 |e| (1.1 >= max |SiLU'|), the product's error is
 * at most |silu(gate)| d_up + 1.1 d_gate (|up| + d_up); the last term covers the fp32
 * SiLU and product.  h_stats
 * (may be NULL) receives {values compared, values that differ from the oracle's own
 * rounding, values that are not a valid rounding}.  h_out (may be NULL, same layout
 * as h_given) receives the h values used; rows of slots without an expert are zero.
 */
/* As qo_forward_h, with the SwiGLU limit swiglu_limit (> 0; +infinity: no clamp)
 * applied to gate and up before h (fc1_rm epilogue, GLM variant).  The clamps are
 * 1-Lipschitz, so the h_given check keeps its bound with the clamped gate and up. */
int qo_forward_hl(const uint16_t* x, const uint8_t* w13, const uint8_t* s13, const float* gs13,
                  const uint8_t* w2, const uint8_t* s2, const float* gs2, const int32_t* ids,
                  const float* topk_w, int64_t M, int64_t H, int64_t I, int E, int top_k,
                  const int64_t* tokens, int64_t n_tokens, uint16_t* out_bf16, double* out_f64,
                  int nthreads, const uint16_t* h_given, int64_t* h_stats, uint16_t* h_out,
                  double swiglu_limit) {
  if (M < 0 || H < 16 || I < 16 || H % 16 || I % 16 || E < 1 || top_k < 1) return QO_ERR_ARG;
  if (!(swiglu_limit > 0.0)) return QO_ERR_ARG; /* also rejects NaN */
  if (tokens == NULL) n_tokens = M;
  for (int64_t t = 0; t < n_tokens; ++t) {
    int64_t m = tokens ? tokens[t] : t;
    if (m < 0 || m >= M) return QO_ERR_ARG;
  }
  int bad_id = 0, nan_scale = 0;
  int64_t n_cmp = 0, n_flip = 0, n_out = 0;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(+ : n_cmp, n_flip, n_out)
  {
    double* g = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* ga = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    const double u = ldexp(1.0, -24);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_tokens; ++t) {
      int64_t m = tokens ? tokens[t] : t;
      for (int64_t j = 0; j < H; ++j) acc[j] = 0.0;
      for (int k = 0; k < top_k; ++k) {
        int e = ids[m * top_k + k];
        if (h_out)
          for (int64_t i = 0; i < I; ++i) h_out[(t * top_k + k) * I + i] = 0;
        if (e < 0) continue;
        if (e >= E) {
          bad_id = 1;
          continue;
        }
        const uint8_t* we = w13 + (int64_t)e * (2 * I) * (H / 2);
        const uint8_t* se = s13 + (int64_t)e * (2 * I) * (H / 16);
        for (int64_t n = 0; n < 2 * I; ++n) {
          double sum = 0.0, slice = 0.0, err = 0.0;
          for (int64_t hh = 0; hh < H; ++hh) {
            double term = qo_bf16_to_double(x[m * H + hh]) * wq(we, se, H, n, hh);
            sum += term;
            slice += term;
            if (hh % 16 == 15) { /* a 16-wide K slice ends: its sum and the running sum */
              err += fabs(slice) + fabs(sum);
              slice = 0.0;
            }
          }
          g[n] = (double)gs13[e] * sum;
          ga[n] = fabs((double)gs13[e]) * 2.0 * u * err;
        }
        for (int64_t i = 0; i < I; ++i) {
          double up = g[i], gate = g[I + i];
          if (gate > swiglu_limit) gate = swiglu_limit;
          if (up > swiglu_limit) up = swiglu_limit;
          if (up < -swiglu_limit) up = -swiglu_limit;
          double silu = gate / (1.0 + exp(-gate));
          double exact = silu * up;
          h[i] = qo_bf16_to_double(qo_bf16_rne(exact));
          if (h_given) {
            double given = qo_bf16_to_double(h_given[(t * top_k + k) * I + i]);
            double d_up = ga[i] + u * fabs(up), d_gate = ga[I + i] + u * fabs(gate);
            double delta = fabs(silu) * d_up + 1.1 * (fabs(up) + d_up) * d_gate +
                           8.0 * u * fabs(exact);
            double lo, hi, lo2, hi2;
            bf16_bracket(exact - delta, &lo, &hi2);
            bf16_bracket(exact + delta, &lo2, &hi);
            n_cmp += 1;
            if (given != h[i]) n_flip += 1;
            if (!(given >= lo && given <= hi)) n_out += 1;
            h[i] = given;
          }
          if (h_out) h_out[(t * top_k + k) * I + i] = qo_bf16_rne(h[i]);
        }
        const uint8_t* w2e = w2 + (int64_t)e * H * (I / 2);
        const uint8_t* s2e = s2 + (int64_t)e * H * (I / 16);
        for (int64_t j = 0; j < H; ++j) {
          double sum = 0.0;
          for (int64_t i = 0; i < I; ++i) sum += h[i] * wq(w2e, s2e, I, j, i);
          double y = (double)gs2[e] * sum;
          acc[j] += (double)topk_w[m * top_k + k] * y;
        }
      }
      for (int64_t j = 0; j < H; ++j) {
        if (isnan(acc[j])) nan_scale = 1; /* a NaN scale (or input) reached the output */
        out_bf16[t * H + j] = qo_bf16_rne(acc[j]);
        if (out_f64) out_f64[t * H + j] = acc[j];
      }
    }
    free(g);
    free(ga);
    free(h);
    free(acc);
  }
  if (h_stats) {
    h_stats[0] = n_cmp;
    h_stats[1] = n_flip;
    h_stats[2] = n_out;
  }
  if (nan_scale) return QO_ERR_NAN_SCALE;
  return bad_id ? QO_WARN_BAD_ID : QO_OK;
}

int qo_forward_h(const uint16_t* x, const uint8_t* w13, const uint8_t* s13, const float* gs13,
                 const uint8_t* w2, const uint8_t* s2, const float* gs2, const int32_t* ids,
                 const float* topk_w, int64_t M, int64_t H, int64_t I, int E, int top_k,
                 const int64_t* tokens, int64_t n_tokens, uint16_t* out_bf16, double* out_f64,
                 int nthreads, const uint16_t* h_given, int64_t* h_stats, uint16_t* h_out) {
  return qo_forward_hl(x, w13, s13, gs13, w2, s2, gs2, ids, topk_w, M, H, I, E, top_k, tokens,
                       n_tokens, out_bf16, out_f64, nthreads, h_given, h_stats, h_out, INFINITY);
}

int qo_forward(const uint16_t* x, const uint8_t* w13, const uint8_t* s13, const float* gs13,
               const uint8_t* w2, const uint8_t* s2, const float* gs2, const int32_t* ids,
               const float* topk_w, int64_t M, int64_t H, int64_t I, int E, int top_k,
               const int64_t* tokens, int64_t n_tokens, uint16_t* out_bf16, double* out_f64,
               int nthreads) {
  return qo_forward_h(x, w13, s13, gs13, w2, s2, gs2, ids, topk_w, M, H, I, E, top_k, tokens,
                      n_tokens, out_bf16, out_f64, nthreads, NULL, NULL, NULL);
}

/*
 * W4A4 variant (tilelang_kernels.py page, module docstring: the native E2M1 x UE4M3
 * block-scaled MMA, which needs the activations in NVFP4 as well).  The pages do not say
 * how activations are quantized; the reading taken is the NVFP4 encoding the workload
 * recipe gives for the weights, applied to each activation row on its own (the row's
 * values are its K dimension):
 *   g     = amax of the row / (6 * 448)            (1 when the row is all zero)
 *   scale = E4M3, round to nearest even, of (amax of the 16-block) / 6 / g
 *   code  = nearest E2M1 value of v / (scale * g), ties to the even mantissa, at most 6
 *   v'    = E2M1(code) * E4M3(scale) * g
 * x is quantized per token, h (after its bf16 rounding) per (token, slot) pair; the rest
 * of the layer is as in qo_forward.
 */

/* E4M3 byte nearest to v >= 0 (ties to even), saturating at 448. */
uint8_t qo_e4m3_rne(double v) {
  if (!(v > 0.0)) return 0;
  if (v >= 448.0) return 0x7E;
  int ex;
  frexp(v, &ex); /* v in [2^(ex-1), 2^ex) */
  int e = ex - 1;
  if (e < -6) e = -6;                 /* subnormal range: spacing 2^-9 */
  double q = ldexp(1.0, e - 3);       /* 3 mantissa bits */
  double r = rint(v / q) * q;         /* nearest, ties to even */
  if (r >= 448.0) return 0x7E;
  if (r < ldexp(1.0, -6)) return (uint8_t)(r / ldexp(1.0, -9)); /* subnormal: m * 2^-9 */
  int ex2;
  double f = frexp(r, &ex2); /* r = f * 2^ex2, f in [0.5, 1) */
  int E = ex2 - 1 + 7;
  int m = (int)((f * 2.0 - 1.0) * 8.0);
  return (uint8_t)((E << 3) | m);
}

/* E2M1 code (sign in bit 3) nearest to r, ties to the even mantissa, saturating at 6;
 * a result of -0 is +0. */
int qo_e2m1_nearest(double r) {
  double a = fabs(r);
  int best = 0;
  double bd = fabs(a - kE2M1Mag[0]);
  for (int c = 1; c < 8; ++c) {
    double d = fabs(a - kE2M1Mag[c]);
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bd = d;
    }
  }
  return (r < 0.0 && best != 0) ? (best | 8) : best;
}

/* NVFP4 encode-decode of one activation row of n values (n % 16 == 0), in place. */
void qo_nvfp4_row(double* v, int64_t n) {
  double amax = 0.0;
  for (int64_t i = 0; i < n; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  double g = amax / (6.0 * 448.0);
  if (g == 0.0) g = 1.0;
  for (int64_t b = 0; b < n; b += 16) {
    double bmax = 0.0;
    for (int64_t i = b; i < b + 16; ++i)
      if (fabs(v[i]) > bmax) bmax = fabs(v[i]);
    double sc = qo_dec_e4m3(qo_e4m3_rne(bmax / 6.0 / g));
    for (int64_t i = b; i < b + 16; ++i)
      v[i] = sc > 0.0 ? qo_dec_e2m1(qo_e2m1_nearest(v[i] / (sc * g))) * sc * g : 0.0;
  }
}

int qo_forward_w4a4(const uint16_t* x, const uint8_t* w13, const uint8_t* s13, const float* gs13,
                    const uint8_t* w2, const uint8_t* s2, const float* gs2, const int32_t* ids,
                    const float* topk_w, int64_t M, int64_t H, int64_t I, int E, int top_k,
                    const int64_t* tokens, int64_t n_tokens, uint16_t* out_bf16, double* out_f64,
                    int nthreads) {
  if (M < 0 || H < 16 || I < 16 || H % 16 || I % 16 || E < 1 || top_k < 1) return QO_ERR_ARG;
  if (tokens == NULL) n_tokens = M;
  for (int64_t t = 0; t < n_tokens; ++t) {
    int64_t m = tokens ? tokens[t] : t;
    if (m < 0 || m >= M) return QO_ERR_ARG;
  }
  int bad_id = 0, nan_scale = 0;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    double* xq = (double*)malloc(sizeof(double) * (size_t)H);
    double* g = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_tokens; ++t) {
      int64_t m = tokens ? tokens[t] : t;
      for (int64_t hh = 0; hh < H; ++hh) xq[hh] = qo_bf16_to_double(x[(size_t)m * H + hh]);
      qo_nvfp4_row(xq, H);
      for (int64_t j = 0; j < H; ++j) acc[j] = 0.0;
      for (int k = 0; k < top_k; ++k) {
        int e = ids[m * top_k + k];
        if (e < 0) {
          continue;  /* no expert in this slot */
        } else if (e >= E) {
          bad_id = 1;
          continue;
        }
        const uint8_t* we = w13 + (int64_t)e * (2 * I) * (H / 2);
        const uint8_t* se = s13 + (int64_t)e * (2 * I) * (H / 16);
        for (int64_t n = 0; n < 2 * I; ++n) {
          double sum = 0.0;
          for (int64_t hh = 0; hh < H; ++hh) sum += xq[hh] * wq(we, se, H, n, hh);
          g[n] = sum * (double)gs13[e];
        }
        for (int64_t i = 0; i < I; ++i) {
          const double upv = g[i], gatev = g[I + i];
          const double sg = gatev / (1.0 + exp(-gatev));
          h[i] = qo_bf16_to_double(qo_bf16_rne(sg * upv));
        }
        qo_nvfp4_row(h, I);
        const uint8_t* w2e = w2 + (int64_t)e * H * (I / 2);
        const uint8_t* s2e = s2 + (int64_t)e * H * (I / 16);
        for (int64_t j = 0; j < H; ++j) {
          double sum = 0.0;
          for (int64_t i = 0; i < I; ++i) sum += h[i] * wq(w2e, s2e, I, j, i);
          acc[j] += (double)topk_w[m * top_k + k] * ((double)gs2[e] * sum);
        }
      }
      for (int64_t j = 0; j < H; ++j) {
        if (isnan(acc[j])) nan_scale = 1;
        out_bf16[t * H + j] = qo_bf16_rne(acc[j]);
        if (out_f64) out_f64[t * H + j] = acc[j];
      }
    }
    free(xq);
    free(g);
    free(h);
    free(acc);
  }
  if (nan_scale) return QO_ERR_NAN_SCALE;
  return bad_id ? QO_WARN_BAD_ID : QO_OK;
}

/* Number of threads OpenMP would use by default (the host's cores). */
int qo_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
