/*
 * gdpa_oracle.c -- plain fp64 CPU oracle for jagged attention (JFA / GDPA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link or call
 * this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (restated from "GEM Training: How Meta Doubled the
 * Efficiency of Its LLM-Scale Ads Foundation Model", the JFA and GDPA
 * paragraphs): attention over jagged (variable-length, unpadded) samples,
 * written as two matrix products with an elementwise activation between
 * them.  Softmax as the activation gives jagged flash attention (JFA);
 * SiLU or GELU in place of softmax gives generalized dot-product attention
 * (GDPA).  Rec-specific features: an additive attention bias, query and
 * key/value lengths that differ per sample, and backward passes.
 *
 * The pages give no formula, so each step below is the plain definition:
 *
 *   s_ij = scale * <q_i, k_j> + bias_h(i - j)        (i < Lq_b, j < Lkv_b)
 *          (or + B_b[h][i][j] with a dense jagged bias, see bias_value)
 *   mask_ij = (j <= i if causal) and (|i - j| < W if W > 0)
 *             and (floor(i / K) == floor(j / K) if K > 0)
 *   softmax: p_ij = exp(s_ij - M_i) / sum_{j' masked-in} exp(s_ij' - M_i)
 *            lse_i = M_i + log sum_j exp(s_ij - M_i)   (natural log)
 *   GDPA:    p_ij = act(s_ij)   (no row normalisation)
 *   masked pairs have p_ij = 0.
 *   o_i = sum_j p_ij v_j
 *
 * Backward (the chain rule applied to the lines above):
 *   dv_j  = sum_i p_ij dO_i
 *   dp_ij = <dO_i, v_j>
 *   softmax: ds_ij = p_ij (dp_ij - sum_j' p_ij' dp_ij')
 *   GDPA:    ds_ij = act'(s_ij) dp_ij
 *   dq_i  = scale * sum_j ds_ij k_j,   dk_j = scale * sum_i ds_ij q_i
 *   dbias_h[t] = sum over unmasked (i, j) of sample b with table index
 *                clamp(i - j + max_rel - 1) == t of ds_ij   (the bias enters s
 *                with weight 1; a learnable table's gradient)
 *   dense bias: its gradient is ds_ij itself, in the bias's layout
 *
 * Readings taken where the pages are silent:
 *   - SiLU(x) = x * sigmoid(x); GELU is the tanh form
 *     0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) or the exact (erf)
 *     form 0.5 x (1 + erf(x / sqrt(2))), both selectable.
 *   - The bias is a per-head relative-position table of 2*max_rel-1 entries,
 *     indexed by (i - j) + (max_rel - 1) with per-sample local positions; an
 *     index outside the table is clamped to its first or last entry.
 *   - Causal is top-left (j <= i) and needs Lq_b == Lkv_b.
 *   - Sliding-window attention (the SWA paragraph: each token attends only
 *     to nearby events, O(L * window) work): a window W > 0 keeps the pairs
 *     with |i - j| < W, so with causal a row sees its W most recent keys
 *     (itself included) and without causal the W - 1 on either side too.
 *     W = 0 means no window.  A window needs Lq_b == Lkv_b (self-attention).
 *   - Block-aligned attention (the same paragraph: fixed 64-token blocks,
 *     each query block attends only to its own key/value block, independent
 *     64 x 64 problems): with a block size K > 0 the tokens of each sample
 *     are cut into blocks of K starting at the sample's first token (the last
 *     block may be shorter) and a pair is kept only inside one block.  K = 0
 *     means no blocks.  Blocks need Lq_b == Lkv_b.
 *   - A softmax row with no masked-in key gets o = 0 and lse = -inf.
 *
 * Layouts: q/out/dq [Tq][H][d], k/v/dk/dv [Tkv][H][d], lse [H][Tq], bias
 * table [H][2*max_rel-1]; offsets int32 [B+1] with o[0] = 0, non-decreasing.
 *
 * MXFP8 (the low-precision paragraph: "end-to-end MXFP8 blockscaled MMA"):
 * the element format is OCP FP8 E4M3 (bias 7, max normal 448, no infinity),
 * rounded to nearest even and saturated at +-448; each block of 32 elements
 * shares an E8M0 scale 2^(floor(log2(amax)) - 8) as in the OCP Microscaling
 * Formats spec v1.0 (8 = exponent of E4M3's largest normal).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
  ORC_ACT_SOFTMAX = 0,
  ORC_ACT_SILU = 1,
  ORC_ACT_GELU_TANH = 2,
  ORC_ACT_IDENTITY = 3,
  ORC_ACT_GELU_ERF = 4
};

static double act_value(int act, double x) {
  switch (act) {
    case ORC_ACT_SILU:
      return x / (1.0 + exp(-x));
    case ORC_ACT_GELU_TANH: {
      const double c = sqrt(2.0 / M_PI);
      return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
    }
    case ORC_ACT_GELU_ERF:
      return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
    default:
      return x;
  }
}

static double act_deriv(int act, double x) {
  switch (act) {
    case ORC_ACT_SILU: {
      const double sg = 1.0 / (1.0 + exp(-x));
      return sg * (1.0 + x * (1.0 - sg));
    }
    case ORC_ACT_GELU_TANH: {
      const double c = sqrt(2.0 / M_PI);
      const double u = c * (x + 0.044715 * x * x * x);
      const double t = tanh(u);
      return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * c * (1.0 + 3.0 * 0.044715 * x * x);
    }
    case ORC_ACT_GELU_ERF: /* Phi(x) + x phi(x), phi the standard normal density */
      return 0.5 * (1.0 + erf(x / sqrt(2.0))) + x * exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
    default:
      return 1.0;
  }
}

static double bias_at(const double* table, int max_rel, int h, long i, long j) {
  if (table == NULL) return 0.0;
  const long width = 2L * max_rel - 1;
  long idx = (i - j) + (max_rel - 1);
  if (idx < 0) idx = 0;
  if (idx > width - 1) idx = width - 1;
  return table[(long)h * width + idx];
}

/* Dense jagged bias (the JFA paragraph's custom biases in their general
 * form): one value per (head, query, key) of each sample, sample b's
 * [H][Lq_b][Lkv_b] block starting at element doff[b] (doff[0] = 0,
 * doff[b+1] - doff[b] = H Lq_b Lkv_b).  NULL: the relative-position table. */
static double bias_value(const double* table, int max_rel, const double* dense,
                         const int64_t* doff, int b, int h, long Lq, long Lkv, long i, long j) {
  if (dense != NULL) return dense[doff[b] + ((long)h * Lq + i) * Lkv + j];
  return bias_at(table, max_rel, h, i, j);
}

static int check_dense(const double* dense, const int64_t* doff, const int32_t* qo,
                       const int32_t* ko, int B, int H) {
  if (dense == NULL) return 1;
  if (doff == NULL || doff[0] != 0) return 0;
  for (int b = 0; b < B; ++b)
    if (doff[b + 1] - doff[b] != (int64_t)H * (qo[b + 1] - qo[b]) * (ko[b + 1] - ko[b])) return 0;
  return 1;
}

static double dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* Row i of sample b, head h: fills s[j] and p[j] for j < Lkv (p = 0 when
 * masked) and returns the row's lse (softmax) or 0.  `live[j]` marks
 * masked-in pairs. */
static double row_probs(const double* q, const double* k, long qrow, long kbase, long Lkv, int H,
                        int d, int h, long i, const double* bias, int max_rel, const double* dense,
                        const int64_t* doff, int b, long Lq, int act, int causal, int window,
                        int block, double scale, double* s, double* p, unsigned char* live) {
  const double* qi = q + (qrow * H + h) * (long)d;
  long n_live = 0;
  for (long j = 0; j < Lkv; ++j) {
    int in = causal ? (j <= i) : 1;
    if (window > 0 && (j <= i - window || j >= i + window)) in = 0;
    if (block > 0 && i / block != j / block) in = 0;
    live[j] = (unsigned char)in;
    if (!live[j]) { s[j] = 0.0; p[j] = 0.0; continue; }
    ++n_live;
    const double* kj = k + ((kbase + j) * H + h) * (long)d;
    s[j] = scale * dot(qi, kj, d) + bias_value(bias, max_rel, dense, doff, b, h, Lq, Lkv, i, j);
  }
  if (act != ORC_ACT_SOFTMAX) {
    for (long j = 0; j < Lkv; ++j) p[j] = live[j] ? act_value(act, s[j]) : 0.0;
    return 0.0;
  }
  if (n_live == 0) {
    for (long j = 0; j < Lkv; ++j) p[j] = 0.0;
    return -INFINITY;
  }
  double m = -INFINITY;
  for (long j = 0; j < Lkv; ++j)
    if (live[j] && s[j] > m) m = s[j];
  double l = 0.0;
  for (long j = 0; j < Lkv; ++j) {
    p[j] = live[j] ? exp(s[j] - m) : 0.0;
    l += p[j];
  }
  for (long j = 0; j < Lkv; ++j) p[j] /= l;
  return m + log(l);
}

static int check_offsets(const int32_t* o, int B) {
  if (o[0] != 0) return 0;
  for (int b = 0; b < B; ++b)
    if (o[b + 1] < o[b]) return 0;
  return 1;
}

/* Forward.  Returns 0 on success, -1 on bad arguments. */
int oracle_fwd(const double* q, const int32_t* qo, const double* k, const double* v,
               const int32_t* ko, int B, int H, int d, const double* bias, int max_rel, int act,
               int causal, int window, int block, double scale, double* out, double* lse,
               const double* dense, const int64_t* doff) {
  if (B < 0 || H <= 0 || d <= 0 || act < 0 || act > 4) return -1;
  if (!check_offsets(qo, B) || !check_offsets(ko, B)) return -1;
  if (!check_dense(dense, doff, qo, ko, B, H)) return -1;
  if (window < 0 || block < 0) return -1;
  if (causal || window > 0 || block > 0)
    for (int b = 0; b < B; ++b)
      if (qo[b + 1] - qo[b] != ko[b + 1] - ko[b]) return -1;
  const long Tq = qo[B];
  /* Every output row is computed on its own, so the work is shared out in
   * chunks of FWD_ROWS query rows of one (sample, head); the schedule does not
   * change any row's arithmetic. */
  enum { FWD_ROWS = 64 };
  long nchunks = 0;
  for (int b = 0; b < B; ++b) nchunks += (long)H * ((qo[b + 1] - qo[b] + FWD_ROWS - 1) / FWD_ROWS);
#pragma omp parallel for schedule(dynamic, 1)
  for (long w = 0; w < nchunks; ++w) {
    long rest = w;
    int b = 0;
    for (;; ++b) {
      const long n = (long)H * ((qo[b + 1] - qo[b] + FWD_ROWS - 1) / FWD_ROWS);
      if (rest < n) break;
      rest -= n;
    }
    const long per_head = (qo[b + 1] - qo[b] + FWD_ROWS - 1) / FWD_ROWS;
    const int h = (int)(rest / per_head);
    const long i0 = (rest % per_head) * FWD_ROWS;
    const long Lq = qo[b + 1] - qo[b], Lkv = ko[b + 1] - ko[b];
    const long i1 = i0 + FWD_ROWS < Lq ? i0 + FWD_ROWS : Lq;
    const long q0 = qo[b], k0 = ko[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
    double* p = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
    unsigned char* live = (unsigned char*)malloc((size_t)(Lkv > 0 ? Lkv : 1));
    for (long i = i0; i < i1; ++i) {
      const double l = row_probs(q, k, q0 + i, k0, Lkv, H, d, h, i, bias, max_rel, dense, doff,
                                 b, Lq, act, causal, window, block, scale, s, p, live);
      double* oi = out + ((q0 + i) * H + h) * (long)d;
      for (int c = 0; c < d; ++c) oi[c] = 0.0;
      for (long j = 0; j < Lkv; ++j) {
        if (p[j] == 0.0) continue;
        const double* vj = v + ((k0 + j) * H + h) * (long)d;
        for (int c = 0; c < d; ++c) oi[c] += p[j] * vj[c];
      }
      if (lse != NULL) lse[(long)h * Tq + q0 + i] = (act == ORC_ACT_SOFTMAX) ? l : 0.0;
    }
    free(s);
    free(p);
    free(live);
  }
  return 0;
}

/* Backward.  dq must be [Tq][H][d]; dk, dv [Tkv][H][d].  All three are
 * overwritten.  dbias, if not NULL, is [H][2*max_rel-1] and overwritten with
 * the bias table's gradient.  Returns 0 on success, -1 on bad arguments. */
int oracle_bwd(const double* q, const int32_t* qo, const double* k, const double* v,
               const int32_t* ko, int B, int H, int d, const double* bias, int max_rel, int act,
               int causal, int window, int block, double scale, const double* dout, double* dq,
               double* dk, double* dv, double* dbias, const double* dense, const int64_t* doff) {
  if (B < 0 || H <= 0 || d <= 0 || act < 0 || act > 4) return -1;
  if (!check_offsets(qo, B) || !check_offsets(ko, B)) return -1;
  if (!check_dense(dense, doff, qo, ko, B, H)) return -1;
  if (window < 0 || block < 0) return -1;
  if (causal || window > 0 || block > 0)
    for (int b = 0; b < B; ++b)
      if (qo[b + 1] - qo[b] != ko[b + 1] - ko[b]) return -1;
  const long nwork = (long)B * H;
  const long width = 2L * (max_rel > 0 ? max_rel : 1) - 1;
  /* With a dense bias its gradient is ds itself, written in the bias's layout
   * (0 for masked pairs); with a table, the per-entry sums below. */
  double* ddense = (dense != NULL) ? dbias : NULL;
  if (ddense != NULL) {
    for (long t = 0; t < (long)doff[B]; ++t) ddense[t] = 0.0;
    dbias = NULL;
  }
  if (dbias != NULL)
    for (long t = 0; t < (long)H * width; ++t) dbias[t] = 0.0;
  /* per-(sample, head) partial sums of the bias gradient, added in a fixed
   * order after the parallel loop */
  double* part = dbias != NULL ? (double*)calloc((size_t)(nwork > 0 ? nwork : 1) * (size_t)width,
                                                 sizeof(double))
                               : NULL;
#pragma omp parallel for schedule(dynamic, 1)
  for (long w = 0; w < nwork; ++w) {
    const int b = (int)(w / H), h = (int)(w % H);
    const long Lq = qo[b + 1] - qo[b], Lkv = ko[b + 1] - ko[b];
    const long q0 = qo[b], k0 = ko[b];
    const size_t n = (size_t)(Lkv > 0 ? Lkv : 1);
    double* s = (double*)malloc(sizeof(double) * n);
    double* p = (double*)malloc(sizeof(double) * n);
    double* dp = (double*)malloc(sizeof(double) * n);
    unsigned char* live = (unsigned char*)malloc(n);
    for (long j = 0; j < Lkv; ++j) {
      double* dkj = dk + ((k0 + j) * H + h) * (long)d;
      double* dvj = dv + ((k0 + j) * H + h) * (long)d;
      for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
    }
    for (long i = 0; i < Lq; ++i) {
      const double* qi = q + ((q0 + i) * H + h) * (long)d;
      const double* doi = dout + ((q0 + i) * H + h) * (long)d;
      double* dqi = dq + ((q0 + i) * H + h) * (long)d;
      for (int c = 0; c < d; ++c) dqi[c] = 0.0;
      row_probs(q, k, q0 + i, k0, Lkv, H, d, h, i, bias, max_rel, dense, doff, b, Lq, act, causal,
                window, block, scale, s, p, live);
      double row_dot = 0.0; /* sum_j p_ij dp_ij (softmax only) */
      for (long j = 0; j < Lkv; ++j) {
        const double* vj = v + ((k0 + j) * H + h) * (long)d;
        dp[j] = live[j] ? dot(doi, vj, d) : 0.0;
        row_dot += p[j] * dp[j];
      }
      for (long j = 0; j < Lkv; ++j) {
        if (!live[j]) continue;
        double ds;
        if (act == ORC_ACT_SOFTMAX)
          ds = p[j] * (dp[j] - row_dot);
        else
          ds = act_deriv(act, s[j]) * dp[j];
        const double* kj = k + ((k0 + j) * H + h) * (long)d;
        double* dkj = dk + ((k0 + j) * H + h) * (long)d;
        double* dvj = dv + ((k0 + j) * H + h) * (long)d;
        for (int c = 0; c < d; ++c) {
          dqi[c] += scale * ds * kj[c];
          dkj[c] += scale * ds * qi[c];
          dvj[c] += p[j] * doi[c];
        }
        if (ddense != NULL) ddense[doff[b] + ((long)h * Lq + i) * Lkv + j] = ds;
        if (part != NULL) {
          long t = (i - j) + (max_rel - 1);
          if (t < 0) t = 0;
          if (t > width - 1) t = width - 1;
          part[w * width + t] += ds;
        }
      }
    }
    free(s);
    free(p);
    free(dp);
    free(live);
  }
  if (part != NULL) {
    for (long w = 0; w < nwork; ++w)
      for (long t = 0; t < width; ++t) dbias[(w % H) * width + t] += part[w * width + t];
    free(part);
  }
  return 0;
}

/* ------------------------------------------------------------ MXFP8 (OCP) */

/* E4M3 code for x, rounded to nearest even, saturated at +-448.  NaN input
 * gives the NaN code 0x7F.  Written from the E4M3 definition: value =
 * (-1)^s 2^(e-7) (1 + m/8) for e in 1..15 (except e=15,m=7 which is NaN),
 * and (-1)^s 2^-6 (m/8) for e = 0. */
uint8_t oracle_e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* find the binade: step between neighbours is 2^(e-10) for normals with
   * unbiased exponent e >= -6, and 2^-9 in the subnormal range. */
  int e;
  if (a < ldexp(1.0, -6)) {
    e = -6;
  } else {
    e = (int)floor(log2(a));
    /* guard against log2 rounding near powers of two */
    if (ldexp(1.0, e) > a) --e;
    if (ldexp(1.0, e + 1) <= a) ++e;
  }
  const double step = ldexp(1.0, e - 3);
  double n = a / step; /* exact: a and step are binary; quotient fits a double */
  double fl = floor(n);
  double frac = n - fl;
  double r;
  if (frac > 0.5)
    r = fl + 1.0;
  else if (frac < 0.5)
    r = fl;
  else
    r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double val = r * step;
  if (val > 448.0) val = 448.0;
  /* encode val */
  if (val == 0.0) return sign;
  int ev;
  if (val < ldexp(1.0, -6)) {
    const int m = (int)(val / ldexp(1.0, -9));
    return (uint8_t)(sign | (uint8_t)m);
  }
  ev = (int)floor(log2(val));
  if (ldexp(1.0, ev) > val) --ev;
  if (ldexp(1.0, ev + 1) <= val) ++ev;
  const int m = (int)(val / ldexp(1.0, ev - 3)) - 8;
  return (uint8_t)(sign | (uint8_t)((ev + 7) << 3) | (uint8_t)m);
}

double oracle_e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* E8M0 code of the shared scale for a block whose largest magnitude is
 * amax: 2^(floor(log2 amax) - 8), biased by 127, clamped to [0, 254]. */
uint8_t oracle_e8m0_scale(double amax) {
  if (!(amax > 0.0)) return 0;
  int e = (int)floor(log2(amax));
  if (ldexp(1.0, e) > amax) --e;
  if (ldexp(1.0, e + 1) <= amax) ++e;
  int code = e - 8 + 127;
  if (code < 0) code = 0;
  if (code > 254) code = 254;
  return (uint8_t)code;
}

uint8_t oracle_e8m0_nosat(double amax);

/* One block of n elements (stride apart): the shared scale is the OCP one,
 * 2^(floor(log2 amax) - 8), or with nosat the smallest power of two X with
 * amax / X <= 448 (no element saturates; see oracle_e8m0_nosat). */
static void quant_block(const double* x, long stride, int n, uint8_t* codes, long cstride,
                        uint8_t* scale, int nosat) {
  double amax = 0.0;
  for (int t = 0; t < n; ++t) {
    const double a = fabs(x[t * stride]);
    if (a > amax) amax = a;
  }
  const uint8_t sc = nosat ? oracle_e8m0_nosat(amax) : oracle_e8m0_scale(amax);
  *scale = sc;
  const double inv = ldexp(1.0, -(sc - 127));
  for (int t = 0; t < n; ++t) codes[t * cstride] = oracle_e4m3_encode(x[t * stride] * inv);
}

/* Q or K: blocks of 32 consecutive channels of each (token, head) row.
 * x [T][H][d] -> codes [T][H][d], scales [T][H][d/32].  d % 32 == 0. */
void oracle_quant_rows(const double* x, long T, int H, int d, int nosat, uint8_t* codes,
                       uint8_t* scales) {
  const int nb = d / 32;
#pragma omp parallel for schedule(static)
  for (long t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int g = 0; g < nb; ++g) {
        const long base = (t * H + h) * (long)d + 32L * g;
        quant_block(x + base, 1, 32, codes + base, 1, scales + (t * H + h) * (long)nb + g, nosat);
      }
}

/* V: blocks of 32 consecutive tokens of one sample (the first block starts
 * at the sample's first token; the last may be partial), per head and
 * channel.  x [T][H][d] -> codes [T][H][d]; scales [NB][H][d] where block
 * row r of sample b is NB-row blk_off[b] + r and blk_off[b] = sum over
 * b' < b of ceil(L_b' / 32). */
void oracle_quant_cols(const double* x, const int32_t* offs, int B, int H, int d, int nosat,
                       uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    long blk = 0;
    for (int bb = 0; bb < b; ++bb) blk += (offs[bb + 1] - offs[bb] + 31) / 32;
    const long L = offs[b + 1] - offs[b];
    for (long r = 0; 32 * r < L; ++r) {
      const long t0 = offs[b] + 32 * r;
      const int n = (int)((L - 32 * r) < 32 ? (L - 32 * r) : 32);
      for (int h = 0; h < H; ++h)
        for (int c = 0; c < d; ++c) {
          const long base = (t0 * H + h) * (long)d + c;
          quant_block(x + base, (long)H * d, n, codes + base, (long)H * d,
                      scales + ((blk + r) * H + h) * (long)d + c, nosat);
        }
    }
  }
}

/* ------------------------------------------------------------ MXFP8 backward
 *
 * The low-precision paragraph runs the backward pass on block-scaled MXFP8
 * products too.  The pages give no recipe, so this is the plain reading:
 * every product of the softmax backward takes the E4M3 + E8M0 version of its
 * operands quantised along that product's contraction axis, and the two
 * matrices made inside the pass, P and dS, are rounded to E4M3 in blocks of
 * 32 keys x 32 queries that share one scale (a 32 x 32 block holds a 32-
 * element block along either axis, so one rounding serves the dK product,
 * whose contraction runs over queries, and the dQ product, over keys).
 *
 *   s_ij  = scale <qd_i, kd_j> + bias_ij          qd, kd: along channels
 *           (bias_ij: the table's bias(i - j), or a dense bias's value)
 *   p_ij  = exp(s_ij - lse_i)  (0 when masked)    lse: the forward's, given
 *   dp_ij = <dOd_i, vd_j>                         dOd, vd: along channels
 *   ds_ij = p_ij (dp_ij - delta_i)                delta_i = <dO_i, O_i>, given
 *   dv_j  = sum_i P_ij dOt_i                      dOt: along tokens
 *   dk_j  = scale sum_i DS_ij qt_i                qt: along tokens
 *   dq_i  = scale sum_j DS_ij kt_j                kt: along tokens
 *
 * Masked pairs (causal, sliding window W > 0: |i - j| >= W) have p = ds = 0.
 * P and DS are p and ds rounded (round_ps = 1) or p and ds (round_ps = 0).
 * The blocks start at the sample's first key and first query.  A block's
 * scale is the smallest power of two X with amax / X <= 448 (no element
 * saturates; see oracle_e8m0_nosat).  Inputs are the decoded operand values
 * [T][H][d]; lse and delta are [H][Tq].
 */

/* E8M0 code of the smallest power of two X = 2^(code - 127) with
 * amax / X <= 448, clamped to [0, 254]; 0 for amax == 0. */
uint8_t oracle_e8m0_nosat(double amax) {
  if (!(amax > 0.0)) return 0;
  int e = (int)ceil(log2(amax / 448.0));
  /* guard against log2 rounding: the result is the least e with 448 * 2^e >= amax */
  while (ldexp(448.0, e) < amax) ++e;
  while (ldexp(448.0, e - 1) >= amax) --e;
  int code = e + 127;
  if (code < 0) code = 0;
  if (code > 254) code = 254;
  return (uint8_t)code;
}

/* Rounds m [R][C] (row-major) to E4M3 in 32 x 32 blocks from (0, 0). */
void oracle_round_blocks_2d(double* m, long R, long C) {
  for (long r0 = 0; r0 < R; r0 += 32)
    for (long c0 = 0; c0 < C; c0 += 32) {
      const long r1 = r0 + 32 < R ? r0 + 32 : R, c1 = c0 + 32 < C ? c0 + 32 : C;
      double amax = 0.0;
      for (long r = r0; r < r1; ++r)
        for (long c = c0; c < c1; ++c)
          if (fabs(m[r * C + c]) > amax) amax = fabs(m[r * C + c]);
      const int sc = oracle_e8m0_nosat(amax);
      const double x = ldexp(1.0, sc - 127);
      for (long r = r0; r < r1; ++r)
        for (long c = c0; c < c1; ++c)
          m[r * C + c] = oracle_e4m3_decode(oracle_e4m3_encode(m[r * C + c] / x)) * x;
    }
}

int oracle_bwd_mx(const double* qd, const double* qt, const double* kd, const double* kt,
                  const double* vd, const double* dod, const double* dot_t, const int32_t* qo,
                  const int32_t* ko, int B, int H, int d, const double* bias, int max_rel,
                  int causal, int window, double scale, const double* lse, const double* delta,
                  int round_ps, double* dq, double* dk, double* dv, const double* dense,
                  const int64_t* doff) {
  if (B < 0 || H <= 0 || d <= 0 || window < 0) return -1;
  if (!check_offsets(qo, B) || !check_offsets(ko, B)) return -1;
  if (!check_dense(dense, doff, qo, ko, B, H)) return -1;
  if (causal || window > 0)
    for (int b = 0; b < B; ++b)
      if (qo[b + 1] - qo[b] != ko[b + 1] - ko[b]) return -1;
  const long Tq = qo[B];
  const long nwork = (long)B * H;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long w = 0; w < nwork; ++w) {
    const int b = (int)(w / H), h = (int)(w % H);
    const long Lq = qo[b + 1] - qo[b], Lkv = ko[b + 1] - ko[b];
    const long q0 = qo[b], k0 = ko[b];
    /* P and dS as [key j][query i] */
    const size_t n = (size_t)(Lq > 0 ? Lq : 1) * (size_t)(Lkv > 0 ? Lkv : 1);
    double* P = (double*)calloc(n, sizeof(double));
    double* DS = (double*)calloc(n, sizeof(double));
    if (P == NULL || DS == NULL) {
      free(P);
      free(DS);
      bad = 1;
      continue;
    }
    for (long i = 0; i < Lq; ++i) {
      const double* qi = qd + ((q0 + i) * H + h) * (long)d;
      const double* doi = dod + ((q0 + i) * H + h) * (long)d;
      const double l = lse[(long)h * Tq + q0 + i];
      const double dl = delta[(long)h * Tq + q0 + i];
      for (long j = 0; j < Lkv; ++j) {
        if (causal && j > i) continue;
        if (window > 0 && (j <= i - window || j >= i + window)) continue;
        const double s = scale * dot(qi, kd + ((k0 + j) * H + h) * (long)d, d) +
                         bias_value(bias, max_rel, dense, doff, b, h, Lq, Lkv, i, j);
        const double p = exp(s - l);
        const double dp = dot(doi, vd + ((k0 + j) * H + h) * (long)d, d);
        P[j * Lq + i] = p;
        DS[j * Lq + i] = p * (dp - dl);
      }
    }
    if (round_ps) {
      oracle_round_blocks_2d(P, Lkv, Lq);
      oracle_round_blocks_2d(DS, Lkv, Lq);
    }
    for (long j = 0; j < Lkv; ++j) {
      double* dkj = dk + ((k0 + j) * H + h) * (long)d;
      double* dvj = dv + ((k0 + j) * H + h) * (long)d;
      for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
      for (long i = 0; i < Lq; ++i) {
        const double pp = P[j * Lq + i], ds = DS[j * Lq + i];
        if (pp == 0.0 && ds == 0.0) continue;
        const double* qti = qt + ((q0 + i) * H + h) * (long)d;
        const double* doi = dot_t + ((q0 + i) * H + h) * (long)d;
        for (int c = 0; c < d; ++c) {
          dvj[c] += pp * doi[c];
          dkj[c] += scale * ds * qti[c];
        }
      }
    }
    for (long i = 0; i < Lq; ++i) {
      double* dqi = dq + ((q0 + i) * H + h) * (long)d;
      for (int c = 0; c < d; ++c) dqi[c] = 0.0;
      for (long j = 0; j < Lkv; ++j) {
        const double ds = DS[j * Lq + i];
        if (ds == 0.0) continue;
        const double* ktj = kt + ((k0 + j) * H + h) * (long)d;
        for (int c = 0; c < d; ++c) dqi[c] += scale * ds * ktj[c];
      }
    }
    free(P);
    free(DS);
  }
  return bad ? -2 : 0;
}
