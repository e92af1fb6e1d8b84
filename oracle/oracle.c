/*
 * CPU oracle for the batch Gumbel-max / HLG token sampler.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded C
 * restatement of what the sampler computes, written so that it can be checked
 * against the source pages by eye. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may call it; the CUDA library never does, and
 * this file shares no code, header, table or constant generator with it.
 *
 * Every floating-point step is done in double from the (exactly upcast) input
 * logits. Sources, by page title and section:
 *
 *   [GUMBEL]  "Softmax-free GPU sampling: Gumbel-max categorical sampling
 *             kernel" (lablup/mlxcel issue #900), sections Background and Task.
 *             Score = logits[i]/temperature + g_i with g_i = -log(-log u_i);
 *             the argmax of the scores is an exact softmax sample; u_i comes
 *             from a counter-based Philox stream derived from
 *             (seed, row, element, offset); greedy argmax when temperature 0.
 *   [PHILOX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *             1, 2, 3", SC'11, section 3 (the Philox round function and the
 *             Weyl key schedule) -- the published definition of Philox4x32-10.
 *   [FILTER]  The same issue, Background: rejection-based top-k / top-p on the
 *             Gumbel path is named as the follow-up work; see the reading in
 *             the section of that name below.
 *   [HLG]     "HLG sampling -- a piecewise tone curve on the logits" (mlx-bun
 *             docs/design/hlg-sampling.md), sections "The transfer function",
 *             "The pivot", "Greedy is untouched", "Temperature semantics".
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes of the repository):
 *   - Philox layout: key = (seed & 0xffffffff, seed >> 32); counter =
 *     (i >> 2, row, offset & 0xffffffff, offset >> 32); element i takes output
 *     word i & 3. One Philox call therefore serves four consecutive elements.
 *   - Uniform: u = ((r >> 9) + 0.5) * 2^-23, an open-interval value that is
 *     exact in binary32; -log(u) is evaluated as -log1p(-(1 - u)) so that the
 *     values of u next to 1 (where the winners live) keep full precision.
 *   - Tie-break: the lowest index wins among equal scores, sampled or greedy.
 *   - NaN logits are never drawn (treated like -inf); a row with no candidate
 *     returns -1; a +inf logit scores +inf (so the lowest +inf index wins);
 *     temperature <= 0 or NaN selects greedy argmax on the raw logits.
 *   - HLG: log-probs are taken from the raw logits; the tone-curve output is
 *     divided by the row temperature before the Gumbel noise is added (the
 *     pages fold temperature into the mid gain, m -> m / T, which is the same
 *     thing because the curve is m times a function of z); the default pivot is
 *     "top" with offset c; the mid branch is |z| <= w inclusive.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F16 2

/* ----------------------------------------------------------------------------
 * Philox4x32-10 [PHILOX]. The two multipliers and the two key-schedule
 * increments (the golden ratio and sqrt(3) - 1 as 32-bit fixed point) are the
 * constants the paper gives for the 4x32 variant.
 * ------------------------------------------------------------------------- */
static const uint32_t PHILOX_MUL_A = 0xD2511F53u;
static const uint32_t PHILOX_MUL_B = 0xCD9E8D57u;
static const uint32_t PHILOX_WEYL_A = 0x9E3779B9u;
static const uint32_t PHILOX_WEYL_B = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t key_in[2], const uint32_t ctr_in[4],
                          uint32_t out[4]) {
  uint32_t k0 = key_in[0], k1 = key_in[1];
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { /* key schedule: bump the key before every round but the first */
      k0 += PHILOX_WEYL_A;
      k1 += PHILOX_WEYL_B;
    }
    uint64_t pa = (uint64_t)PHILOX_MUL_A * (uint64_t)c0;
    uint64_t pb = (uint64_t)PHILOX_MUL_B * (uint64_t)c2;
    uint32_t hi_a = (uint32_t)(pa >> 32), lo_a = (uint32_t)pa;
    uint32_t hi_b = (uint32_t)(pb >> 32), lo_b = (uint32_t)pb;
    uint32_t n0 = hi_b ^ c1 ^ k0;
    uint32_t n1 = lo_b;
    uint32_t n2 = hi_a ^ c3 ^ k1;
    uint32_t n3 = lo_a;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The raw 32-bit word element i of row `row` draws at decode step `offset`. */
uint32_t oracle_stream_word(uint64_t seed, uint32_t row, uint64_t i, uint64_t offset) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {(uint32_t)(i >> 2), row, (uint32_t)offset, (uint32_t)(offset >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(key, ctr, out);
  return out[i & 3];
}

/* u in (0, 1): 23 random bits centred in their cell. */
double oracle_uniform(uint32_t r) { return ((double)(r >> 9) + 0.5) * 0x1p-23; }

/* Standard Gumbel from a uniform [GUMBEL]: g = -log(-log u). */
double oracle_gumbel(double u) {
  double neg_log_u = -log1p(-(1.0 - u));
  return -log(neg_log_u);
}

/* ----------------------------------------------------------------------------
 * Input decoding: binary32 / bfloat16 / binary16 to double, exactly.
 * ------------------------------------------------------------------------- */
static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int exponent = (h >> 10) & 0x1f;
  int mantissa = h & 0x3ff;
  double v;
  if (exponent == 0) {
    v = ldexp((double)mantissa, -24); /* subnormal: m * 2^-24 */
  } else if (exponent == 31) {
    v = mantissa ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + mantissa), exponent - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

static double decode_bf16(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

double oracle_load(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F32) {
    float f;
    memcpy(&f, (const char*)base + 4 * idx, sizeof f);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char*)base + 2 * idx, sizeof h);
  return dtype == ORACLE_BF16 ? decode_bf16(h) : decode_f16(h);
}

static int64_t elt_size(int dtype) { return dtype == ORACLE_F32 ? 4 : 2; }

/* ----------------------------------------------------------------------------
 * Greedy argmax [GUMBEL Background: "greedy argmax when temperature == 0";
 * HLG "Greedy is untouched"]: the lowest index of the largest non-NaN,
 * non-(-inf) logit; -1 if there is none.
 * ------------------------------------------------------------------------- */
static int64_t greedy_row(const void* row, int dtype, int64_t V, double* gap) {
  int64_t best = -1;
  double b1 = -INFINITY, b2 = -INFINITY;
  for (int64_t i = 0; i < V; ++i) {
    double x = oracle_load(row, dtype, i);
    if (isnan(x) || x == -INFINITY) continue;
    if (best < 0 || x > b1) {
      b2 = b1;
      b1 = x;
      best = i;
    } else if (x > b2) {
      b2 = x;
    }
  }
  if (gap) *gap = (best < 0 || b2 == -INFINITY) ? INFINITY : (b1 == b2 ? 0.0 : b1 - b2);
  return best;
}

/* Keep the best and second-best candidate scores; ties keep the lower index,
 * because indices are visited in increasing order and only a strictly larger
 * score replaces the best. */
typedef struct {
  int64_t idx;
  double s1, s2;
} top2_t;

static void top2_init(top2_t* t) {
  t->idx = -1;
  t->s1 = -INFINITY;
  t->s2 = -INFINITY;
}

static void top2_push(top2_t* t, int64_t i, double s) {
  if (s == -INFINITY || isnan(s)) return;
  if (t->idx < 0 || s > t->s1) {
    t->s2 = t->s1;
    t->s1 = s;
    t->idx = i;
  } else if (s > t->s2) {
    t->s2 = s;
  }
}

static double top2_gap(const top2_t* t) {
  if (t->idx < 0 || t->s2 == -INFINITY) return INFINITY;
  if (t->s1 == t->s2) return 0.0; /* includes a tie of two +inf scores */
  return t->s1 - t->s2;
}

/* ----------------------------------------------------------------------------
 * Plain Gumbel-max sample of one row [GUMBEL Background and Task 1]:
 * argmax_i ( x_i / T + g_i ), g_i from the element's Philox word.
 * ------------------------------------------------------------------------- */
int64_t oracle_sample_row(const void* row, int dtype, int64_t V, float temperature,
                          uint64_t seed, uint32_t row_id, uint64_t offset, double* gap,
                          double* best_score) {
  double T = (double)temperature;
  if (!(T > 0.0)) { /* greedy for T <= 0 or NaN */
    int64_t r = greedy_row(row, dtype, V, gap);
    if (best_score) *best_score = r >= 0 ? oracle_load(row, dtype, r) : -INFINITY;
    return r;
  }
  top2_t t;
  top2_init(&t);
  for (int64_t i = 0; i < V; ++i) {
    double x = oracle_load(row, dtype, i);
    if (isnan(x) || x == -INFINITY) continue; /* masked: never drawn */
    double s;
    if (x == INFINITY) {
      s = INFINITY;
    } else {
      double g = oracle_gumbel(oracle_uniform(oracle_stream_word(seed, row_id, (uint64_t)i, offset)));
      s = x / T + g;
    }
    top2_push(&t, i, s);
  }
  if (gap) *gap = top2_gap(&t);
  if (best_score) *best_score = t.s1;
  return t.idx;
}

/* Batch entry: row b uses temperature[b], seed[b], offset[b] and the row index b
 * in its Philox counter. out_gap may be NULL. */
void oracle_gumbel_argmax(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld,
                          const float* temperature, const uint64_t* seed,
                          const uint64_t* offset, int64_t* out_idx, double* out_gap) {
  for (int64_t b = 0; b < B; ++b) {
    const char* row = (const char*)logits + b * ld * elt_size(dtype);
    out_idx[b] = oracle_sample_row(row, dtype, V, temperature[b], seed[b], (uint32_t)b,
                                   offset[b], out_gap ? &out_gap[b] : NULL, NULL);
  }
}

void oracle_argmax(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld,
                   int64_t* out_idx, double* out_gap) {
  for (int64_t b = 0; b < B; ++b) {
    const char* row = (const char*)logits + b * ld * elt_size(dtype);
    out_idx[b] = greedy_row(row, dtype, V, out_gap ? &out_gap[b] : NULL);
  }
}

/* Many decode steps of one batch: step k uses offset base_offset + k for every
 * row (the statistical test draws 1e6 samples per row this way).
 * out_idx is [steps][B]. */
void oracle_gumbel_argmax_steps(const void* logits, int dtype, int64_t B, int64_t V,
                                int64_t ld, const float* temperature, const uint64_t* seed,
                                uint64_t base_offset, int64_t steps, int64_t* out_idx,
                                double* out_gap) {
  for (int64_t k = 0; k < steps; ++k) {
    for (int64_t b = 0; b < B; ++b) {
      const char* row = (const char*)logits + b * ld * elt_size(dtype);
      out_idx[k * B + b] =
          oracle_sample_row(row, dtype, V, temperature[b], seed[b], (uint32_t)b,
                            base_offset + (uint64_t)k, out_gap ? &out_gap[k * B + b] : NULL, NULL);
    }
  }
}

/* ----------------------------------------------------------------------------
 * HLG tone curve [HLG "The transfer function"]:
 *   z <  -w :  -m*w - m*beta_t*ln(1 + (-z - w)/beta_t)    (toe)
 *   |z| <= w:   m*z                                       (linear mid)
 *   z >   w :   m*w + m*beta_h*ln(1 + ( z - w)/beta_h)    (shoulder)
 * ------------------------------------------------------------------------- */
double oracle_hlg_curve(double z, double m, double w, double beta_t, double beta_h) {
  if (z < -w) return -m * w - m * beta_t * log1p((-z - w) / beta_t);
  if (z > w) return m * w + m * beta_h * log1p((z - w) / beta_h);
  return m * z;
}

#define ORACLE_PIVOT_TOP 0
#define ORACLE_PIVOT_ENTROPY 1

/* Per-row log-softmax statistics over the finite logits [HLG "The pivot": the
 * pivot is computed from the full normalised log-prob vector].
 * Returns the number of finite entries; sets *has_pinf if a +inf logit exists. */
static int64_t row_logsumexp(const void* row, int dtype, int64_t V, double* lse_out,
                             double* max_out, int* has_pinf) {
  double M = -INFINITY;
  int64_t n = 0;
  *has_pinf = 0;
  for (int64_t i = 0; i < V; ++i) {
    double x = oracle_load(row, dtype, i);
    if (x == INFINITY) *has_pinf = 1;
    if (isnan(x) || isinf(x)) continue;
    if (x > M) M = x;
    ++n;
  }
  double S = 0.0;
  for (int64_t i = 0; i < V; ++i) {
    double x = oracle_load(row, dtype, i);
    if (isnan(x) || isinf(x)) continue;
    S += exp(x - M);
  }
  *max_out = M;
  *lse_out = n ? M + log(S) : -INFINITY;
  return n;
}

/* The pivot mu of one row [HLG "The pivot"]:
 *   top     : mu = l_max - c            (l = log-softmax of the logits)
 *   entropy : mu = sum_i p_i l_i = -H   (p = softmax of the logits)
 * Returns 0 on success, -1 if the row has no finite logit. */
int oracle_hlg_pivot(const void* row, int dtype, int64_t V, int pivot_mode, double c,
                     double* lse_out, double* mu_out) {
  double lse, M;
  int has_pinf;
  int64_t n = row_logsumexp(row, dtype, V, &lse, &M, &has_pinf);
  if (n == 0) return -1;
  double mu;
  if (pivot_mode == ORACLE_PIVOT_ENTROPY) {
    double acc = 0.0;
    for (int64_t i = 0; i < V; ++i) {
      double x = oracle_load(row, dtype, i);
      if (isnan(x) || isinf(x)) continue;
      double l = x - lse;
      acc += exp(l) * l;
    }
    mu = acc;
  } else {
    double l_max = M - lse;
    mu = l_max - c;
  }
  *lse_out = lse;
  *mu_out = mu;
  return 0;
}

/* Tone-mapped log-probs of one row: out[i] = g(l_i - mu), -inf for masked
 * entries (NaN or -inf logits). Returns -1 if the row has no finite logit. */
int oracle_hlg_transform_row(const void* row, int dtype, int64_t V, double m, double w,
                             double beta_t, double beta_h, double c, int pivot_mode,
                             double* out, double* lse_out, double* mu_out) {
  double lse, mu;
  if (oracle_hlg_pivot(row, dtype, V, pivot_mode, c, &lse, &mu) != 0) return -1;
  for (int64_t i = 0; i < V; ++i) {
    double x = oracle_load(row, dtype, i);
    if (isnan(x) || x == -INFINITY) {
      out[i] = -INFINITY;
      continue;
    }
    double l = x - lse;
    double z = l - mu;
    out[i] = oracle_hlg_curve(z, m, w, beta_t, beta_h);
  }
  if (lse_out) *lse_out = lse;
  if (mu_out) *mu_out = mu;
  return 0;
}

/* HLG sample of one row: argmax_i ( g(l_i - mu) / T + g_i ) with the same Gumbel
 * stream as the plain sampler. T <= 0 or NaN: greedy on the raw logits (the
 * curve is monotone, so it cannot change the argmax). A row holding a +inf
 * logit returns its lowest +inf index (the whole softmax mass sits there). */
int64_t oracle_hlg_sample_row(const void* row, int dtype, int64_t V, float temperature,
                              uint64_t seed, uint32_t row_id, uint64_t offset, double m,
                              double w, double beta_t, double beta_h, double c,
                              int pivot_mode, double* gap, double* best_score) {
  double T = (double)temperature;
  if (!(T > 0.0)) {
    int64_t r = greedy_row(row, dtype, V, gap);
    if (best_score) *best_score = r >= 0 ? oracle_load(row, dtype, r) : -INFINITY;
    return r;
  }
  for (int64_t i = 0; i < V; ++i) {
    if (oracle_load(row, dtype, i) == INFINITY) {
      if (gap) *gap = 0.0;
      if (best_score) *best_score = INFINITY;
      return i;
    }
  }
  double lse, mu;
  top2_t t;
  top2_init(&t);
  if (oracle_hlg_pivot(row, dtype, V, pivot_mode, c, &lse, &mu) == 0) {
    for (int64_t i = 0; i < V; ++i) {
      double x = oracle_load(row, dtype, i);
      if (isnan(x) || x == -INFINITY) continue;
      double l = x - lse;
      double z = l - mu;
      double tone = oracle_hlg_curve(z, m, w, beta_t, beta_h);
      double g = oracle_gumbel(oracle_uniform(oracle_stream_word(seed, row_id, (uint64_t)i, offset)));
      top2_push(&t, i, tone / T + g);
    }
  }
  if (gap) *gap = top2_gap(&t);
  if (best_score) *best_score = t.s1;
  return t.idx;
}

/* Batch HLG entry with per-row curve parameters (arrays of length B). */
void oracle_hlg_gumbel_argmax(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld,
                              const float* temperature, const uint64_t* seed,
                              const uint64_t* offset, const double* m, const double* w,
                              const double* beta_t, const double* beta_h, const double* c,
                              const int* pivot_mode, int64_t* out_idx, double* out_gap) {
  for (int64_t b = 0; b < B; ++b) {
    const char* row = (const char*)logits + b * ld * elt_size(dtype);
    out_idx[b] = oracle_hlg_sample_row(row, dtype, V, temperature[b], seed[b], (uint32_t)b,
                                       offset[b], m[b], w[b], beta_t[b], beta_h[b], c[b],
                                       pivot_mode[b], out_gap ? &out_gap[b] : NULL, NULL);
  }
}

/* ----------------------------------------------------------------------------
 * [CATEG] The categorical path that the issue benchmarks Gumbel-max against
 * ("Softmax-free GPU sampling", Background: a normalisation pass over the
 * vocabulary, then a categorical draw; "Performance validation": baseline
 * categorical path vs Gumbel-max). Plain inverse-CDF sampling of
 * softmax(x / T) with one uniform per row:
 *   M = the largest finite logit, p_i = exp((x_i - M) / T) (0 for -inf/NaN),
 *   S = sum_i p_i, t = u * S, and the answer is the smallest i whose running
 *   sum C_i = p_0 + ... + p_i exceeds t (i.e. t lies in [C_{i-1}, C_i)).
 * The uniform u is the one the Gumbel path gives element 0 (same Philox
 * stream, same mapping). Temperature <= 0 or NaN is greedy; a row with a +inf
 * logit returns its lowest +inf index; a row with no candidate returns -1.
 *   margin (may be NULL): distance from t to the nearer end of the chosen
 *     interval, relative to S.
 *   probe >= 0: *probe_dist = distance from t to the interval of element
 *     `probe`, relative to S (0 when t lies inside it; +inf when p_probe = 0).
 * ------------------------------------------------------------------------- */
static double categ_weight(const void* row, int dtype, int64_t i, double M, double T) {
  double x = oracle_load(row, dtype, i);
  if (isnan(x) || x == -INFINITY) return 0.0;
  return exp((x - M) / T);
}

int64_t oracle_categorical_row(const void* row, int dtype, int64_t V, float temperature,
                               uint64_t seed, uint32_t row_id, uint64_t offset, int64_t probe,
                               double* probe_dist, double* margin) {
  double T = (double)temperature;
  int64_t ans = -1;
  if (probe_dist) *probe_dist = INFINITY;
  if (margin) *margin = INFINITY;
  if (!(T > 0.0)) {
    ans = greedy_row(row, dtype, V, NULL);
    if (probe_dist && probe == ans) *probe_dist = 0.0;
    return ans;
  }
  double M = -INFINITY;
  for (int64_t i = 0; i < V; ++i) {
    double x = oracle_load(row, dtype, i);
    if (x == INFINITY) { /* +inf takes all the mass: its lowest index */
      if (probe_dist && probe == i) *probe_dist = 0.0;
      return i;
    }
    if (!isnan(x) && x > M) M = x;
  }
  if (M == -INFINITY) return -1;
  double S = 0.0;
  for (int64_t i = 0; i < V; ++i) S += categ_weight(row, dtype, i, M, T);
  double u = oracle_uniform(oracle_stream_word(seed, row_id, 0, offset));
  double t = u * S;
  double C = 0.0;
  int64_t last = -1;
  for (int64_t i = 0; i < V; ++i) {
    double p = categ_weight(row, dtype, i, M, T);
    if (p == 0.0) continue;
    double lo = C;
    C += p;
    last = i;
    if (probe_dist && probe == i) *probe_dist = t < lo ? (lo - t) / S : t >= C ? (t - C) / S : 0.0;
    if (ans < 0 && t < C) {
      ans = i;
      if (margin) *margin = fmin(t - lo, C - t) / S;
    }
  }
  if (ans < 0) ans = last; /* t == S after rounding: the last element with mass */
  return ans;
}

void oracle_categorical(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld,
                        const float* temperature, const uint64_t* seed, const uint64_t* offset,
                        const int64_t* probe, int64_t* out_idx, double* out_margin,
                        double* out_probe_dist) {
  for (int64_t b = 0; b < B; ++b) {
    const char* row = (const char*)logits + b * ld * elt_size(dtype);
    out_idx[b] = oracle_categorical_row(row, dtype, V, temperature[b], seed[b], (uint32_t)b,
                                        offset[b], probe ? probe[b] : -1,
                                        out_probe_dist ? &out_probe_dist[b] : NULL,
                                        out_margin ? &out_margin[b] : NULL);
  }
}

/* ----------------------------------------------------------------------------
 * [FILTER] Top-k / top-p (nucleus) sampling on the Gumbel path. The issue
 * names "rejection-based top-k/top-p" on Gumbel-max as its follow-up without
 * specifying it. Reading:
 *   - the candidates (logits that are neither NaN nor -inf) are ordered by
 *     logit, larger first, equal logits by lower index;
 *   - the filter set K is the first r of that order, r = min(r_k, r_p):
 *       r_k = top_k when top_k >= 1 (at most the number of candidates), else
 *             every candidate;
 *       r_p = the smallest r whose softmax(x / T) mass reaches top_p * S
 *             (S = the total mass) when top_p < 1; r_p = 1 when top_p <= 0;
 *             every candidate when top_p >= 1 or NaN. A row with +inf logits
 *             gives each +inf entry mass 1 and every other entry 0;
 *   - the sample is the Gumbel-max over K alone, with the same per-element
 *     noise: argmax over i in K of x_i / T + g_i, lowest index on ties. The
 *     Gumbel-max property holds on any subset, so this is an exact draw of
 *     softmax(x / T) restricted to K.
 * "Rejection": the unrestricted Gumbel-max draw is a proposal; when it lies
 * in K it is also the argmax over K (the maximum over a superset that falls in
 * the subset), so it is kept, and only otherwise is K needed. Both give the
 * index defined above, which is what this function computes directly: a
 * library sort of the candidates, the prefix, then the restricted argmax.
 * Temperature <= 0 or NaN: greedy argmax (the filters keep the top element).
 * Outputs: gap = the top-two score gap within K (as oracle_sample_row);
 * edge = how far top_p * S (relative to S) may move before the answer
 * changes: down to the mass of the candidates before the winner (the winner
 * leaves K; never for the first candidate, which K always keeps), or up to the mass before the first later candidate, within r_k,
 * whose score beats the winner's (it joins K); +inf when the nucleus does
 * not decide K (top_p inactive, or r_k < r_p).
 * ------------------------------------------------------------------------- */
typedef struct {
  int64_t idx;
  double x;
} filt_cand_t;

static int filt_order(const void* a, const void* b) {
  const filt_cand_t* p = (const filt_cand_t*)a;
  const filt_cand_t* q = (const filt_cand_t*)b;
  if (p->x > q->x) return -1;
  if (p->x < q->x) return 1;
  return p->idx < q->idx ? -1 : (p->idx > q->idx ? 1 : 0);
}

int64_t oracle_filtered_sample_row(const void* row, int dtype, int64_t V, float temperature,
                                   uint64_t seed, uint32_t row_id, uint64_t offset,
                                   int32_t top_k, float top_p, double* gap, double* edge) {
  double T = (double)temperature;
  if (edge) *edge = INFINITY;
  if (!(T > 0.0)) return greedy_row(row, dtype, V, gap);
  filt_cand_t* c = (filt_cand_t*)malloc((size_t)(V > 0 ? V : 1) * sizeof(filt_cand_t));
  int64_t n = 0, n_inf = 0;
  double M = -INFINITY;
  for (int64_t i = 0; i < V; ++i) {
    double x = oracle_load(row, dtype, i);
    if (isnan(x) || x == -INFINITY) continue;
    c[n].idx = i;
    c[n].x = x;
    ++n;
    if (x == INFINITY) ++n_inf;
    if (x > M) M = x;
  }
  if (n == 0) {
    free(c);
    if (gap) *gap = INFINITY;
    return -1;
  }
  qsort(c, (size_t)n, sizeof(filt_cand_t), filt_order);
  int64_t r_k = (top_k >= 1 && (int64_t)top_k < n) ? (int64_t)top_k : n;
  int64_t r_p = n;
  double p = (double)top_p;
  if (p <= 0.0) {
    r_p = 1;
  } else if (p < 1.0) {
    double S = 0.0;
    for (int64_t j = 0; j < n; ++j)
      S += n_inf ? (c[j].x == INFINITY ? 1.0 : 0.0) : exp((c[j].x - M) / T);
    double cum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      cum += n_inf ? (c[j].x == INFINITY ? 1.0 : 0.0) : exp((c[j].x - M) / T);
      if (cum >= p * S) {
        r_p = j + 1;
        break;
      }
    }
  }
  int64_t r = r_k < r_p ? r_k : r_p;
  /* Scores of the candidates in order, as far as the answer needs them: K,
   * and, when the nucleus decides K and the edge is wanted, the candidates a
   * larger top_p could add (up to r_k). */
  int nucleus = p > 0.0 && p < 1.0 && r_p <= r_k;
  int64_t limit = (edge && nucleus) ? r_k : r; /* >= r >= 1 */
  double* sc = (double*)malloc((size_t)limit * sizeof(double));
  for (int64_t j = 0; j < limit; ++j) {
    double x = c[j].x;
    sc[j] = x == INFINITY ? INFINITY
                          : x / T + oracle_gumbel(oracle_uniform(oracle_stream_word(
                                        seed, row_id, (uint64_t)c[j].idx, offset)));
  }
  /* The argmax over K (larger score, then lower index) and the top-two gap. */
  int64_t best = 0;
  double s1 = limit > 0 ? sc[0] : -INFINITY, s2 = -INFINITY;
  for (int64_t j = 1; j < r; ++j) {
    if (sc[j] > s1 || (sc[j] == s1 && c[j].idx < c[best].idx)) {
      s2 = s1;
      s1 = sc[j];
      best = j;
    } else if (sc[j] > s2) {
      s2 = sc[j];
    }
  }
  if (gap) *gap = (r < 2 || s2 == -INFINITY) ? INFINITY : (s1 == s2 ? 0.0 : s1 - s2);
  if (edge && nucleus) {
    /* How far top_p * S may move before the answer changes: down to the
     * mass before the winner (it leaves K), or up to the mass before the
     * first later candidate that would beat it (it joins K). */
    double S = 0.0, cum = 0.0, before_best = 0.0, e = INFINITY;
    for (int64_t j = 0; j < n; ++j)
      S += n_inf ? (c[j].x == INFINITY ? 1.0 : 0.0) : exp((c[j].x - M) / T);
    for (int64_t j = 0; j < limit; ++j) {
      if (j == best) before_best = cum;
      if (j >= r && (sc[j] > s1 || (sc[j] == s1 && c[j].idx < c[best].idx))) {
        e = (cum - p * S) / S;
        break;
      }
      cum += n_inf ? (c[j].x == INFINITY ? 1.0 : 0.0) : exp((c[j].x - M) / T);
    }
    /* the first candidate never leaves K (every filter keeps it) */
    *edge = best > 0 ? fmin(e, (p * S - before_best) / S) : e;
  }
  int64_t ans = c[best].idx;
  free(sc);
  free(c);
  return ans;
}

void oracle_filtered_gumbel_argmax(const void* logits, int dtype, int64_t B, int64_t V,
                                   int64_t ld, const float* temperature, const uint64_t* seed,
                                   const uint64_t* offset, const int32_t* top_k,
                                   const float* top_p, int64_t* out_idx, double* out_gap,
                                   double* out_edge) {
  for (int64_t b = 0; b < B; ++b) {
    const char* row = (const char*)logits + b * ld * elt_size(dtype);
    out_idx[b] = oracle_filtered_sample_row(
        row, dtype, V, temperature[b], seed[b], (uint32_t)b, offset[b], top_k ? top_k[b] : 0,
        top_p ? top_p[b] : 1.0f, out_gap ? &out_gap[b] : NULL, out_edge ? &out_edge[b] : NULL);
  }
}

/* Many decode steps of one filtered batch (offset base_offset + k for every
 * row at step k); out_idx is [steps][B]. */
void oracle_filtered_steps(const void* logits, int dtype, int64_t B, int64_t V, int64_t ld,
                           const float* temperature, const uint64_t* seed, uint64_t base_offset,
                           int64_t steps, const int32_t* top_k, const float* top_p,
                           int64_t* out_idx) {
  for (int64_t k = 0; k < steps; ++k)
    for (int64_t b = 0; b < B; ++b) {
      const char* row = (const char*)logits + b * ld * elt_size(dtype);
      out_idx[k * B + b] = oracle_filtered_sample_row(
          row, dtype, V, temperature[b], seed[b], (uint32_t)b, base_offset + (uint64_t)k,
          top_k ? top_k[b] : 0, top_p ? top_p[b] : 1.0f, NULL, NULL);
    }
}

/* ----------------------------------------------------------------------------
 * Batched conveniences for the tests: plain loops over the functions above.
 * ------------------------------------------------------------------------- */
void oracle_philox_blocks(uint32_t key0, uint32_t key1, const uint32_t* ctrs, int64_t n,
                          uint32_t* out) {
  uint32_t key[2] = {key0, key1};
  for (int64_t j = 0; j < n; ++j) oracle_philox4x32_10(key, ctrs + 4 * j, out + 4 * j);
}

void oracle_stream_words(uint64_t seed, uint32_t row, uint64_t offset, int64_t i0, int64_t n,
                         uint32_t* out) {
  for (int64_t j = 0; j < n; ++j) out[j] = oracle_stream_word(seed, row, (uint64_t)(i0 + j), offset);
}

void oracle_gumbel_of_words(const uint32_t* words, int64_t n, double* out) {
  for (int64_t j = 0; j < n; ++j) out[j] = oracle_gumbel(oracle_uniform(words[j]));
}

void oracle_uniform_of_words(const uint32_t* words, int64_t n, double* out) {
  for (int64_t j = 0; j < n; ++j) out[j] = oracle_uniform(words[j]);
}

void oracle_hlg_curve_many(const double* z, int64_t n, double m, double w, double beta_t,
                           double beta_h, double* out) {
  for (int64_t j = 0; j < n; ++j) out[j] = oracle_hlg_curve(z[j], m, w, beta_t, beta_h);
}

void oracle_decode(const void* base, int dtype, int64_t n, double* out) {
  for (int64_t j = 0; j < n; ++j) out[j] = oracle_load(base, dtype, j);
}
