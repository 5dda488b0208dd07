/*
 * sv_oracle.c -- CPU oracle for the speculative-decoding verify-and-sample step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (tests, smoke check and the bench's
 * cpu_baseline/reference leg only).  Plain, single-threaded, double precision,
 * written for a reader to check against the pages by eye.  Nothing here is
 * blocked, fused or reordered for speed.
 *
 * Sources (page title, section):
 *  [A1]  "Fast Inference from Transformers via Speculative Decoding"
 *        (intuitivepapers.ai), "The loop: draft, verify in one pass, keep a
 *        prefix", Algorithm 1: walk drafts left to right, accept x_i w.p.
 *        min(1, p_i(x_i)/q_i(x_i)), stop at the first rejection, then one token
 *        from the residual or, after a clean sweep, from p_{gamma+1}.
 *  [A2]  same page, "Speculative sampling: the accept/reject rule": residual
 *        p'(x) = max(0, p(x)-q(x)) / (1-beta), beta = sum_x min(p,q)
 *        (Appendix A.1).
 *  [A3]  same page, the paragraph on the distributions being "already adjusted":
 *        temperature rescales the logits before the softmax; argmax is the
 *        one-hot limit.
 *  [B1]  "Speculative Decoding" (course notes), "The algorithm": u ~ U(0,1),
 *        accept iff u <= min(1, p/q); "Exactness": residual normaliser.
 *  [C1]  lihaoran.work essay, "What does unchanged output mean?": greedy mode
 *        keeps the prefix matching the target's own selection.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - temperature: s = z * fl32(1/T) for target and draft rows alike;
 *  - the accept comparison is "<=", with IEEE p/q (p/0 = inf accepts, 0/0 rejects);
 *  - "sample" the target's own token = Gumbel-max (the default): the argmax over
 *    the entries of positive weight of log w_v + g_v, g_v = -log(-log u_v), ties
 *    to the lowest index, with u_v from Philox4x32-10 tag 1 at the draw position
 *    (counter word 0 = v>>2, output lane v&3).  Opt-in alternative: the inverse
 *    transform, one uniform U in [0, 1) with 53 random bits (tag 1 at the draw
 *    position, counter word 0 = 0) and the smallest v, in vocabulary order, whose
 *    cumulative weight exceeds U times the total weight;
 *  - "sample" a draft token (the draft side) = Gumbel-max argmax(log w_v + g_v),
 *    g = -log(-log u), ties to the lowest index, u from Philox tag 2;
 *  - an all-zero residual (possible only by rounding) falls back to p_n;
 *  - an empty row (no finite logit) emits token 0 and sets ZERO_MASS.
 */
#include "sv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Philox4x32-10, from the SC'11 paper "Parallel random numbers: as easy as   */
/* 1, 2, 3": two 32x32->64 multiplies per round, the high halves xored with   */
/* the other two counter words and the round key, a Weyl-sequence key bump    */
/* between rounds, ten rounds.                                                */
/* ------------------------------------------------------------------------ */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void svo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

double svo_uniform(uint64_t seed, uint32_t tag, uint32_t pos, uint32_t b,
                   uint64_t round, uint32_t c0, int lane) {
  uint32_t ctr[4] = {c0, (tag << 24) | (pos & 0xFFFFFFu), b, (uint32_t)round};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  svo_philox4x32_10(ctr, key, out);
  uint32_t x = out[lane & 3];
  /* 23 random bits -> odd multiple of 2^-24: strictly inside (0, 1). */
  return (2.0 * (double)(x >> 9) + 1.0) * 0x1p-24;
}

void svo_uniform_row(uint64_t seed, uint32_t tag, uint32_t pos, uint32_t b, uint64_t round,
                     int64_t v0, int64_t n, double* out) {
  for (int64_t j = 0; j < n; ++j) {
    int64_t v = v0 + j;
    out[j] = svo_uniform(seed, tag, pos, b, round, (uint32_t)(v >> 2), (int)(v & 3));
  }
}

/* Gumbel noise for vocabulary entry v: tag 1 at the target's draw position, tag 2
 * at a draft position. */
static double gumbel_tag(uint64_t seed, uint32_t tag, uint32_t pos, uint32_t b, uint64_t round,
                         int64_t v) {
  double u = svo_uniform(seed, tag, pos, b, round, (uint32_t)(v >> 2), (int)(v & 3));
  return -log(-log(u));
}

/* The uniform of the target's own draw at position pos: counter (0, 1<<24 | pos,
 * b, round); the top 21 bits of word 0 and all 32 bits of word 1 form a 53-bit
 * integer k, and U = k 2^-53 lies in [0, 1). */
double svo_draw_uniform(uint64_t seed, uint32_t pos, uint32_t b, uint64_t round) {
  uint32_t ctr[4] = {0u, (1u << 24) | (pos & 0xFFFFFFu), b, (uint32_t)round};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  svo_philox4x32_10(ctr, key, out);
  uint64_t k = ((uint64_t)(out[0] >> 11) << 32) | (uint64_t)out[1];
  return (double)k * 0x1p-53;
}

/* ------------------------------------------------------------------------ */
/* Probability-level pieces ([A2], [B1]).                                     */
/* ------------------------------------------------------------------------ */

/* Accepted mass per token, min(p, q); returns beta = its sum. */
double svo_accept_mass(const double* p, const double* q, int64_t V, double* out_min) {
  double beta = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double m = p[v] < q[v] ? p[v] : q[v];
    if (out_min) out_min[v] = m;
    beta += m;
  }
  return beta;
}

/* Residual distribution max(0, p - q) normalised by its sum; returns the sum
 * (the rejection probability 1 - beta).  A zero sum is not normalised. */
double svo_residual(const double* p, const double* q, int64_t V, double* out_resid) {
  double mass = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double r = p[v] - q[v];
    r = r > 0.0 ? r : 0.0;
    if (out_resid) out_resid[v] = r;
    mass += r;
  }
  if (out_resid && mass > 0.0)
    for (int64_t v = 0; v < V; ++v) out_resid[v] /= mass;
  return mass;
}

/* Max-subtracted softmax; returns S = sum_v exp(s_v - max). */
double svo_softmax(const double* s, int64_t V, double* p) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v)
    if (s[v] > m) m = s[v];
  if (m == -INFINITY) { /* no finite entry */
    if (p) for (int64_t v = 0; v < V; ++v) p[v] = 0.0;
    return 0.0;
  }
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v) S += exp(s[v] - m);
  if (p) for (int64_t v = 0; v < V; ++v) p[v] = exp(s[v] - m) / S;
  return S;
}

/* ------------------------------------------------------------------------ */
/* Logit rows.                                                               */
/* ------------------------------------------------------------------------ */
static double logit_at(const void* base, int dtype, int64_t idx) {
  if (dtype == SVO_F32) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  double* s;   /* scaled logits s_v = z_v * invT          */
  double m;    /* max_v s_v                                */
  double S;    /* sum_v exp(s_v - m), 0 if no finite entry */
  double gap;  /* top-p: distance of top_p from the cumulative masses around the cut */
} row_t;

/* Descending order for qsort. */
static int cmp_desc(const void* a, const void* b) {
  const double x = *(const double*)a, y = *(const double*)b;
  return (x < y) - (x > y);
}

/* The k-th largest of the row's values that are not NaN (counting repeats);
 * -inf when the row has fewer than k of them.  `buf` holds V doubles. */
static double kth_largest(const double* s, int64_t V, int k, double* buf) {
  int64_t n = 0;
  for (int64_t v = 0; v < V; ++v)
    if (!isnan(s[v])) buf[n++] = s[v];
  if (k > n) return -INFINITY;
  qsort(buf, (size_t)n, sizeof(double), cmp_desc);
  return buf[k - 1];
}

/* Temperature, the top-k adjustment, then softmax statistics of one row ([A3]).
 * Top-k ([A3]: top-k zeroes the tail and renormalises): with top_k > 0 every
 * entry below the k-th largest scaled logit gets weight 0 (-inf); entries equal
 * to it are kept, and NaN entries are left as they are (they mark the row
 * non-finite).  `buf` holds V doubles. */
static void row_stats(row_t* r, int64_t V) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v)
    if (r->s[v] > m) m = r->s[v];
  double S = 0.0;
  if (m != -INFINITY)
    for (int64_t v = 0; v < V; ++v) S += exp(r->s[v] - m);
  r->m = m;
  r->S = S;
}

/* Top-p (nucleus; [A3]: nucleus zeroes the tail and renormalises): the
 * smallest set of largest-logit entries whose probability reaches top_p,
 * with every entry equal to the last one kept.  Groups of equal scaled logits
 * are added largest first; the cut is the first group at which the cumulative
 * probability reaches top_p.  r->gap is the distance of top_p from the
 * cumulative probabilities just before and at the cut.  Rows that are empty
 * or not finite are left as they are. */
static void nucleus(row_t* r, int64_t V, double top_p, double* buf) {
  r->gap = INFINITY;
  if (!(top_p < 1.0) || !(r->S > 0.0) || !isfinite(r->S) || !isfinite(r->m)) return;
  int64_t n = 0;
  for (int64_t v = 0; v < V; ++v)
    if (r->s[v] > -INFINITY) buf[n++] = r->s[v];
  qsort(buf, (size_t)n, sizeof(double), cmp_desc);
  double C = 0.0, prev = 0.0, tau = -INFINITY;
  for (int64_t i = 0; i < n;) {
    int64_t j = i;
    while (j < n && buf[j] == buf[i]) ++j;
    C += (double)(j - i) * exp(buf[i] - r->m) / r->S;
    if (C >= top_p) {
      tau = buf[i];
      r->gap = fmin(C - top_p, top_p - prev);
      break;
    }
    prev = C;
    i = j;
  }
  if (tau == -INFINITY) return; /* rounding left the total below top_p: keep all */
  for (int64_t v = 0; v < V; ++v)
    if (r->s[v] < tau) r->s[v] = -INFINITY;
  row_stats(r, V);
}

static void load_row(row_t* r, const void* base, int dtype, int64_t off, int64_t V, double invT,
                     int top_k, double top_p, double* buf) {
  for (int64_t v = 0; v < V; ++v) r->s[v] = logit_at(base, dtype, off + v) * invT;
  if (top_k > 0) {
    const double tau = kth_largest(r->s, V, top_k, buf);
    for (int64_t v = 0; v < V; ++v)
      if (r->s[v] < tau) r->s[v] = -INFINITY;
  }
  row_stats(r, V);
  nucleus(r, V, top_p, buf);
}

static double prob(const row_t* r, int64_t v) {
  if (!(r->S > 0.0)) return 0.0;
  return exp(r->s[v] - r->m) / r->S;
}

static int row_nonfinite(const row_t* r) { return !isfinite(r->S) || isnan(r->m) || r->m == INFINITY; }

/* Gumbel-max draw (the default sampler of the target's own token): the argmax
 * over the entries with w(v) > 0 of log w(v) + g_v, g_v the Gumbel noise of entry
 * v (tag 1 at position pos), ties to the lowest v.  Returns -1 when no weight is
 * positive.  *gap is the top-1 key minus the top-2 key (inf with one candidate),
 * the margin by which the draw was decided. */
typedef double (*weight_fn)(const void* ctx, int64_t v);

static int64_t gumbel_draw(weight_fn w, const void* ctx, int64_t V, uint64_t seed, uint32_t pos,
                           uint32_t b, uint64_t round, double* gap) {
  int64_t best = -1;
  double k1 = -INFINITY, k2 = -INFINITY;
  for (int64_t v = 0; v < V; ++v) {
    double x = w(ctx, v);
    if (!(x > 0.0) || x == INFINITY) continue;
    double key = log(x) + gumbel_tag(seed, 1u, pos, b, round, v);
    if (best < 0 || key > k1) {
      k2 = k1;
      k1 = key;
      best = v;
    } else if (key > k2) {
      k2 = key;
    }
  }
  if (gap) *gap = best < 0 ? NAN : k1 - k2;
  return best;
}

/* Inverse-transform draw: with W the sum of the weights w(v) >= 0 and
 * C_v = w(0) + ... + w(v), the smallest v with C_v > U W.  Returns -1 when no
 * weight is positive.  *gap is the distance of U W from the nearer end of the
 * chosen entry's interval [C_{v-1}, C_v) (in the weights' units).  When the
 * rounded sums leave U W at or above C_{V-1}, the last positive entry is taken
 * with gap 0. */
static int64_t inverse_cdf_draw(weight_fn w, const void* ctx, int64_t V, double U, double* gap) {
  double W = 0.0;
  int64_t last = -1;
  for (int64_t v = 0; v < V; ++v) {
    double x = w(ctx, v);
    if (x > 0.0) {
      W += x;
      last = v;
    }
  }
  if (gap) *gap = NAN;
  if (last < 0) return -1;
  const double t = U * W;
  double C = 0.0;
  for (int64_t v = 0; v <= last; ++v) {
    double x = w(ctx, v);
    if (!(x > 0.0)) continue;
    double Cn = C + x;
    if (Cn > t) {
      if (gap) *gap = fmin(t - C, Cn - t);
      return v;
    }
    C = Cn;
  }
  if (gap) *gap = 0.0;
  return last;
}

/* p(v) of a loaded row. */
static double weight_prob(const void* ctx, int64_t v) { return prob((const row_t*)ctx, v); }

typedef struct {
  const row_t* t;
  const row_t* d;
} pair_t;

/* max(0, p(v) - q(v)) with p, q the normalised target/draft probabilities ([A2]). */
static double weight_residual(const void* ctx, int64_t v) {
  const pair_t* pr = (const pair_t*)ctx;
  double r = prob(pr->t, v) - prob(pr->d, v);
  return r > 0.0 ? r : 0.0;
}

/* ------------------------------------------------------------------------ */
/* The verify step ([A1], [B1]).                                             */
/* ------------------------------------------------------------------------ */
int svo_spec_verify(const void* zt, const void* zd, const int32_t* xt,
                    int B, int gamma, int64_t V, int dtype,
                    float temperature, const float* row_temperature,
                    uint64_t seed, uint64_t round,
                    int32_t* tokens, int32_t* counts,
                    double* p_at, double* q_at, double* ratio_out, double* u_out,
                    double* beta_out, double* draw_gap, double* resid_mass,
                    uint8_t* flags) {
  return svo_spec_verify_rows(zt, zd, xt, B, gamma, V, dtype, temperature, row_temperature, seed,
                              round, tokens, counts, p_at, q_at, ratio_out, u_out, beta_out,
                              draw_gap, resid_mass, flags, 0, B);
}

int svo_spec_verify_rows(const void* zt, const void* zd, const int32_t* xt,
                         int B, int gamma, int64_t V, int dtype,
                         float temperature, const float* row_temperature,
                         uint64_t seed, uint64_t round,
                         int32_t* tokens, int32_t* counts,
                         double* p_at, double* q_at, double* ratio_out, double* u_out,
                         double* beta_out, double* draw_gap, double* resid_mass,
                         uint8_t* flags, int b_begin, int b_end) {
  return svo_spec_verify_ex(zt, zd, xt, B, gamma, V, dtype, temperature, row_temperature, seed,
                            round, tokens, counts, p_at, q_at, ratio_out, u_out, beta_out,
                            draw_gap, resid_mass, flags, b_begin, b_end, NULL);
}

int svo_spec_verify_ex(const void* zt, const void* zd, const int32_t* xt,
                       int B, int gamma, int64_t V, int dtype,
                       float temperature, const float* row_temperature,
                       uint64_t seed, uint64_t round,
                       int32_t* tokens, int32_t* counts,
                       double* p_at, double* q_at, double* ratio_out, double* u_out,
                       double* beta_out, double* draw_gap, double* resid_mass,
                       uint8_t* flags, int b_begin, int b_end, const svo_options* opt) {
  /* Lenience l (Appendix A.5 as the page summarises it): the comparison uses l q(x). */
  const double l = opt ? opt->lenience : 1.0;
  const int top_k = opt ? opt->top_k : 0;
  const double top_p = opt ? opt->top_p : 1.0;
  const int sampler = opt ? opt->sampler : SVO_SAMPLER_GUMBEL;
  if (!(l > 0.0 && l <= 1.0)) return -1;
  if (sampler != SVO_SAMPLER_GUMBEL && sampler != SVO_SAMPLER_INVERSE) return -1;
  if (top_k < 0 || !(top_p > 0.0 && top_p <= 1.0)) return -1;
  if (B < 0 || gamma < 1 || gamma > 64 || V < 1 || (dtype != SVO_F32 && dtype != SVO_BF16))
    return -1;
  if (b_begin < 0 || b_end > B || b_begin > b_end) return -1;
  if (B == 0 || b_begin == b_end) return 0;
  if (!zt || !zd || !xt || !tokens || !counts) return -1;

  const int R = 2 * gamma + 1; /* rows 0..gamma: target, gamma+1..2gamma: draft */
  row_t* rows = (row_t*)calloc((size_t)R, sizeof(row_t));
  if (!rows) return -1;
  for (int r = 0; r < R; ++r) {
    rows[r].s = (double*)malloc((size_t)V * sizeof(double));
    if (!rows[r].s) {
      for (int k = 0; k < r; ++k) free(rows[k].s);
      free(rows);
      return -1;
    }
  }
  double* kbuf = NULL; /* scratch of the top-k and top-p selections */
  if (top_k > 0 || top_p < 1.0) {
    kbuf = (double*)malloc((size_t)V * sizeof(double));
    if (!kbuf) {
      for (int r = 0; r < R; ++r) free(rows[r].s);
      free(rows);
      return -1;
    }
  }

  for (int b = b_begin; b < b_end; ++b) {
    float T = row_temperature ? row_temperature[b] : temperature;
    /* Both sides use the single-precision reciprocal of T as the scale. */
    float invT_f = 1.0f / T;
    double invT = (double)invT_f;
    uint8_t flag = 0;

    for (int i = 0; i <= gamma; ++i)
      load_row(&rows[i], zt, dtype, ((int64_t)b * (gamma + 1) + i) * V, V, invT, top_k, top_p,
               kbuf);
    for (int i = 0; i < gamma; ++i)
      load_row(&rows[gamma + 1 + i], zd, dtype, ((int64_t)b * gamma + i) * V, V, invT, top_k,
               top_p, kbuf);
    double ngap = INFINITY;
    for (int r = 0; r < R; ++r) {
      if (rows[r].m == -INFINITY) flag |= SVO_FLAG_ZERO_MASS;
      if (row_nonfinite(&rows[r])) flag |= SVO_FLAG_NONFINITE;
      ngap = fmin(ngap, rows[r].gap);
    }
    if (opt && opt->nucleus_gap) opt->nucleus_gap[b] = ngap;

    /* p(x~_i), q(x~_i) and the ratio for every draft position. */
    double P[64], Q[64], RATIO[64], U[64];
    for (int i = 0; i < gamma; ++i) {
      int32_t x = xt[(int64_t)b * gamma + i];
      const row_t* rt = &rows[i];
      const row_t* rd = &rows[gamma + 1 + i];
      if (x < 0 || (int64_t)x >= V) {
        flag |= SVO_FLAG_BAD_TOKEN;
        P[i] = 0.0;
        Q[i] = 0.0;
      } else {
        P[i] = prob(rt, x);
        Q[i] = prob(rd, x);
      }
      RATIO[i] = P[i] / (l * Q[i]); /* IEEE: p/0 = inf, 0/0 = NaN (rejects) */
      U[i] = svo_uniform(seed, 0u, (uint32_t)i, (uint32_t)b, round, 0u, 0);
      if (p_at) p_at[(int64_t)b * gamma + i] = P[i];
      if (q_at) q_at[(int64_t)b * gamma + i] = Q[i];
      if (ratio_out) ratio_out[(int64_t)b * gamma + i] = RATIO[i];
      if (u_out) u_out[(int64_t)b * gamma + i] = U[i];
    }

    /* Left-to-right test, stop at the first rejection. */
    int n = gamma;
    for (int i = 0; i < gamma; ++i) {
      if (!(Q[i] > 0.0)) flag |= SVO_FLAG_NONFINITE; /* tested position with q(x~)=0 */
      if (U[i] <= RATIO[i]) continue;
      n = i;
      break;
    }

    /* The target's own token at position n: Gumbel-max (default) or the inverse
     * transform with the uniform of position n (opt-in). */
    int64_t t;
    double gap = NAN, rmass = NAN;
    const double Ud = svo_draw_uniform(seed, (uint32_t)n, (uint32_t)b, round);
#define SVO_DRAW(wfn, ctx)                                                        \
  (sampler == SVO_SAMPLER_INVERSE ? inverse_cdf_draw((wfn), (ctx), V, Ud, &gap)   \
                                  : gumbel_draw((wfn), (ctx), V, seed, (uint32_t)n, \
                                                (uint32_t)b, round, &gap))
    if (n == gamma) {
      /* Clean sweep: bonus token from p_gamma. */
      t = SVO_DRAW(weight_prob, &rows[gamma]);
      if (t < 0) { t = 0; flag |= SVO_FLAG_ZERO_MASS; }
    } else {
      /* Rejection at n: residual max(0, p_n - q_n). */
      pair_t pr = {&rows[n], &rows[gamma + 1 + n]};
      rmass = 0.0;
      for (int64_t v = 0; v < V; ++v) rmass += weight_residual(&pr, v);
      t = SVO_DRAW(weight_residual, &pr);
      if (t < 0) {
        /* Residual empty in floating point: sample p_n itself (same noise). */
        flag |= SVO_FLAG_RESIDUAL_FALLBACK;
        t = SVO_DRAW(weight_prob, &rows[n]);
        if (t < 0) { t = 0; flag |= SVO_FLAG_ZERO_MASS; }
      }
    }
#undef SVO_DRAW

    /* Emit x~_0..x~_{n-1}, t, then -1 padding. */
    int32_t* out = tokens + (int64_t)b * (gamma + 1);
    for (int i = 0; i < n; ++i) out[i] = xt[(int64_t)b * gamma + i];
    out[n] = (int32_t)t;
    for (int i = n + 1; i <= gamma; ++i) out[i] = -1;
    counts[b] = n;

    if (beta_out) {
      for (int i = 0; i < gamma; ++i) {
        double beta = 0.0;
        for (int64_t v = 0; v < V; ++v) {
          double pv = prob(&rows[i], v), qv = prob(&rows[gamma + 1 + i], v);
          beta += pv < qv ? pv : qv;
        }
        beta_out[(int64_t)b * gamma + i] = beta;
      }
    }
    if (draw_gap) draw_gap[b] = gap;
    if (resid_mass) resid_mass[b] = rmass;
    if (flags) flags[b] = flag;
  }

  for (int r = 0; r < R; ++r) free(rows[r].s);
  free(rows);
  free(kbuf);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Greedy verify ([C1]; argmax is the one-hot limit of [A3]).  NaN counts as  */
/* -inf; ties (including an all -inf row) go to the lowest index.            */
/* ------------------------------------------------------------------------ */
int svo_spec_verify_greedy(const void* zt, const int32_t* xt, int B, int gamma,
                           int64_t V, int dtype, int32_t* tokens, int32_t* counts) {
  if (B < 0 || gamma < 1 || gamma > 64 || V < 1 || (dtype != SVO_F32 && dtype != SVO_BF16))
    return -1;
  if (B == 0) return 0;
  if (!zt || !xt || !tokens || !counts) return -1;
  int32_t tgt[65];
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i <= gamma; ++i) {
      int64_t off = ((int64_t)b * (gamma + 1) + i) * V;
      double best = -INFINITY;
      int64_t arg = 0;
      for (int64_t v = 0; v < V; ++v) {
        double z = logit_at(zt, dtype, off + v);
        if (isnan(z)) z = -INFINITY;
        if (z > best) {
          best = z;
          arg = v;
        }
      }
      tgt[i] = (int32_t)arg;
    }
    int n = gamma;
    for (int i = 0; i < gamma; ++i) {
      if (xt[(int64_t)b * gamma + i] != tgt[i]) {
        n = i;
        break;
      }
    }
    int32_t* out = tokens + (int64_t)b * (gamma + 1);
    for (int i = 0; i < n; ++i) out[i] = xt[(int64_t)b * gamma + i];
    out[n] = tgt[n];
    for (int i = n + 1; i <= gamma; ++i) out[i] = -1;
    counts[b] = n;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* LM head reference: the target pass's final projection, logits = h W.      */
/* ------------------------------------------------------------------------ */
static double bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

void svo_lmhead_logits(const uint16_t* h, const uint16_t* W, int M, int H, int64_t V,
                       const int64_t* cols, int64_t ncols, float* out) {
  int64_t nc = cols ? ncols : V;
  for (int m = 0; m < M; ++m) {
    for (int64_t j = 0; j < nc; ++j) {
      int64_t v = cols ? cols[j] : j;
      double acc = 0.0;
      for (int k = 0; k < H; ++k)
        acc += bf16_to_double(h[(int64_t)m * H + k]) * bf16_to_double(W[(int64_t)k * V + v]);
      out[(int64_t)m * nc + j] = (float)acc;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Draft sampling ([A1] step 1: x_i ~ q_i, drawn autoregressively by the     */
/* draft model; [B1] "The algorithm": x~_{t+i} ~ q(. | ...)).                */
/* ------------------------------------------------------------------------ */
int svo_draft_sample(const float* logits, int B, int64_t V, float temperature, uint64_t seed,
                     uint64_t round, int pos, int32_t* tokens, double* q_at, double* lse,
                     double* gumbel_gap) {
  if (B < 0 || V < 1 || pos < 0 || !(temperature > 0.0f) || !isfinite(temperature)) return -1;
  if (B == 0) return 0;
  if (!logits || !tokens) return -1;
  /* the single-precision reciprocal of T, as for the verify step ([A3]) */
  const float invT_f = 1.0f / temperature;
  const double invT = (double)invT_f;
  for (int b = 0; b < B; ++b) {
    const float* z = logits + (int64_t)b * V;
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
      if ((double)z[v] * invT > m) m = (double)z[v] * invT;
    double S = 0.0;
    if (m != -INFINITY)
      for (int64_t v = 0; v < V; ++v) S += exp((double)z[v] * invT - m);
    /* Gumbel-max: argmax_v s_v + g_v over the finite s_v, ties to the lowest v */
    int64_t best = -1;
    double k1 = -INFINITY, k2 = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
      const double sv = (double)z[v] * invT;
      if (!(sv > -INFINITY) || sv == INFINITY) continue;
      const double key = sv + gumbel_tag(seed, 2u, (uint32_t)pos, (uint32_t)b, round, v);
      if (best < 0 || key > k1) {
        k2 = k1;
        k1 = key;
        best = v;
      } else if (key > k2) {
        k2 = key;
      }
    }
    tokens[b] = best < 0 ? 0 : (int32_t)best;
    if (q_at) q_at[b] = (best < 0 || !(S > 0.0)) ? 0.0 : exp((double)z[best] * invT - m) / S;
    if (lse) lse[b] = m + log(S);
    if (gumbel_gap) gumbel_gap[b] = (best < 0) ? INFINITY : k1 - k2;
  }
  return 0;
}
