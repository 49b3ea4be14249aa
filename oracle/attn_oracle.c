/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct fp64 CPU attention forward.  It exists to
 * check the CUDA path; nothing in the library calls it, links it or shares
 * code with it.  Only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg load it.
 *
 * What it computes (the plain definition, no tiling, no online rescaling):
 *
 *   for every sequence s, query head h, query row i of s:
 *     kv      = floor(h / (Hq / Hkv))                 grouped-query head map
 *     p       = i + Lk(s) - Lq(s)                      the row's key position
 *                                                       (queries are the last
 *                                                       Lq(s) positions)
 *     valid   = { j : 0 <= j < Lk(s) }  and, if causal, j <= p
 *     s_ij    = scale * sum_t q[i,h,t] * k[j,kv,t]     (fp64, inputs widened
 *                                                       exactly from bf16)
 *     m_i     = max_{j in valid} s_ij
 *     l_i     = sum_{j in valid} exp(s_ij - m_i)
 *     o[i,h,:]= sum_{j in valid} exp(s_ij - m_i) * v[j,kv,:] / l_i
 *     lse[i,h]= m_i + ln(l_i)
 *
 * Score and mask variants (oracle_attn_fwd_var; all off by default):
 *
 *     window  : valid additionally requires p - wl <= j <= p + wr (wl, wr >= 0;
 *               a negative bound is unbounded; causal makes wr = 0)
 *     soft cap: s_ij <- cap * tanh(s_ij / cap)                 (cap > 0)
 *     ALiBi   : s_ij <- s_ij - slope[h] * |p - j|              (after the cap)
 *
 *   and m, l, o, lse as above over the modified scores and the valid keys.
 *
 * Sources:
 *  - tang (muni.works/research/tang), section 2.2 "Comprehensions and
 *    monoids" and section 2.3 "Rewrites" (stabilize_softmax): attention is
 *    the score contraction followed by max, sum of exponentials and the
 *    weighted value sum over the same scores; the fused online form is
 *    equal to this two-pass form (section 6, the Lean theorem that online
 *    softmax equals two-pass softmax).  So the oracle is the two-pass form.
 *  - tang, section 2.1 "Views": grouped-query attention splits the query
 *    head into (kv head, group); read here as contiguous groups.
 *  - tang, section 2.4, Table 1 row "logsumexp": the per-row LSE output,
 *    read here as the natural logarithm m + ln(l).
 *  - tang, section 4 "Precision is a schedule": an f64 evaluator is the
 *    reference; the optional round_p switch mimics its emulated mode for
 *    one value only (P rounded to bf16, round-to-nearest-even, before the
 *    P.V product), as a diagnostic.
 *  - TileLang explainer (ai.thesatyajit.com/articles/tilelang), section
 *    "FlashAttention, in tiles": the per-block loop casts P to the input
 *    type before the P.V product; that is what round_p imitates.
 *  - tang, section 2.3 (the variant lab) and section 7.3, "Attention variants
 *    against FlexAttention and FA2": soft cap, ALiBi and a sliding window of
 *    128 change only the score or the mask, not the monoid.  The pages print
 *    no formulas for them; the readings above are the common ones (cap
 *    applied to the scaled score, a linear distance penalty per head, a
 *    window of keys around the query row).
 *
 * Rows with no valid key cannot occur when causal rows see themselves; if
 * one is requested anyway it gets o = 0 and lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bits -> double, exactly (bf16 is the top half of an IEEE binary32). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* double -> the nearest bf16 value (ties to the even significand), returned
 * as a double.  One rounding, taken from the double itself (going through
 * float first would round twice, which can settle a near-tie the wrong way).
 * bf16 keeps 8 significant bits: in the binade [2^(e-1), 2^e) its values are
 * the multiples of 2^(e-1-7); below 2^-126 (subnormals) the multiples of
 * 2^-133.  Scaling x by a power of two is exact, and rint() rounds to the
 * nearest integer with ties to even (the default rounding mode), so the
 * scaled value rounds exactly as the definition asks; a result of 2^8 times
 * the spacing is the next binade's first value, which is right too.  Used
 * only by the round_p diagnostic; x is finite and below the largest bf16. */
static double round_to_bf16(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  const double ax = fabs(x);
  int e;
  (void)frexp(ax, &e);               /* ax = f * 2^e with f in [0.5, 1) */
  int spacing_exp = (e - 1) - 7;
  if (spacing_exp < -133) spacing_exp = -133;
  const double y = ldexp(rint(ldexp(ax, -spacing_exp)), spacing_exp);
  return x < 0.0 ? -y : y;
}

/* Test hook for the rounding above: y[i] = round_to_bf16(x[i]). */
void oracle_round_bf16(const double *x, double *y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = round_to_bf16(x[i]);
}

/*
 * One query row against the keys of its sequence.
 *   qrow : pointer to q[i, h, 0]            (bf16 bits, d values)
 *   kbase: pointer to k[k_start, kv, 0]     (row stride kstride elements)
 *   vbase: pointer to v[k_start, kv, 0]
 *   i    : the row's key position (its index among the keys)
 *   jlo, jhi: the visible keys jlo .. jhi (none if jhi < jlo)
 *   cap  : soft cap (0: none); slope: ALiBi slope of the head (0: none)
 *   scores: scratch of at least jhi - jlo + 1 doubles
 *   out: d doubles; *lse_out: one double
 */
static void one_row(const uint16_t *qrow, const uint16_t *kbase,
                    const uint16_t *vbase, int64_t kstride, int64_t i,
                    int64_t jlo, int64_t jhi, int d, double scale, double cap,
                    double slope, int round_p, double *scores, double *out,
                    double *lse_out) {
  for (int t = 0; t < d; ++t) out[t] = 0.0;
  const int64_t nvalid = jhi - jlo + 1;
  if (nvalid <= 0) {
    *lse_out = -INFINITY;
    return;
  }
  /* pass 0: the score row (keys jlo + n) */
  for (int64_t n = 0; n < nvalid; ++n) {
    const int64_t j = jlo + n;
    const uint16_t *krow = kbase + j * kstride;
    double acc = 0.0;
    for (int t = 0; t < d; ++t) acc += bf16_to_double(qrow[t]) * bf16_to_double(krow[t]);
    double sc = scale * acc;
    if (cap > 0.0) sc = cap * tanh(sc / cap);
    sc -= slope * (double)(i > j ? i - j : j - i);
    scores[n] = sc;
  }
  /* pass 1: the row maximum */
  double m = scores[0];
  for (int64_t n = 1; n < nvalid; ++n)
    if (scores[n] > m) m = scores[n];
  /* pass 2: the sum of exponentials and the weighted value sum */
  double l = 0.0;
  for (int64_t n = 0; n < nvalid; ++n) {
    double p = exp(scores[n] - m);
    l += p;
    double pw = round_p ? round_to_bf16(p) : p;
    const uint16_t *vrow = vbase + (jlo + n) * kstride;
    for (int t = 0; t < d; ++t) out[t] += pw * bf16_to_double(vrow[t]);
  }
  for (int t = 0; t < d; ++t) out[t] /= l;
  *lse_out = m + log(l);
}

/*
 * oracle_attn_fwd
 *
 * q: [*, Hq, d] bf16 bits; k, v: [*, Hkv, d] bf16 bits (token rows packed;
 * row r of sequence s is token q_start[s] + r, resp. k_start[s] + r).
 * nseq sequences; sequence s has q_len[s] query rows and k_len[s] keys.
 * causal requires q_len[s] <= k_len[s]; key j is visible from row i iff
 * j <= i + k_len[s] - q_len[s] (the queries are the sequence's last q_len[s]
 * positions: equal lengths give j <= i).
 *
 * If nsel < 0, every row is computed:
 *   o  [(q_start[s] + i) * Hq + h) * d + t]
 *   lse[(q_start[s] + i) * Hq + h]
 * Otherwise sel holds nsel triples (s, h, i) and the results go to
 *   o[n * d + t], lse[n]  for triple n.
 *
 * nthreads <= 0 uses the OpenMP default.  Returns 0, or a negative code on
 * invalid arguments (nothing is written then).
 *
 * oracle_attn_fwd_var adds the variants: window bounds wl, wr (negative:
 * unbounded), soft cap (0: none) and ALiBi slopes (Hq values, or NULL).
 */
int oracle_attn_fwd_var(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        double *o, double *lse, int nseq, const int64_t *q_start,
                        const int64_t *q_len, const int64_t *k_start,
                        const int64_t *k_len, int Hq, int Hkv, int d, double scale,
                        int causal, int64_t wl, int64_t wr, double cap,
                        const double *slopes, int round_p, int64_t nsel,
                        const int32_t *sel, int nthreads) {
  if (nseq < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return -1;
  if (!(cap >= 0.0)) return -6;
  int64_t kmax = 0;
  for (int s = 0; s < nseq; ++s) {
    if (q_len[s] < 0 || k_len[s] < 0) return -2;
    if (causal && q_len[s] > k_len[s]) return -3;
    if (k_len[s] > kmax) kmax = k_len[s];
  }
  const int group = Hq / Hkv;
  const int64_t qstride = (int64_t)Hq * d;  /* elements between token rows */
  const int64_t kstride = (int64_t)Hkv * d;

  /* the list of (s, h, i) jobs */
  int64_t njobs = 0;
  int32_t *jobs = NULL;
  if (nsel >= 0) {
    njobs = nsel;
    for (int64_t n = 0; n < nsel; ++n) {
      int32_t s = sel[3 * n], h = sel[3 * n + 1], i = sel[3 * n + 2];
      if (s < 0 || s >= nseq || h < 0 || h >= Hq || i < 0 || i >= q_len[s]) return -4;
    }
  } else {
    for (int s = 0; s < nseq; ++s) njobs += q_len[s] * (int64_t)Hq;
    jobs = (int32_t *)malloc(sizeof(int32_t) * 3 * (size_t)(njobs > 0 ? njobs : 1));
    if (!jobs) return -5;
    int64_t n = 0;
    for (int s = 0; s < nseq; ++s)
      for (int64_t i = 0; i < q_len[s]; ++i)
        for (int h = 0; h < Hq; ++h) {
          jobs[3 * n] = s;
          jobs[3 * n + 1] = h;
          jobs[3 * n + 2] = (int32_t)i;
          ++n;
        }
  }
  const int32_t *list = (nsel >= 0) ? sel : jobs;

#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif

  int failed = 0;
#pragma omp parallel
  {
    double *scores = (double *)malloc(sizeof(double) * (size_t)(kmax > 0 ? kmax : 1));
    if (!scores) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t n = 0; n < njobs; ++n) {
        int s = list[3 * n], h = list[3 * n + 1];
        int64_t i = list[3 * n + 2];
        int kv = h / group;
        const int64_t pos = i + k_len[s] - q_len[s];       /* the row's key position */
        int64_t jhi = causal ? pos : k_len[s] - 1;         /* visible keys jlo..jhi */
        if (!causal && wr >= 0 && pos + wr < jhi) jhi = pos + wr;
        if (jhi > k_len[s] - 1) jhi = k_len[s] - 1;
        int64_t jlo = (wl >= 0 && pos - wl > 0) ? pos - wl : 0;
        const uint16_t *qrow = q + (q_start[s] + i) * qstride + (int64_t)h * d;
        const uint16_t *kb = k + k_start[s] * kstride + (int64_t)kv * d;
        const uint16_t *vb = v + k_start[s] * kstride + (int64_t)kv * d;
        double *orow;
        double *lrow;
        if (nsel >= 0) {
          orow = o + n * d;
          lrow = lse + n;
        } else {
          int64_t r = (q_start[s] + i) * Hq + h;
          orow = o + r * d;
          lrow = lse + r;
        }
        one_row(qrow, kb, vb, kstride, pos, jlo, jhi, d, scale, cap,
                slopes ? slopes[h] : 0.0, round_p, scores, orow, lrow);
      }
      free(scores);
    }
  }
  free(jobs);
  return failed ? -5 : 0;
}

/* The plain definition: no window, soft cap or ALiBi. */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    double *o, double *lse, int nseq, const int64_t *q_start,
                    const int64_t *q_len, const int64_t *k_start,
                    const int64_t *k_len, int Hq, int Hkv, int d, double scale,
                    int causal, int round_p, int64_t nsel, const int32_t *sel,
                    int nthreads) {
  return oracle_attn_fwd_var(q, k, v, o, lse, nseq, q_start, q_len, k_start, k_len, Hq,
                             Hkv, d, scale, causal, -1, -1, 0.0, NULL, round_p, nsel,
                             sel, nthreads);
}

/* The number of threads an OpenMP region would use (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * oracle_attn_bwd -- gradients of attention (fixed or packed batches; query
 * and key lengths equal per sequence), fp64, from the plain definition:
 * with P the softmax rows of the forward (masked keys excluded) and dO the
 * output gradient, for every sequence s, head h (kv = h / group) and row i:
 *
 *     dP_ij = dO_i . v_j                      D_i = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - D_i)               (the softmax Jacobian)
 *     dQ_i  = scale sum_j dS_ij k_j
 *     dK_j += scale dS_ij q_i                  (summed over rows and the
 *     dV_j += P_ij dO_i                         group's query heads)
 *
 * Source: tang, section 3 "Gradients are comprehensions": the gradient of
 * the attention comprehension is again a set of contractions over the same
 * scores (the flash backward identity of section 6 is D_i = sum_j P_ij dP_ij
 * = dO_i . O_i).  Jobs are (sequence, kv head); dq, dk, dv are written in the
 * input layouts (token rows x heads x d).  Returns 0 or a negative code.
 */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const uint16_t *dout, double *dq, double *dk, double *dv, int nseq,
                    const int64_t *start, const int64_t *len, int Hq, int Hkv, int d,
                    double scale, int causal, int nthreads) {
  if (nseq < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return -1;
  int64_t lmax = 0;
  for (int s = 0; s < nseq; ++s) {
    if (len[s] < 0) return -2;
    if (len[s] > lmax) lmax = len[s];
  }
  const int group = Hq / Hkv;
  const int64_t qstride = (int64_t)Hq * d, kstride = (int64_t)Hkv * d;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel
  {
    double *p = (double *)malloc(sizeof(double) * (size_t)(lmax > 0 ? lmax : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(lmax > 0 ? lmax : 1));
    if (!p || !dp) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t job = 0; job < (int64_t)nseq * Hkv; ++job) {
        const int s = (int)(job / Hkv), kv = (int)(job % Hkv);
        const int64_t L = len[s], r0 = start[s];
        for (int64_t j = 0; j < L; ++j)
          for (int t = 0; t < d; ++t) {
            dk[((r0 + j) * Hkv + kv) * d + t] = 0.0;
            dv[((r0 + j) * Hkv + kv) * d + t] = 0.0;
          }
        for (int g = 0; g < group; ++g) {
          const int h = kv * group + g;
          for (int64_t i = 0; i < L; ++i) {
            const uint16_t *qi = q + (r0 + i) * qstride + (int64_t)h * d;
            const uint16_t *doi = dout + (r0 + i) * qstride + (int64_t)h * d;
            const int64_t n = causal ? i + 1 : L;   /* visible keys 0 .. n-1 */
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
              const uint16_t *kj = k + (r0 + j) * kstride + (int64_t)kv * d;
              double acc = 0.0;
              for (int t = 0; t < d; ++t) acc += bf16_to_double(qi[t]) * bf16_to_double(kj[t]);
              p[j] = scale * acc;
              if (p[j] > m) m = p[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) {
              p[j] = exp(p[j] - m);
              l += p[j];
            }
            double D = 0.0;
            for (int64_t j = 0; j < n; ++j) {
              p[j] /= l;
              const uint16_t *vj = v + (r0 + j) * kstride + (int64_t)kv * d;
              double acc = 0.0;
              for (int t = 0; t < d; ++t) acc += bf16_to_double(doi[t]) * bf16_to_double(vj[t]);
              dp[j] = acc;
              D += p[j] * acc;
            }
            double *dqi = dq + ((r0 + i) * Hq + h) * d;
            for (int t = 0; t < d; ++t) dqi[t] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
              const double ds = p[j] * (dp[j] - D);
              const uint16_t *kj = k + (r0 + j) * kstride + (int64_t)kv * d;
              double *dkj = dk + ((r0 + j) * Hkv + kv) * d;
              double *dvj = dv + ((r0 + j) * Hkv + kv) * d;
              for (int t = 0; t < d; ++t) {
                dqi[t] += scale * ds * bf16_to_double(kj[t]);
                dkj[t] += scale * ds * bf16_to_double(qi[t]);
                dvj[t] += p[j] * bf16_to_double(doi[t]);
              }
            }
          }
        }
      }
    }
    free(p);
    free(dp);
  }
  return failed ? -5 : 0;
}
