/*
 * oracle.c -- fp64 CPU oracle for speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): the plain definition, written step
 * by step in fp64, single-threaded, with a full sort wherever an order is
 * needed.  Nothing here is tuned; it is what the CUDA path is checked against.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- reading one logit exactly as fp64 ---------------------------------- */

static double read_logit(const void* row, int32_t dtype, int64_t i) {
  if (dtype == ORACLE_F32) return (double)((const float*)row)[i];
  /* bf16 = the top 16 bits of an IEEE binary32 value */
  uint32_t bits = (uint32_t)((const uint16_t*)row)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static size_t elem_size(int32_t dtype) { return dtype == ORACLE_F32 ? 4 : 2; }

static const void* row_ptr(const void* base, int32_t dtype, int64_t off) {
  return (const char*)base + off * (int64_t)elem_size(dtype);
}

/* ---- the token order used by top-k and top-p ------------------------------
 * Raw logit descending, ties broken by the lower vocabulary index.  Ordering
 * on the raw logit (not on l/T) keeps the order exact for any T > 0. */

typedef struct {
  double l;
  int32_t x;
} keyed_token;

static int by_logit_desc_index_asc(const void* a, const void* b) {
  const keyed_token* p = (const keyed_token*)a;
  const keyed_token* q = (const keyed_token*)b;
  if (p->l > q->l) return -1;
  if (p->l < q->l) return 1;
  return (p->x > q->x) - (p->x < q->x);
}

/* ---- adjusted distribution of one row -------------------------------------
 * Temperature, then top-k, then top-p, then renormalise over the kept set;
 * greedy is the one-hot argmax.  Filters are applied before rejection
 * sampling ("Accelerating Large Language Model Decoding with Speculative
 * Sampling", paperlayer.ai summary, section "Speculative Sampling", bullet
 * "Modified Rejection Sampling"). */

int oracle_row_probs(const void* row, int32_t dtype, int32_t V, float temperature,
                     int32_t top_k, float top_p, int32_t greedy, double* probs,
                     int32_t* argmax, int32_t* near_topp, double* stats) {
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  unsigned char* kept = (unsigned char*)malloc((size_t)V);
  int status = ORACLE_OK;
  int32_t best = -1;
  double lmax = -INFINITY;
  int any_finite = 0;

  if (near_topp) *near_topp = 0;

  /* 1. read the row; NaN or +inf anywhere, or no finite logit, is an error */
  for (int32_t x = 0; x < V; ++x) {
    l[x] = read_logit(row, dtype, x);
    if (isnan(l[x]) || (isinf(l[x]) && l[x] > 0)) status = ORACLE_ERR_NONFINITE;
    if (isfinite(l[x])) any_finite = 1;
    if (best < 0 || l[x] > lmax) { /* strict: the first (lowest) index wins ties */
      lmax = l[x];
      best = x;
    }
  }
  if (!any_finite) status = ORACLE_ERR_NONFINITE;
  if (argmax) *argmax = best;
  if (status != ORACLE_OK) goto done;

  /* 2. greedy decoding is the argmax special case */
  if (greedy) {
    for (int32_t x = 0; x < V; ++x) probs[x] = (x == best) ? 1.0 : 0.0;
    if (stats) { stats[0] = lmax; stats[1] = 1.0; }
    goto done;
  }

  /* 3. temperature: s = l / T, m = max s, w = exp(s - m) */
  {
    const double T = (double)temperature;
    const double m = lmax / T;
    for (int32_t x = 0; x < V; ++x) {
      w[x] = isinf(l[x]) ? 0.0 : exp(l[x] / T - m);
      kept[x] = 1;
    }
  }

  /* 4. top-k, then top-p, on the order (raw logit desc, index asc) */
  {
    const int use_k = top_k > 0 && top_k < V;
    const int use_p = top_p < 1.0f;
    if (use_k || use_p) {
      keyed_token* order = (keyed_token*)malloc(sizeof(keyed_token) * (size_t)V);
      for (int32_t x = 0; x < V; ++x) { order[x].l = l[x]; order[x].x = x; }
      qsort(order, (size_t)V, sizeof(keyed_token), by_logit_desc_index_asc);
      int32_t nkeep = V;
      if (use_k) {
        nkeep = top_k;
        for (int32_t j = nkeep; j < V; ++j) kept[order[j].x] = 0;
      }
      if (use_p) {
        const double p = (double)top_p;
        double zk = 0.0;
        for (int32_t j = 0; j < nkeep; ++j) zk += w[order[j].x];
        double cum = 0.0, prev = 0.0;
        int32_t cut = nkeep - 1; /* rounding may leave the crossing unreached */
        for (int32_t j = 0; j < nkeep; ++j) {
          prev = cum;
          cum += w[order[j].x];
          if (cum / zk >= p) { cut = j; break; }
        }
        if (near_topp &&
            (fabs(cum / zk - p) < ORACLE_NEAR_EPS || (cut > 0 && fabs(prev / zk - p) < ORACLE_NEAR_EPS)))
          *near_topp = 1;
        for (int32_t j = cut + 1; j < nkeep; ++j) kept[order[j].x] = 0;
      }
      free(order);
    }
  }

  /* 5. renormalise over the kept set */
  {
    double zf = 0.0;
    for (int32_t x = 0; x < V; ++x)
      if (kept[x]) zf += w[x];
    for (int32_t x = 0; x < V; ++x) probs[x] = kept[x] ? w[x] / zf : 0.0;
    if (stats) { stats[0] = lmax; stats[1] = zf; }
  }

done:
  free(l);
  free(w);
  free(kept);
  return status;
}

/* ---- inverse-CDF draw in vocabulary index order ---------------------------
 * Smallest x with u*R < sum_{y<=x} r(y), R = sum r.  If rounding leaves no
 * such x, the last x with r(x) > 0.  Returns -1 if R == 0.  *near is set when
 * u lies within ORACLE_NEAR_EPS of the chosen token's CDF edges. */

static int32_t draw_index_order(const double* r, int32_t V, double u, int* near) {
  double R = 0.0;
  for (int32_t x = 0; x < V; ++x) R += r[x];
  *near = 0;
  if (!(R > 0.0)) return -1;
  const double target = u * R;
  double cum = 0.0, prev = 0.0;
  int32_t last = -1;
  for (int32_t x = 0; x < V; ++x) {
    if (!(r[x] > 0.0)) continue;
    prev = cum;
    cum += r[x];
    last = x;
    if (target < cum) {
      *near = fabs(u - prev / R) < ORACLE_NEAR_EPS || fabs(u - cum / R) < ORACLE_NEAR_EPS;
      return x;
    }
  }
  *near = fabs(u - cum / R) < ORACLE_NEAR_EPS || fabs(u - 1.0) < ORACLE_NEAR_EPS;
  return last;
}

/* ---- verification of one sequence ---------------------------------------- */

static int verify_one(const void* tgt, const void* drf, const int32_t* d, const double* u,
                      const oracle_params* p, int32_t* out_tok, int32_t* out_n, int32_t* flags,
                      double* stats) {
  const int32_t K = p->K, V = p->V;
  const int nt = K + 1, nd = p->greedy ? 0 : K;
  double* P = (double*)malloc(sizeof(double) * (size_t)V * (size_t)(nt + nd));
  int32_t* amax = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nt + nd));
  int status = ORACLE_OK;
  int32_t fl = 0;

  for (int32_t t = 0; t <= K; ++t) out_tok[t] = -1;
  *out_n = -1;

  for (int32_t t = 0; t < K; ++t)
    if (d[t] < 0 || d[t] >= V) status = ORACLE_ERR_TOKEN_RANGE;

  /* adjusted distributions: target rows 0..K, draft rows 0..K-1 */
  for (int r = 0; r < nt + nd && status == ORACLE_OK; ++r) {
    const int is_t = r < nt;
    const int32_t t = is_t ? r : r - nt;
    const void* row = is_t ? row_ptr(tgt, p->dtype, t * p->tgt_row_stride)
                           : row_ptr(drf, p->dtype, t * p->drf_row_stride);
    int32_t near = 0;
    double st[2] = {0.0, 0.0};
    int s = oracle_row_probs(row, p->dtype, V, p->temperature, p->top_k, p->top_p, p->greedy,
                             P + (size_t)r * V, &amax[r], &near, st);
    if (s != ORACLE_OK) { status = s; break; }
    if (near) fl |= ORACLE_NEAR_TOPP;
    if (stats) {
      stats[3 * r + 0] = st[0];
      stats[3 * r + 1] = st[1];
      stats[3 * r + 2] = (t < K) ? P[(size_t)r * V + d[t]] : 0.0;
    }
  }
  if (status != ORACLE_OK) goto done;

  {
    int32_t n = K;
    if (p->greedy) {
      /* argmax special case: keep d_t while it equals the target's argmax */
      for (int32_t t = 0; t < K; ++t)
        if (d[t] != amax[t]) { n = t; break; }
      for (int32_t t = 0; t < n; ++t) out_tok[t] = d[t];
      out_tok[n] = amax[n];
    } else {
      /* accept d_t with probability min(1, tgt/drf), left to right */
      for (int32_t t = 0; t < K; ++t) {
        const double a = P[(size_t)t * V + d[t]];        /* tgt_t(d_t) */
        const double b = P[(size_t)(nt + t) * V + d[t]]; /* drf_t(d_t) */
        const double ratio = b > 0.0 ? fmin(1.0, a / b) : 1.0;
        if (fabs(u[t] - ratio) < ORACLE_NEAR_EPS) fl |= ORACLE_NEAR_ACCEPT;
        if (!(u[t] * b < a)) { n = t; break; }
      }
      for (int32_t t = 0; t < n; ++t) out_tok[t] = d[t];
      /* first rejection: residual max(0, tgt - drf); all accepted: bonus row K */
      double* r = (double*)malloc(sizeof(double) * (size_t)V);
      const double* pt = P + (size_t)n * V;
      if (n < K) {
        const double* pd = P + (size_t)(nt + n) * V;
        for (int32_t x = 0; x < V; ++x) r[x] = fmax(0.0, pt[x] - pd[x]);
      } else {
        memcpy(r, pt, sizeof(double) * (size_t)V);
      }
      int near = 0;
      int32_t tok = draw_index_order(r, V, u[K], &near);
      if (tok < 0) tok = draw_index_order(pt, V, u[K], &near); /* zero residual mass */
      if (near) fl |= ORACLE_NEAR_DRAW;
      out_tok[n] = tok;
      free(r);
    }
    *out_n = n;
  }

done:
  if (status != ORACLE_OK) {
    for (int32_t t = 0; t <= K; ++t) out_tok[t] = -1;
    *out_n = -1;
  }
  if (flags) *flags = fl;
  free(P);
  free(amax);
  return status;
}

static int params_ok(const oracle_params* p) {
  if (!p || p->B < 0 || p->K < 1 || p->V < 1) return 0;
  if (p->dtype != ORACLE_F32 && p->dtype != ORACLE_BF16) return 0;
  if (!p->greedy) {
    if (!(p->temperature > 0.0f) || isinf(p->temperature)) return 0;
    if (!(p->top_p > 0.0f && p->top_p <= 1.0f)) return 0;
    if (p->top_k < 0) return 0;
  }
  return 1;
}

int oracle_verify(const void* tgt, const void* drf, const int32_t* tokens, const double* u,
                  const oracle_params* p, int32_t* out_tokens, int32_t* out_num_accepted,
                  int32_t* out_flags, double* row_stats) {
  if (!params_ok(p)) return ORACLE_ERR_INVALID_ARG;
  int first_err = ORACLE_OK;
  const int32_t K = p->K;
  for (int32_t b = 0; b < p->B; ++b) {
    int32_t fl = 0;
    int s = verify_one(row_ptr(tgt, p->dtype, b * p->tgt_seq_stride),
                       p->greedy ? NULL : row_ptr(drf, p->dtype, b * p->drf_seq_stride),
                       tokens + (size_t)b * K, p->greedy ? NULL : u + (size_t)b * (K + 1), p,
                       out_tokens + (size_t)b * (K + 1), out_num_accepted + b, &fl,
                       row_stats ? row_stats + (size_t)b * (2 * K + 1) * 3 : NULL);
    if (out_flags) out_flags[b] = fl;
    if (s != ORACLE_OK && first_err == ORACLE_OK) first_err = s;
  }
  return first_err;
}

int oracle_sample_draft(const void* drf, const double* u, const oracle_params* p,
                        int32_t* out_tokens, int32_t* out_flags) {
  if (!params_ok(p)) return ORACLE_ERR_INVALID_ARG;
  const int32_t K = p->K, V = p->V;
  double* P = (double*)malloc(sizeof(double) * (size_t)V);
  int first_err = ORACLE_OK;
  for (int32_t b = 0; b < p->B; ++b) {
    for (int32_t t = 0; t < K; ++t) {
      const void* row = row_ptr(drf, p->dtype, b * p->drf_seq_stride + t * p->drf_row_stride);
      int32_t amax = -1, near_p = 0;
      int near_d = 0;
      int32_t tok = -1;
      int s = oracle_row_probs(row, p->dtype, V, p->temperature, p->top_k, p->top_p, p->greedy, P,
                               &amax, &near_p, NULL);
      if (s == ORACLE_OK) tok = p->greedy ? amax : draw_index_order(P, V, u[(size_t)b * K + t], &near_d);
      else if (first_err == ORACLE_OK) first_err = s;
      out_tokens[(size_t)b * K + t] = tok;
      if (out_flags)
        out_flags[(size_t)b * K + t] = (near_p ? ORACLE_NEAR_TOPP : 0) | (near_d ? ORACLE_NEAR_DRAW : 0);
    }
  }
  free(P);
  return first_err;
}

/* Acceptance telemetry: count the sequences per number of accepted draft
 * tokens; anything outside [0, K] (an error) goes to the last bin. */
void oracle_accept_histogram(const int32_t* num_accepted, int64_t B, int32_t K, int64_t* hist) {
  for (int32_t j = 0; j < K + 2; ++j) hist[j] = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int32_t n = num_accepted[b];
    if (n >= 0 && n <= K)
      hist[n] += 1;
    else
      hist[K + 1] += 1;
  }
}
