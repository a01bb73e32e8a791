/*
 * oracle.h -- fp64 CPU oracle for speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the tests, `__graft_entry__.smoke()` and the
 * `cpu_baseline` / `--impl reference` legs of `bench.py` use it, as the
 * independent definition the CUDA path is checked against.  It shares no
 * header, helper, table or constant with the CUDA library.
 *
 * What it computes (all in fp64, one sequence at a time, no blocking or
 * fusion beyond the definition):
 *   - the adjusted distribution of one vocabulary row: temperature, then
 *     top-k, then top-p (nucleus), renormalised; greedy = one-hot argmax.
 *     ("Accelerating Large Language Model Decoding with Speculative Sampling",
 *     paperlayer.ai summary, section "Speculative Sampling", bullet
 *     "Modified Rejection Sampling" on nucleus / top-k / temperature applied
 *     before rejection sampling; "Speculative decoding: how to run large models
 *     faster", section "How it works", on rewriting argmax, top-k, nucleus and
 *     temperature as sampling from an adjusted distribution.)
 *   - the verification of K draft tokens against K+1 target rows: accept
 *     d_t with probability min(1, tgt_t(d_t)/drf_t(d_t)) left to right,
 *     resample at the first rejection from the normalised positive part of
 *     tgt - drf, or take a bonus token from target row K if every draft token
 *     survives.  ("Speculative Decoding", roadtointelligence.com, section
 *     "Draft, then verify", steps 3-4; the FDE Interviews breakdown of the
 *     same paper, section "01 The paper in one minute".)
 *   - drawing draft tokens from the adjusted draft distribution
 *     ("Speculative Decoding", section "Draft, then verify", step 1).
 *
 * Readings where the pages are silent (the CUDA library takes the same ones):
 *   accept test written as  u * drf < tgt  (no division; drf = 0 accepts iff
 *   tgt > 0); inverse-CDF draws walk the vocabulary in ascending index order
 *   and pick the smallest x with  u * R < cumsum(x);  if rounding leaves no
 *   such x the last x with positive weight is taken; a zero residual mass
 *   falls back to the target row; uniforms are laid out [B, K+1] (column t
 *   for the accept test at t, column K for the one final draw); top-k / top-p
 *   order tokens by raw logit descending, ties by lower index, and top-p keeps
 *   the shortest prefix whose mass reaches top_p (crossing token included).
 */
#ifndef SPECV_ORACLE_H
#define SPECV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_INVALID_ARG = 1,
  ORACLE_ERR_NONFINITE = 3,
  ORACLE_ERR_TOKEN_RANGE = 4
};

/* Per-sequence (verify) or per-row (sample_draft) near-threshold flags. */
enum {
  ORACLE_NEAR_ACCEPT = 1, /* |u_t - min(1, tgt/drf)| < ORACLE_NEAR_EPS at a test taken */
  ORACLE_NEAR_DRAW = 2,   /* u within ORACLE_NEAR_EPS of the chosen token's CDF edges */
  ORACLE_NEAR_TOPP = 4    /* a top-p cut whose cumulative mass is within the eps of top_p */
};

#define ORACLE_NEAR_EPS 1e-6

typedef struct {
  int32_t B, K, V;
  int32_t dtype;                       /* ORACLE_F32 or ORACLE_BF16 (raw uint16 bits) */
  int64_t tgt_seq_stride, tgt_row_stride; /* elements */
  int64_t drf_seq_stride, drf_row_stride; /* elements */
  float temperature;                   /* > 0 unless greedy */
  int32_t top_k;                       /* 0 (or >= V) = off */
  float top_p;                         /* (0, 1]; 1 = off */
  int32_t greedy;                      /* 1 = argmax special case */
} oracle_params;

/* Adjusted distribution of one row.  probs[V] receives P(x) in fp64.
 * *argmax receives the lowest index of the largest logit.  *near_topp is set
 * when the top-p cut is within ORACLE_NEAR_EPS.  If stats != NULL it receives
 * {max raw logit, Z_f} where Z_f = sum over kept x of exp((l_x - max)/T).
 * Returns ORACLE_OK or ORACLE_ERR_NONFINITE (NaN / +inf present, or no finite
 * logit). */
int oracle_row_probs(const void* row, int32_t dtype, int32_t V, float temperature,
                     int32_t top_k, float top_p, int32_t greedy, double* probs,
                     int32_t* argmax, int32_t* near_topp, double* stats);

/* Verification of B sequences.  Host arrays:
 *   tgt     target logits, row (b, t) at tgt + b*tgt_seq_stride + t*tgt_row_stride, t in [0, K]
 *   drf     draft logits,  row (b, t) likewise with drf strides, t in [0, K-1]
 *           (not read when greedy)
 *   tokens  [B, K] draft tokens
 *   u       [B, K+1] uniforms (not read when greedy)
 *   out_tokens [B, K+1] (-1 after the emitted ones), out_num_accepted [B]
 *   out_flags  [B] near-threshold bitmask (may be NULL)
 *   row_stats  optional [B, 2K+1, 3] doubles: {max, Z_f, p(d_t)} for target
 *              rows 0..K then draft rows 0..K-1 (p(d_t) = 0 for row K)
 * A sequence with an error gets out_num_accepted = -1 and out_tokens = -1.
 * Returns ORACLE_OK, ORACLE_ERR_INVALID_ARG, or the first sequence error. */
int oracle_verify(const void* tgt, const void* drf, const int32_t* tokens, const double* u,
                  const oracle_params* p, int32_t* out_tokens, int32_t* out_num_accepted,
                  int32_t* out_flags, double* row_stats);

/* Draft-token drawing: for every draft row (b, t), t in [0, K-1], draw from
 * the adjusted draft distribution with uniform u[b*K + t] (argmax if greedy).
 * out_tokens [B, K]; out_flags [B, K] (may be NULL).  A row with an error gets
 * token -1. */
int oracle_sample_draft(const void* drf, const double* u, const oracle_params* p,
                        int32_t* out_tokens, int32_t* out_flags);

/* Acceptance telemetry: hist[j] = number of sequences b with
 * num_accepted[b] == j for j in [0, K]; hist[K+1] = the rest (sequences that
 * ended in an error, num_accepted = -1).  hist has K+2 entries and is
 * overwritten.  ("Speculative decoding: how to run large models faster",
 * section "Limitations and open issues": the share of draft tokens accepted
 * per round is the quantity to watch.) */
void oracle_accept_histogram(const int32_t* num_accepted, int64_t B, int32_t K, int64_t* hist);

#ifdef __cplusplus
}
#endif

#endif
