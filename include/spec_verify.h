/*
 * spec_verify.h -- C ABI of the GB300 speculative-sampling verification library
 * (libspecverify.so, CUDA kernels for sm_103a).
 *
 * The operation is the verification step of speculative sampling as the pages
 * state it:
 *   - "Speculative Decoding" (roadtointelligence.com), section "Draft, then
 *     verify": a draft proposes K tokens, the target scores all K positions
 *     plus one more in one pass, each draft token x is kept with probability
 *     min(1, target(x)/draft(x)) left to right, the first rejection is
 *     replaced by a draw from the normalised max(0, target - draft) and the
 *     rest of the draft is discarded; if every draft token is kept, one more
 *     token is drawn from the target's extra position.  Each round emits
 *     between 1 and K+1 tokens.
 *   - "Accelerating Large Language Model Decoding with Speculative Sampling"
 *     (paperlayer.ai summary), section "Speculative Sampling", bullets
 *     "Modified Rejection Sampling": nucleus, top-k and temperature are
 *     applied before rejection sampling; the FDE Interviews breakdown of the
 *     same paper, section "01 The paper in one minute", adds greedy decoding.
 *   - "Speculative decoding: how to run large models faster" (ai-trend.me),
 *     section "How it works": argmax, top-k, nucleus and temperature are each
 *     sampling from an adjusted distribution.
 *
 * Conventions (all entry points):
 *   - Every buffer is owned by the caller.  Device pointers must stay valid
 *     until the work queued on params->stream has finished.  The library
 *     allocates no device memory per call: it needs a caller-provided
 *     workspace (see *_workspace_size) that is zero-filled once before its
 *     first use (cudaMemset).  Its first 64 KB hold the per-call counters;
 *     every call leaves them at zero again, so a workspace is reused across
 *     calls of any shape without clearing.  Calls that share one workspace
 *     must not overlap in time on the GPU.
 *   - Calls are asynchronous on params->stream (a cudaStream_t; NULL = the
 *     legacy default stream).  Argument errors are detected on the host,
 *     returned synchronously, and nothing is launched.
 *   - Errors found on the device never trap: the affected sequence (verify)
 *     or row (sample_draft) gets -1 in its outputs, and, when params->status
 *     is not NULL, the first error code is stored there (atomically, from 0;
 *     the caller zeroes it).  When several sequences fail with different
 *     codes, which code is stored is unspecified.
 *   - Inputs are never modified.
 *
 * Readings where the pages are silent (the same ones the fp64 test oracle
 * takes): the accept test is  u_t * drf_t(d_t) < tgt_t(d_t)  (no division,
 * so a draft probability of 0 accepts iff the target's is positive); draws walk
 * the vocabulary in ascending index order and return the smallest x with
 * u * R < sum_{y<=x} r(y), or, if rounding leaves none, the last x with
 * r(x) > 0; a zero residual mass draws from the target row instead; top-k and
 * top-p order tokens by raw logit (descending, ties to the lower index), apply
 * top-k first, then keep the shortest prefix whose mass reaches top_p
 * (crossing token included); -inf logits have probability 0; NaN or +inf
 * logits, or a row with no finite logit, are errors.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,  /* host: bad shape, pointer, stride, parameter or workspace */
  SPEC_ERR_CUDA = 2,         /* host: a CUDA runtime call failed (launch, attribute) */
  SPEC_ERR_NONFINITE = 3,    /* device: NaN or +inf logit, or no finite logit, in a row read */
  SPEC_ERR_TOKEN_RANGE = 4,  /* device: a draft token outside [0, V) */
  SPEC_ERR_TIMEOUT = 5,      /* device: reserved; a bulk copy that misses its bounded wait is
                                replaced by plain loads, so this version never reports it */
  SPEC_ERR_UNSUPPORTED = 6,  /* host: more shared memory than the device offers, or more than
                                2^31 - 1 row segments in one call */
  SPEC_ERR_SCRATCH_LIMIT = 7 /* host: spec_verify_noalloc asked for more than its fixed scratch */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef struct {
  int32_t B;                 /* sequences, >= 0 */
  int32_t K;                 /* draft tokens per sequence, >= 1 */
  int32_t V;                 /* vocabulary size, >= 1 */
  int32_t dtype;             /* spec_dtype of both logit tensors */
  /* Strides in ELEMENTS.  Row (b, t) of the target starts at
   * target_logits + b*target_seq_stride + t*target_row_stride; likewise for the
   * draft.  Any non-negative values are accepted (0 repeats rows); rows whose
   * start is 16-byte aligned take the bulk-copy path, others a plain-load path. */
  int64_t target_seq_stride, target_row_stride;
  int64_t draft_seq_stride, draft_row_stride;
  float temperature;         /* > 0 and finite unless greedy */
  int32_t top_k;             /* >= 0; 0 or >= V = no top-k */
  float top_p;               /* in (0, 1]; 1 = no nucleus filter */
  int32_t greedy;            /* nonzero: argmax special case (uniforms and draft rows unused) */
  void* stream;              /* cudaStream_t */
  int32_t* status;           /* optional device int32[1]: first device-detected error */
  void* workspace;           /* device, 256-byte aligned, zero-filled before first use */
  size_t workspace_bytes;
} spec_params;

/* Per-row record kept in the workspace (read back by spec_read_row_stats).
 * For every row the kernels read: zf = sum over kept x of 2^((l_x - m) * log2(e)/T),
 * the normaliser of the adjusted distribution relative to the row max m;
 * p_tok = adjusted probability of the sequence's draft token at this row
 * (verify, rows t < K; 0 otherwise); kept x satisfy l_x > tau_val, or
 * l_x == tau_val and x <= tau_idx; list_len >= 0 when the kept set (index order)
 * is stored in the workspace; flags: bit 0 non-finite row, bit 1 token out of
 * range, bit 2 timeout.  token = the drawn token (sample_draft only). */
typedef struct {
  double zf;
  double p_tok;
  float m;
  float tau_val;
  int32_t tau_idx;
  int32_t argmax;
  int32_t list_len;
  int32_t flags;
  int32_t token;
  int32_t pad_;
} spec_row_stat;

/* Workspace bytes spec_verify needs for these parameters (0 if they are invalid).
 * Rows per sequence: 2K+1 (sampling) or K+1 (greedy). */
size_t spec_verify_workspace_size(const spec_params* params);

/* Workspace bytes spec_sample_draft needs (0 if the parameters are invalid). */
size_t spec_sample_draft_workspace_size(const spec_params* params);

/* Verification step, one call for B independent sequences.
 *   target_logits     device, [B, K+1, V] rows (strides above), dtype
 *   draft_logits      device, [B, K, V] rows; may be NULL when greedy
 *   draft_tokens      device int32 [B, K], contiguous
 *   uniforms          device fp64 [B, K+1], contiguous: column t < K drives the
 *                     accept test at t, column K the single final draw (residual
 *                     or bonus); may be NULL when greedy
 *   out_tokens        device int32 [B, K+1]: the accepted draft tokens, then the
 *                     replacement or bonus token, then -1 padding
 *   out_num_accepted  device int32 [B]: accepted draft tokens n in [0, K]
 *                     (n+1 tokens emitted), or -1 for a sequence with an error */
spec_status spec_verify(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const double* uniforms,
                        const spec_params* params, int32_t* out_tokens,
                        int32_t* out_num_accepted);

/* Workspace bytes spec_verify_ragged needs (0 if the parameters are invalid):
 * the bytes of spec_verify with K the longest draft, plus the rows' index. */
size_t spec_verify_ragged_workspace_size(const spec_params* params);

/* Verification of a ragged batch: sequence b has its own draft length
 * 1 <= draft_lengths[b] <= K, and only its K_b + 1 target rows and K_b draft
 * rows are read ("Speculative Decoding", section "Draft, then verify", per
 * sequence; in a serving batch the sequences' lookaheads differ).  The result
 * for each sequence is spec_verify's with K = K_b.
 *   target_logits, draft_logits  device [B, K+1, V] / [B, K, V] rows (strides as
 *                     spec_verify); rows past a sequence's length are not read
 *   draft_tokens      device int32 [B, K]; columns >= K_b are not read
 *   uniforms          device fp64 [B, K+1]: column t < K_b the accept test at t,
 *                     column K_b the final draw (later columns are not read);
 *                     may be NULL when greedy
 *   draft_lengths     HOST int32 [B]: K_b (read before the call returns)
 *   params            as spec_verify, with K = the longest draft; the workspace
 *                     is spec_verify_ragged_workspace_size(params) bytes
 *   out_tokens        device int32 [B, K+1]: the n accepted tokens, the emitted
 *                     token, then -1 up to column K
 *   out_num_accepted  device int32 [B]: n in [0, K_b], or -1 on an error
 * Returns SPEC_ERR_INVALID_ARG (nothing launched) for a length outside [1, K]
 * or a NULL draft_lengths, plus spec_verify's checks. */
spec_status spec_verify_ragged(const void* target_logits, const void* draft_logits,
                               const int32_t* draft_tokens, const double* uniforms,
                               const int32_t* draft_lengths, const spec_params* params,
                               int32_t* out_tokens, int32_t* out_num_accepted);

/* Drafting step and verification fused, for K = 1: draw each sequence's one
 * draft token from its draft row (as spec_sample_draft), then verify it against
 * the two target rows (as spec_verify with that token) -- in one call, so the
 * draft row is read once.  The result is the same as the two calls in a row
 * with the same uniforms.  ("Speculative Decoding", section "Draft, then
 * verify", steps 1-4, with a lookahead of one token.)
 *   target_logits     device [B, 2, V] rows (target strides)
 *   draft_logits      device [B, 1, V] rows (draft strides)
 *   draft_uniforms    device fp64 [B]: the draft draws
 *   uniforms          device fp64 [B, 2]: column 0 the accept test, column 1
 *                     the final draw
 *   out_draft_tokens  device int32 [B]: the drawn draft tokens (-1 for a row
 *                     with an error)
 *   out_tokens, out_num_accepted  as spec_verify with K = 1
 * params->K must be 1 and params->greedy 0 (else SPEC_ERR_INVALID_ARG); the
 * workspace is spec_verify_workspace_size(params). */
spec_status spec_sample_verify(const void* target_logits, const void* draft_logits,
                               const double* draft_uniforms, const double* uniforms,
                               const spec_params* params, int32_t* out_draft_tokens,
                               int32_t* out_tokens, int32_t* out_num_accepted);

/* Draw the K draft tokens of each sequence from the adjusted draft distribution
 * (same temperature / top-k / top-p / greedy as verification), one inverse-CDF
 * draw per row in index order ("Speculative Decoding", section "Draft, then
 * verify", step 1).  In real decoding drafting is sequential and each call
 * draws K = 1 token per sequence; any K is accepted.
 *   draft_logits  device [B, K, V] rows (draft strides)
 *   uniforms      device fp64 [B, K], contiguous; may be NULL when greedy
 *   out_tokens    device int32 [B, K] (-1 for a row with an error)
 * The target fields of params are ignored. */
spec_status spec_sample_draft(const void* draft_logits, const double* uniforms,
                              const spec_params* params, int32_t* out_tokens);

/* Copy the per-row records of the last call made with this workspace and these
 * parameters into host memory: rows ordered by sequence, then target rows
 * 0..K followed by draft rows 0..K-1 (verify; greedy: target rows only), or
 * draft rows 0..K-1 (sample_draft, is_verify = 0).  Synchronises params->stream.
 * Returns SPEC_ERR_INVALID_ARG if max_rows is smaller than the row count. */
spec_status spec_read_row_stats(const spec_params* params, int32_t is_verify,
                                spec_row_stat* host_out, int64_t max_rows);

/* Scratch size of spec_verify_noalloc: 8 MiB.  Rows per call (B * (2K+1)
 * sampling, B * (K+1) greedy) that fit: about 1900 greedy; sampling, about 800
 * at V = 32000 and 150 at V = 256000 (bf16; every 24 KB segment of a row
 * keeps a candidate list). */
#define SPEC_NOALLOC_SCRATCH_BYTES (8u << 20)

/* spec_verify for callers that cannot allocate device memory.  Not a step of
 * the method: the pages have no counterpart; it only changes where the scratch
 * lives.
 *
 * Who needs it: a plugin inside a serving framework that has already reserved
 * the GPU's memory for its own pool (weights, KV cache) and hands the plugin
 * only the tensors it works on -- a cudaMalloc from the plugin would fail or
 * fragment that pool, and a plain C ABI gives it no handle to the framework's
 * allocator; and decode loops that must not allocate between tokens, because
 * cudaMalloc can synchronise the device.
 *
 * Same arguments and results as spec_verify; params->workspace and
 * params->workspace_bytes are ignored.  The scratch is one array of
 * SPEC_NOALLOC_SCRATCH_BYTES in device global memory, defined in the library,
 * which every GPU that loads the library keeps until the process exits.  The
 * first call on a device (made with that device current) looks up the array's
 * device address once; make that first call before any stream capture.  The
 * address is kept for the life of the process, so do not call this entry point
 * again after cudaDeviceReset on that device.  params->stream must belong to
 * the current device (else SPEC_ERR_INVALID_ARG, nothing launched).
 *
 *   - Every call uses the same array, which keeps the last call's contents.
 *     The array starts zeroed and every call leaves its counters at zero, so
 *     no clearing is needed between calls.
 *   - Calls whose work overlaps on the GPU (other streams, other threads)
 *     share the array and race: serialise them.
 *   - Returns SPEC_ERR_SCRATCH_LIMIT, with nothing launched, when
 *     spec_verify_workspace_size(params) exceeds SPEC_NOALLOC_SCRATCH_BYTES.
 *   - Never calls cudaMalloc, cudaFree or any allocating routine. */
spec_status spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                const int32_t* draft_tokens, const double* uniforms,
                                const spec_params* params, int32_t* out_tokens,
                                int32_t* out_num_accepted);

/* Static description of a status code. */
const char* spec_status_string(spec_status status);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t spec_launch_count(void);

/* Acceptance telemetry: adds the histogram of one call's accepted-draft counts
 * to hist.  The share of draft tokens accepted per round is the quantity to
 * watch ("Speculative decoding: how to run large models faster", ai-trend.me,
 * section "Limitations and open issues": fewer accepted tokens per round
 * means more target work), and out_num_accepted carries it per sequence.
 *   out_num_accepted  device int32 [B], as written by spec_verify
 *   B                 sequences (>= 0; 0 launches nothing)
 *   K                 draft tokens per sequence, 1 <= K <= 8192
 *   hist              device int32 [K+2], caller-owned and caller-zeroed:
 *                     hist[j] += sequences with j accepted tokens (0 <= j <= K),
 *                     hist[K+1] += sequences that ended in an error (-1) or
 *                     hold any other value
 *   stream            cudaStream_t (NULL = default stream)
 * Asynchronous on stream (one kernel); repeated calls accumulate.
 * Returns SPEC_ERR_INVALID_ARG (nothing launched) for B < 0, K outside
 * [1, 8192] or a NULL pointer with B > 0; SPEC_ERR_CUDA if the launch fails. */
spec_status spec_accept_histogram(const int32_t* out_num_accepted, int32_t B, int32_t K, int32_t* hist,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif
