// spec_verify.cu -- the host side of libspecverify: argument checks, launch
// planning, the C ABI entry points, the acceptance histogram kernel and the
// fixed scratch of spec_verify_noalloc.  The kernels live in spec_kernels.cuh;
// kernel_unit.cu instantiates them in groups that compile in parallel, and
// kernel_table.h names the groups.
#include "spec_kernels.cuh"
#include "kernel_table.h"


// ---------------------------------------------------------------------------
// Acceptance telemetry: a histogram of the accepted-draft counts of a call.
// Bins 0..K count the sequences by accepted tokens; bin K+1 the sequences that
// ended in an error.  Each CTA counts in shared memory, then adds its nonzero
// bins to the caller's histogram.

__global__ void __launch_bounds__(256) spec_hist_kernel(const int32_t* __restrict__ n_acc, int B, int K,
                                                        int32_t* __restrict__ hist) {
  extern __shared__ int32_t bins[];
  for (int i = threadIdx.x; i < K + 2; i += blockDim.x) bins[i] = 0;
  __syncthreads();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < B; i += gridDim.x * blockDim.x) {
    const int v = __ldg(&n_acc[i]);
    atomicAdd(&bins[(v >= 0 && v <= K) ? v : K + 1], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < K + 2; i += blockDim.x)
    if (bins[i] != 0) atomicAdd(&hist[i], bins[i]);
}

// ===========================================================================
// host side

namespace {

std::atomic<uint64_t> g_launches{0};

struct DevInfo {
  int sms = 0;
  int max_smem = 0;
  size_t smem_set[8] = {};  // dynamic smem attribute set: [kernel * 4 + ragged * 2 + dtype]
  int per_sm[4] = {};       // resident segment-kernel CTAs per SM: [ragged * 2 + dtype]
  size_t ssmem_set[6] = {};  // streaming kernel: [mode * 2 + dtype]
  int sper_sm[6] = {};       // resident streaming-kernel CTAs per SM, same index
};
std::mutex g_mu;
DevInfo g_dev[64];

bool dev_info(DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo& d = g_dev[dev];
  if (d.sms == 0) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return false;
  }
  *out = &d;
  return true;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int esize = 0, R = 0, S = 0, nseg = 0, n0 = 0, grid = 0, row_grid = 0, seg_bytes = 0;
  bool clear_counters = false;  // more counters than the area that calls keep zeroed
  bool ragged = false;          // per-sequence draft lengths (the kernels' RAG instantiation)
  bool aligned = false;         // every row start is 16-byte aligned
  bool stream = false;          // the one-launch streaming kernel (else segment + row kernels)
  int smode = kSMGreedy;        // its instantiation: kSMGreedy, kSMTopK, kSMTopP
  int nseg_ws = 0;              // segment records per row the workspace holds
  size_t counter_bytes = 0;
  int64_t nrows = 0, items = 0;
  size_t smem = 0, row_smem = 0;  // dynamic shared memory of the segment and row kernels
  size_t off_tickets = 0, off_rows = 0, off_lidx = 0, off_lw = 0, off_segs = 0, off_cand = 0, ws_bytes = 0;
};

bool finite_positive(float x) { return x > 0.0f && x < INFINITY; }

// Validates the parameters shared by both entry points, cuts rows into equal
// segments of at most kNV vectors per thread and sizes the workspace -- all
// from the parameters alone (no CUDA call), so the *_workspace_size queries work
// without a device.
spec_status make_plan(const spec_params* p, bool verify, Plan* pl) {
  if (!p) return SPEC_ERR_INVALID_ARG;
  if (p->B < 0 || p->K < 1 || p->V < 1) return SPEC_ERR_INVALID_ARG;
  if (p->dtype != SPEC_F32 && p->dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (p->target_seq_stride < 0 || p->target_row_stride < 0 || p->draft_seq_stride < 0 ||
      p->draft_row_stride < 0)
    return SPEC_ERR_INVALID_ARG;
  if (!p->greedy) {
    if (!finite_positive(p->temperature)) return SPEC_ERR_INVALID_ARG;
    if (!(p->top_p > 0.0f && p->top_p <= 1.0f)) return SPEC_ERR_INVALID_ARG;
    if (p->top_k < 0) return SPEC_ERR_INVALID_ARG;
  }
  pl->esize = (p->dtype == SPEC_F32) ? 4 : 2;
  pl->R = verify ? (p->greedy ? p->K + 1 : 2 * p->K + 1) : p->K;
  pl->nrows = static_cast<int64_t>(p->B) * pl->R;
  if (pl->nrows > (int64_t(1) << 30)) return SPEC_ERR_INVALID_ARG;
  const int64_t V = p->V;
  const int64_t N = 16 / pl->esize;  // elements per 16-byte vector
  const int64_t smax = static_cast<int64_t>(kNV) * kThreads * N;
  int64_t nseg = (V + smax - 1) / smax;
  int64_t S = (V + nseg - 1) / nseg;
  S = (S + N - 1) / N * N;
  nseg = (V + S - 1) / S;
  pl->S = static_cast<int>(S);
  pl->nseg = static_cast<int>(nseg);
  pl->items = pl->nrows * nseg;
  if (pl->items > INT_MAX) return SPEC_ERR_UNSUPPORTED;
  // candidate floor rank: a segment's top-k for top-k; for top-p alone a floor
  // whose candidates (about 1.4 n0 per segment) leave the row's pool room
  const bool use_k = !p->greedy && p->top_k > 0 && p->top_k < p->V;
  const bool use_p = !p->greedy && p->top_p < 1.0f;
  pl->n0 = use_k ? p->top_k : use_p ? static_cast<int>(std::min<int64_t>(128, std::max<int64_t>(16, 560 / nseg))) : 0;
  // segment kernel: two segment buffers; row kernel: the pool, its sort keys and
  // the merge's entry table
  pl->seg_bytes = static_cast<int>(round_up(static_cast<size_t>(S) * pl->esize, 128));
  pl->smem = sizeof(Scratch) + 2 * static_cast<size_t>(pl->seg_bytes);
  pl->row_smem = sizeof(Scratch) + kPool * (sizeof(int32_t) + sizeof(float) + sizeof(unsigned long long)) + kListTable;
  pl->nseg_ws = pl->nseg;
  const size_t nr = static_cast<size_t>(pl->nrows);
  const size_t ni = static_cast<size_t>(pl->items);
  // the counter area: at offset 0 and at least kCounterArea bytes, so that a
  // later call with another layout still finds the zeros this call leaves
  const size_t counters = static_cast<size_t>(p->B) * sizeof(unsigned long long);
  pl->off_tickets = 0;
  pl->counter_bytes = counters;
  pl->clear_counters = counters > kCounterArea;
  pl->off_rows = std::max(kCounterArea, round_up(counters, 256));
  pl->off_lidx = pl->off_rows + round_up(nr * sizeof(spec_row_stat), 256);
  pl->off_lw = pl->off_lidx + round_up(nr * kCap * 4, 256);
  pl->off_segs = pl->off_lw + round_up(nr * kCap * 4, 256);
  pl->off_cand = pl->off_segs + round_up(ni * sizeof(SegRec), 256);
  // candidate lists whenever sampling (the size must not depend on top-k / top-p)
  pl->ws_bytes = pl->off_cand + (p->greedy ? 0 : round_up(ni * kSegCap * sizeof(uint2), 256));
  return SPEC_OK;
}

const void* seg_fn(bool f32, bool rag) { return f32 ? specv_units::seg_f32(rag) : specv_units::seg_bf16(rag); }
const void* row_fn(bool f32, bool rag) { return f32 ? specv_units::row_f32(rag) : specv_units::row_bf16(rag); }
const void* stream_fn(bool f32, int mode) {
  using namespace specv_units;
  if (mode == kSMTopK) return f32 ? stream_f32_k() : stream_bf16_k();
  if (mode == kSMTopP) return f32 ? stream_f32_topp() : stream_bf16_topp();
  return f32 ? stream_f32_greedy() : stream_bf16_greedy();
}

spec_status set_smem(DevInfo& di, int slot, const void* fn, size_t bytes) {
  if (di.smem_set[slot] >= bytes) return SPEC_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) != cudaSuccess ||
      cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return SPEC_ERR_CUDA;
  di.smem_set[slot] = bytes;
  return SPEC_OK;
}

// The streaming kernel takes greedy, top-k (k <= kSK, with or without top-p)
// and top-p calls (ragged or not) whose rows start on 16-byte boundaries: a
// persistent grid, as many CTAs as fit at once, one row at a time each (the row record and the kept list go
// where the two-kernel path puts them; its per-row part record is written only
// for the general path).
spec_status plan_stream(const spec_params* p, DevInfo& di, Plan* pl) {
  const bool use_k = !p->greedy && p->top_k > 0 && p->top_k < p->V;
  const bool use_p = !p->greedy && p->top_p < 1.0f;
  // no filter stays on the two-kernel path (the kept set is the whole row)
  if (!pl->aligned) return SPEC_OK;
  // a candidate group's first vector shares its buffer word with the mask of its vectors
  if ((static_cast<int64_t>(p->V) * pl->esize + 15) / 16 >= (int64_t(1) << kSVShift)) return SPEC_OK;
  int mode;
  if (p->greedy) mode = kSMGreedy;            // max and argmax
  else if (use_k && p->top_k <= kSK) mode = kSMTopK;  // candidate groups (top-p within them)
  else if (use_p && !use_k) mode = kSMTopP;   // candidate groups and the normaliser
  else return SPEC_OK;
  const bool cand = mode != kSMGreedy;
  const size_t smem = cand ? stream_smem_bytes<1>() : stream_smem_bytes<0>();
  if (smem > static_cast<size_t>(di.max_smem)) return SPEC_OK;
  const int which = (p->dtype == SPEC_F32) ? 0 : 1;
  const int slot = mode * 2 + which;
  const void* fn = stream_fn(which == 0, mode);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (di.ssmem_set[slot] < smem) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
              cudaSuccess ||
          cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return SPEC_ERR_CUDA;
      di.ssmem_set[slot] = smem;
    }
    if (di.sper_sm[slot] == 0) {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem) != cudaSuccess || per_sm < 1)
        return SPEC_ERR_CUDA;
      di.sper_sm[slot] = per_sm;
    }
  }
  const int64_t slots = static_cast<int64_t>(di.sper_sm[slot]) * di.sms;
  pl->stream = true;
  pl->smode = mode;
  pl->S = p->V;
  pl->nseg = 1;
  pl->items = pl->nrows;
  pl->smem = smem;
  pl->grid = static_cast<int>(std::min<int64_t>(pl->nrows, slots));
  return SPEC_OK;
}

// Segment kernel: a persistent grid, as many CTAs as fit at once (never more
// than the items).  Row kernel: one CTA per row.
spec_status plan_launch(const spec_params* p, DevInfo& di, Plan* pl) {
  spec_status st = plan_stream(p, di, pl);
  if (st != SPEC_OK || pl->stream) return st;
  if (pl->smem > static_cast<size_t>(di.max_smem) || pl->row_smem > static_cast<size_t>(di.max_smem))
    return SPEC_ERR_UNSUPPORTED;
  const int which = (p->dtype == SPEC_F32) ? 0 : 1;
  const bool rag = pl->ragged;
  const void* fs = seg_fn(which == 0, rag);
  const void* fr = row_fn(which == 0, rag);
  const int slot = (rag ? 2 : 0) + which;
  std::lock_guard<std::mutex> lock(g_mu);
  const size_t before = di.smem_set[slot];
  spec_status s = set_smem(di, slot, fs, pl->smem);
  if (s != SPEC_OK) return s;
  s = set_smem(di, 4 + slot, fr, pl->row_smem);
  if (s != SPEC_OK) return s;
  if (di.per_sm[slot] == 0 || di.smem_set[slot] != before) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fs, kThreads, pl->smem) != cudaSuccess || per_sm < 1)
      return SPEC_ERR_CUDA;
    di.per_sm[slot] = per_sm;
  }
  pl->grid = static_cast<int>(std::min<int64_t>(pl->items, static_cast<int64_t>(di.per_sm[slot]) * di.sms));
  pl->row_grid = static_cast<int>(std::min<int64_t>(pl->nrows, int64_t(1) << 20));
  return SPEC_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

spec_status launch(const spec_params* p, const Plan& pl, KArgs& a, DevInfo* di) {
  (void)di;
  if (pl.nrows == 0) return SPEC_OK;
  const dim3 grid(static_cast<unsigned>(pl.grid)), rgrid(static_cast<unsigned>(pl.row_grid)), block(kThreads);
  cudaStream_t st = static_cast<cudaStream_t>(p->stream);
  if (pl.clear_counters && cudaMemsetAsync(p->workspace, 0, pl.counter_bytes, st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (pl.stream) {
    const void* fn = stream_fn(p->dtype == SPEC_F32, pl.smode);
    void* args[] = {&a};
    if (cudaLaunchKernel(fn, grid, block, args, pl.smem, st) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
  }
  // the row kernel is a programmatic dependent launch: it may be scheduled
  // while the segment kernel's last CTAs finish, and waits in its prologue
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = rgrid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = pl.row_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  const bool f32 = p->dtype == SPEC_F32;
  if (cudaLaunchKernel(seg_fn(f32, pl.ragged), grid, block, args, pl.smem, st) != cudaSuccess) return SPEC_ERR_CUDA;
  const cudaError_t e = cudaLaunchKernelExC(&cfg, row_fn(f32, pl.ragged), args);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  g_launches.fetch_add(2, std::memory_order_relaxed);
  return SPEC_OK;
}

// Multiplier and shift for division by d (1 <= d < 2^31) of 0 <= n < 2^31 by
// a multiply-high: q = (umulhi(n, m) + n) >> s (Granlund and Montgomery,
// "Division by Invariant Integers using Multiplication", 1994).
void div_magic(uint32_t d, uint32_t* m, uint32_t* s) {
  uint32_t sh = 0;
  while ((uint64_t(1) << sh) < d) ++sh;
  *m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << sh) - d)) / d + 1);
  *s = sh;
}

void fill_common(const spec_params* p, const Plan& pl, KArgs& a) {
  char* ws = static_cast<char*>(p->workspace);
  a.tickets = reinterpret_cast<unsigned long long*>(ws + pl.off_tickets);
  a.rows = reinterpret_cast<spec_row_stat*>(ws + pl.off_rows);
  a.list_idx = reinterpret_cast<int32_t*>(ws + pl.off_lidx);
  a.list_w = reinterpret_cast<float*>(ws + pl.off_lw);
  a.segs = reinterpret_cast<SegRec*>(ws + pl.off_segs);
  a.seg_cand = reinterpret_cast<uint2*>(ws + pl.off_cand);
  a.B = p->B;
  a.K = p->K;
  a.V = p->V;
  a.R = pl.R;
  a.S = pl.S;
  a.nseg = pl.nseg;
  div_magic(static_cast<uint32_t>(pl.nseg), &a.nseg_m, &a.nseg_s);
  a.seg_bytes = pl.seg_bytes;
  a.nrows = static_cast<int>(pl.nrows);
  a.greedy = p->greedy ? 1 : 0;
  a.top_k = (p->greedy || p->top_k >= p->V) ? 0 : p->top_k;
  a.top_p = p->greedy ? 1.0f : p->top_p;
  a.temp = p->greedy ? 1.0f : p->temperature;
  a.c = p->greedy ? 1.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(p->temperature));
  const bool use_k = a.top_k > 0, use_p = a.top_p < 1.0f;
  a.filt = (!p->greedy && (use_k || use_p)) ? 1 : 0;
  a.need_z = (!p->greedy && !use_k) ? 1 : 0;
  a.n0 = pl.n0;
  a.status = p->status;
}

// rows per sequence for the fast division (after a.mode is set)
void fill_rows_div(KArgs& a) {
  div_magic(static_cast<uint32_t>(a.mode == kModeVerify ? a.R : a.K), &a.rows_m, &a.rows_s);
}

bool workspace_ok(const spec_params* p, const Plan& pl) {
  return p->workspace && (reinterpret_cast<uintptr_t>(p->workspace) & 255u) == 0 &&
         p->workspace_bytes >= pl.ws_bytes;
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(const spec_params* params) {
  Plan pl;
  return make_plan(params, true, &pl) == SPEC_OK ? pl.ws_bytes : 0;
}

size_t spec_sample_draft_workspace_size(const spec_params* params) {
  Plan pl;
  return make_plan(params, false, &pl) == SPEC_OK ? pl.ws_bytes : 0;
}

spec_status spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                        const double* uniforms, const spec_params* params, int32_t* out_tokens,
                        int32_t* out_num_accepted) {
  Plan pl;
  spec_status s = make_plan(params, true, &pl);
  if (s != SPEC_OK) return s;
  const spec_params* p = params;
  if (p->B == 0) return SPEC_OK;
  if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted) return SPEC_ERR_INVALID_ARG;
  if (!p->greedy && (!draft_logits || !uniforms)) return SPEC_ERR_INVALID_ARG;
  if (!workspace_ok(p, pl)) return SPEC_ERR_INVALID_ARG;
  const int64_t es = pl.esize;
  bool al = aligned16(target_logits) && (p->target_seq_stride * es) % 16 == 0 && (p->target_row_stride * es) % 16 == 0;
  if (!p->greedy)
    al = al && aligned16(draft_logits) && (p->draft_seq_stride * es) % 16 == 0 && (p->draft_row_stride * es) % 16 == 0;
  pl.aligned = al;
  DevInfo* di = nullptr;
  if (!dev_info(&di)) return SPEC_ERR_CUDA;
  s = plan_launch(p, *di, &pl);
  if (s != SPEC_OK) return s;
  KArgs a = {};
  a.tgt = target_logits;
  a.drf = draft_logits;
  a.tgt_seq = p->target_seq_stride;
  a.tgt_row = p->target_row_stride;
  a.drf_seq = p->draft_seq_stride;
  a.drf_row = p->draft_row_stride;
  a.tokens = draft_tokens;
  a.u = uniforms;
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.mode = kModeVerify;
  a.aligned = al ? 1 : 0;
  fill_common(p, pl, a);
  fill_rows_div(a);
  return launch(p, pl, a, di);
}

size_t spec_verify_ragged_workspace_size(const spec_params* params) {
  Plan pl;
  if (make_plan(params, true, &pl) != SPEC_OK) return 0;
  return pl.ws_bytes + round_up(static_cast<size_t>(pl.nrows) * sizeof(int2), 256);
}

spec_status spec_verify_ragged(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                               const double* uniforms, const int32_t* draft_lengths, const spec_params* params,
                               int32_t* out_tokens, int32_t* out_num_accepted) {
  Plan pl;
  spec_status s = make_plan(params, true, &pl);
  if (s != SPEC_OK) return s;
  const spec_params* p = params;
  if (p->B == 0) return SPEC_OK;
  if (!draft_lengths || !target_logits || !draft_tokens || !out_tokens || !out_num_accepted)
    return SPEC_ERR_INVALID_ARG;
  if (!p->greedy && (!draft_logits || !uniforms)) return SPEC_ERR_INVALID_ARG;
  // the rows of every sequence, from its draft length (host array): one
  // {sequence, position | K_b << 16} entry per row
  if (p->K >= 32768) return SPEC_ERR_UNSUPPORTED;
  std::vector<int2> map;
  map.reserve(static_cast<size_t>(pl.nrows));
  for (int b = 0; b < p->B; ++b) {
    const int kb = draft_lengths[b];
    if (kb < 1 || kb > p->K) return SPEC_ERR_INVALID_ARG;
    const int nr = p->greedy ? kb + 1 : 2 * kb + 1;
    for (int r = 0; r < nr; ++r) map.push_back(make_int2(b, r | (kb << 16)));
  }
  const int64_t total = static_cast<int64_t>(map.size());
  const size_t off_start = pl.ws_bytes;
  const size_t need = off_start + round_up(static_cast<size_t>(pl.nrows) * sizeof(int2), 256);
  if (!p->workspace || (reinterpret_cast<uintptr_t>(p->workspace) & 255u) != 0 || p->workspace_bytes < need)
    return SPEC_ERR_INVALID_ARG;
  pl.nrows = total;  // <= the padded B (2K+1) the workspace was sized for
  pl.ragged = true;
  pl.items = total * pl.nseg;
  const int64_t es = pl.esize;
  bool al = aligned16(target_logits) && (p->target_seq_stride * es) % 16 == 0 && (p->target_row_stride * es) % 16 == 0;
  if (!p->greedy)
    al = al && aligned16(draft_logits) && (p->draft_seq_stride * es) % 16 == 0 && (p->draft_row_stride * es) % 16 == 0;
  pl.aligned = al;
  DevInfo* di = nullptr;
  if (!dev_info(&di)) return SPEC_ERR_CUDA;
  s = plan_launch(p, *di, &pl);
  if (s != SPEC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(p->stream);
  int2* d_map = reinterpret_cast<int2*>(static_cast<char*>(p->workspace) + off_start);
  // pageable source: the copy is staged before this call returns
  if (cudaMemcpyAsync(d_map, map.data(), map.size() * sizeof(int2), cudaMemcpyHostToDevice, st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  KArgs a = {};
  a.tgt = target_logits;
  a.drf = draft_logits;
  a.tgt_seq = p->target_seq_stride;
  a.tgt_row = p->target_row_stride;
  a.drf_seq = p->draft_seq_stride;
  a.drf_row = p->draft_row_stride;
  a.tokens = draft_tokens;
  a.u = uniforms;
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.mode = kModeVerify;
  a.aligned = al ? 1 : 0;
  a.row_map = d_map;
  fill_common(p, pl, a);
  fill_rows_div(a);
  return launch(p, pl, a, di);
}

spec_status spec_sample_verify(const void* target_logits, const void* draft_logits, const double* draft_uniforms,
                               const double* uniforms, const spec_params* params, int32_t* out_draft_tokens,
                               int32_t* out_tokens, int32_t* out_num_accepted) {
  if (!params) return SPEC_ERR_INVALID_ARG;
  if (params->K != 1 || params->greedy) return SPEC_ERR_INVALID_ARG;
  Plan pl;
  spec_status s = make_plan(params, true, &pl);
  if (s != SPEC_OK) return s;
  const spec_params* p = params;
  if (p->B == 0) return SPEC_OK;
  if (!target_logits || !draft_logits || !draft_uniforms || !uniforms || !out_draft_tokens || !out_tokens ||
      !out_num_accepted)
    return SPEC_ERR_INVALID_ARG;
  if (!workspace_ok(p, pl)) return SPEC_ERR_INVALID_ARG;
  const int64_t es = pl.esize;
  const bool al = aligned16(target_logits) && (p->target_seq_stride * es) % 16 == 0 &&
                  (p->target_row_stride * es) % 16 == 0 && aligned16(draft_logits) &&
                  (p->draft_seq_stride * es) % 16 == 0 && (p->draft_row_stride * es) % 16 == 0;
  pl.aligned = al;
  DevInfo* di = nullptr;
  if (!dev_info(&di)) return SPEC_ERR_CUDA;
  s = plan_launch(p, *di, &pl);
  if (s != SPEC_OK) return s;
  KArgs a = {};
  a.tgt = target_logits;
  a.drf = draft_logits;
  a.tgt_seq = p->target_seq_stride;
  a.tgt_row = p->target_row_stride;
  a.drf_seq = p->draft_seq_stride;
  a.drf_row = p->draft_row_stride;
  a.tokens = out_draft_tokens;  // written by the draft rows, read by the sequence epilogue
  a.u = uniforms;
  a.out_tokens = out_tokens;
  a.out_n = out_num_accepted;
  a.mode = kModeVerify;
  a.aligned = al ? 1 : 0;
  a.fused = 1;
  a.u_draft = draft_uniforms;
  a.out_draft = out_draft_tokens;
  fill_common(p, pl, a);
  fill_rows_div(a);
  return launch(p, pl, a, di);
}

spec_status spec_sample_draft(const void* draft_logits, const double* uniforms, const spec_params* params,
                              int32_t* out_tokens) {
  Plan pl;
  spec_status s = make_plan(params, false, &pl);
  if (s != SPEC_OK) return s;
  const spec_params* p = params;
  if (p->B == 0) return SPEC_OK;
  if (!draft_logits || !out_tokens || (!p->greedy && !uniforms)) return SPEC_ERR_INVALID_ARG;
  if (!workspace_ok(p, pl)) return SPEC_ERR_INVALID_ARG;
  const int64_t es = pl.esize;
  const bool al = aligned16(draft_logits) && (p->draft_seq_stride * es) % 16 == 0 && (p->draft_row_stride * es) % 16 == 0;
  pl.aligned = al;
  DevInfo* di = nullptr;
  if (!dev_info(&di)) return SPEC_ERR_CUDA;
  s = plan_launch(p, *di, &pl);
  if (s != SPEC_OK) return s;
  KArgs a = {};
  a.tgt = draft_logits;  // unused in sample mode
  a.drf = draft_logits;
  a.drf_seq = p->draft_seq_stride;
  a.drf_row = p->draft_row_stride;
  a.u = uniforms;
  a.out_tokens = out_tokens;
  a.mode = kModeSample;
  a.aligned = al ? 1 : 0;
  fill_common(p, pl, a);
  fill_rows_div(a);
  return launch(p, pl, a, di);
}

spec_status spec_read_row_stats(const spec_params* params, int32_t is_verify, spec_row_stat* host_out,
                                int64_t max_rows) {
  Plan pl;
  spec_status s = make_plan(params, is_verify != 0, &pl);
  if (s != SPEC_OK) return s;
  if (!host_out || max_rows < pl.nrows || !workspace_ok(params, pl)) return SPEC_ERR_INVALID_ARG;
  if (pl.nrows == 0) return SPEC_OK;
  cudaStream_t st = static_cast<cudaStream_t>(params->stream);
  const char* src = static_cast<const char*>(params->workspace) + pl.off_rows;
  if (cudaMemcpyAsync(host_out, src, static_cast<size_t>(pl.nrows) * sizeof(spec_row_stat), cudaMemcpyDeviceToHost,
                      st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

const char* spec_status_string(spec_status status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_NONFINITE: return "non-finite logits (NaN, +inf, or no finite value in a row)";
    case SPEC_ERR_TOKEN_RANGE: return "draft token outside [0, V)";
    case SPEC_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case SPEC_ERR_UNSUPPORTED: return "problem too large for one launch (rows x segments, or shared memory)";
    case SPEC_ERR_SCRATCH_LIMIT: return "request needs more scratch than spec_verify_noalloc's fixed array";
  }
  return "unknown status";
}

uint64_t spec_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

spec_status spec_accept_histogram(const int32_t* out_num_accepted, int32_t B, int32_t K, int32_t* hist,
                                  void* stream) {
  if (B < 0 || K < 1 || K > kHistMaxK) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!out_num_accepted || !hist) return SPEC_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const int blocks = static_cast<int>(std::min<int64_t>((static_cast<int64_t>(B) + 255) / 256, 2 * sms));
  const size_t smem = static_cast<size_t>(K + 2) * sizeof(int32_t);
  spec_hist_kernel<<<blocks, 256, smem, static_cast<cudaStream_t>(stream)>>>(out_num_accepted, B, K, hist);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SPEC_OK;
}

}  // extern "C"

// ===========================================================================
// spec_verify without caller memory: the scratch is a fixed device array.

namespace {

constexpr size_t kNoAllocBytes = SPEC_NOALLOC_SCRATCH_BYTES;
// Lives in every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// The array's name is only a host-side stand-in: its device address is looked
// up once per device, with that device current, and reused.  The stream must
// belong to that device, or the kernels would be given another GPU's address.
spec_status noalloc_address(void* stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
  if (stream) {
    int sdev = -1;
    if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) return SPEC_ERR_CUDA;
    if (sdev != dev) return SPEC_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SPEC_ERR_CUDA;
    g_noalloc_addr[dev] = ptr;
  }
  *out = g_noalloc_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                           const int32_t* draft_tokens, const double* uniforms,
                                           const spec_params* params, int32_t* out_tokens,
                                           int32_t* out_num_accepted) {
  if (!params) return SPEC_ERR_INVALID_ARG;
  spec_params p = *params;
  p.workspace = nullptr;
  p.workspace_bytes = 0;
  const size_t need = spec_verify_workspace_size(&p);
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (need > kNoAllocBytes) return SPEC_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const spec_status s = noalloc_address(p.stream, &scratch);
  if (s != SPEC_OK) return s;
  p.workspace = scratch;
  p.workspace_bytes = kNoAllocBytes;
  return spec_verify(target_logits, draft_logits, draft_tokens, uniforms, &p, out_tokens, out_num_accepted);
}
