#pragma once
// spec_kernels.cuh -- the device code of libspecverify: every kernel template and
// the device functions they share.  Each kernel translation unit (kernel_unit.cu,
// compiled once per kernel group) and the host unit (spec_verify.cu) include it;
// a unit compiles only the kernels it instantiates.
//
// Operation: "Speculative Decoding" (roadtointelligence.com), section "Draft,
// then verify", steps 1-4; filters before rejection sampling per the
// paperlayer.ai summary of "Accelerating Large Language Model Decoding with
// Speculative Sampling", section "Speculative Sampling"; greedy as argmax per
// the FDE Interviews breakdown of that paper, section "01 The paper in one
// minute".
//
// Two paths, picked per call on the host; neither has a thread block wait for
// another (completion is detected by self-resetting counters, never by
// spinning).
//
//   * spec_stream_kernel, one launch per call: rows whose starts are 16-byte
//     aligned (ragged batches included), greedy, top-k with k <= 64, or top-p
//     alone.  A persistent grid of four 128-thread CTAs per SM takes whole
//     rows in order.  Each warp keeps a ring of bulk-copy buffers full and
//     reduces its stages to a running max and first argmax; top-k and top-p
//     also keep the lane groups (six 16-byte vectors of a stage) whose max
//     reaches a rising threshold, since a row's top k elements lie in its k
//     largest groups, and top-p sums the normaliser as it streams.  At the
//     row end the groups that can hold the kept set are read back and ranked
//     (a warp sort for top-k; a counting cut over the bf16 grid, or a block
//     sort, for top-p), and the kept set (index order) and the row record are
//     written; the CTA that completes a sequence runs its accept tests and
//     final draw.  Rows it cannot settle (ties past its buffers, nuclei longer
//     than its pool, non-finite values) take the exact general path below.
//   * spec_seg_kernel + spec_row_kernel, two launches: everything else (no
//     filter, top-k > 64, unaligned rows).  The segment kernel
//     streams 24 KB segments of every row (max, first argmax, the normaliser
//     where the row needs the full sum, a candidate list above a floor); the
//     row kernel, a programmatic dependent launch, merges each row's segment
//     records and lists, sorts and cuts the pool (top-k exactly, top-p when
//     the cut lies above every segment's floor), and otherwise runs the exact
//     general path over the row in global memory: an 8-probe bracket search
//     over order-preserving keys, ending in an on-chip sort or a tie cut by
//     index.  The CTA that completes a sequence runs its epilogue.
//
// Both write the same row records (normaliser, cut, draft-token probability,
// the kept set in index order) to the caller's workspace.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <vector>

#include "spec_verify.h"

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 512;       // on-chip sort capacity == stored kept-list capacity
constexpr int kProbes = 8;      // thresholds evaluated per probe pass
constexpr int kPool = 1024;     // row candidate pool (shared memory), sorted at the row merge
constexpr int kSegCap = 256;    // candidates one segment may contribute
constexpr int kListTable = 4096; // listed entries a row merge can index (one byte each)
constexpr int kRunCap = 128;    // top-k handled by a running set in the segment kernel
constexpr size_t kCounterArea = 64 * 1024;  // workspace bytes kept zeroed between calls
constexpr int kNV = 12;         // 16-byte vectors of a segment per thread (24 KB per segment)
constexpr int kHistMaxK = 8192;  // acceptance histogram: K + 2 bins in shared memory
constexpr int kMaxPasses = 40;  // bound on probe passes (16-bit keys need <= 6, 32-bit <= 11)
constexpr unsigned FULL = 0xffffffffu;

constexpr int kFlagNonfinite = 1, kFlagToken = 2, kFlagTimeout = 4;
constexpr int kSegBad = 1, kSegOver = 2;  // segment record flags

enum { kModeVerify = 0, kModeSample = 1 };

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, bulk copy, timer

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// The thread sleeps in hardware until the phase completes or ~1 ms passes, so
// waiting warps do not spin and take no issue slots from the working ones.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Order this CTA's generic-proxy accesses of shared memory before later bulk
// copies (async proxy) into it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bounded wait for the phase with the given parity: gives up after ~2 s of wall
// time (and a hard iteration cap), so a lost copy cannot hang the GPU.
__device__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < 100000u; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > 2000000000ull) break;
  }
  return false;
}

// ---------------------------------------------------------------------------
// element formats, order-preserving keys

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

template <typename E>
struct Fmt;

template <>
struct Fmt<float> {
  static constexpr int N = 4;  // elements per 16-byte vector
  __device__ static void load(const float* s, int v, float (&x)[4]) {
    const float4 q = reinterpret_cast<const float4*>(s)[v];
    x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
  }
  __device__ static void load_global(const float* g, int v, float (&x)[4]) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(g) + v);
    x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
  }
  __device__ static float at(const float* s, int64_t e) { return s[e]; }
  // vector v of a row in global memory of length L (scalar loads at the tail or
  // when the row start is not 16-byte aligned)
  __device__ static void load_row(const float* g, int v, int L, bool aligned, float (&x)[4]) {
    const int e0 = v * 4;
    if (aligned && e0 + 4 <= L) { load_global(g, v, x); return; }
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = (e0 + j < L) ? __ldg(g + e0 + j) : -INFINITY;
  }
  // max of vector v (NaN-propagating) and whether it holds a NaN
  __device__ static float vec_max(const float* s, int v, bool& nan) {
    const float4 q = reinterpret_cast<const float4*>(s)[v];
    float a, b, r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(a) : "f"(q.x), "f"(q.y));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(b) : "f"(q.z), "f"(q.w));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    nan = r != r;
    return r;
  }
  __device__ static float at_global(const float* g, int64_t e) { return __ldg(g + e); }
  // order-preserving key over the data's own grid (32-bit for fp32)
  __device__ static uint32_t key(float f) {
    const uint32_t b = __float_as_uint(f + 0.0f);  // -0 -> +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  __device__ static float val(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
  }
  __device__ static float round_to_grid(float f) { return f; }
};

template <>
struct Fmt<uint16_t> {  // bf16 carried as raw bits
  static constexpr int N = 8;
  __device__ static void unpack(const uint4 q, float (&x)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static void load(const uint16_t* s, int v, float (&x)[8]) {
    unpack(reinterpret_cast<const uint4*>(s)[v], x);
  }
  __device__ static void load_global(const uint16_t* g, int v, float (&x)[8]) {
    unpack(__ldg(reinterpret_cast<const uint4*>(g) + v), x);
  }
  __device__ static float at(const uint16_t* s, int64_t e) { return bf16_bits_to_float(s[e]); }
  __device__ static void load_row(const uint16_t* g, int v, int L, bool aligned, float (&x)[8]) {
    const int e0 = v * 8;
    if (aligned && e0 + 8 <= L) { load_global(g, v, x); return; }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      x[j] = (e0 + j < L) ? bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(g) + e0 + j)) : -INFINITY;
  }
  // max of vector v (NaN-propagating, on packed bf16 pairs) and whether it holds a NaN
  __device__ static float vec_max(const uint16_t* s, int v, bool& nan) {
    const uint4 q = reinterpret_cast<const uint4*>(s)[v];
    __nv_bfloat162 a, b, c, d;
    memcpy(&a, &q.x, 4);
    memcpy(&b, &q.y, 4);
    memcpy(&c, &q.z, 4);
    memcpy(&d, &q.w, 4);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    uint32_t mw;
    memcpy(&mw, &m, 4);
    const float lo = __uint_as_float(mw << 16), hi = __uint_as_float(mw & 0xffff0000u);
    nan = (lo != lo) || (hi != hi);
    return fmaxf(lo, hi);
  }
  __device__ static float at_global(const uint16_t* g, int64_t e) {
    return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(g) + e));
  }
  // 16-bit order-preserving key of a bf16 value (f must lie on the bf16 grid)
  __device__ static uint32_t key(float f) {
    const uint32_t h = __float_as_uint(f + 0.0f) >> 16;
    return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
  }
  __device__ static float val(uint32_t k) {
    const uint32_t h = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
    return bf16_bits_to_float(h);
  }
  // a probe threshold only has to lie on the grid: truncate to bf16
  __device__ static float round_to_grid(float f) { return __uint_as_float(__float_as_uint(f) & 0xffff0000u); }
};

// 32-bit order-preserving key of any float, for the on-chip sort
__device__ __forceinline__ uint32_t okey32(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey32_val(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// weight of one logit relative to the row max m; c = log2(e)/T
// 2^x by the hardware approximation (relative error below 2^-22; results
// below 2^-126 flush to zero)
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float wexp(float l, float m, float c) { return ex2f((l - m) * c); }

// ---------------------------------------------------------------------------
// float-float ("double-single") sums.  GB300 runs FP64 at a small fraction of
// its FP32 rate, so running totals, prefix sums and block reductions keep a
// (hi, lo) pair of floats: Knuth's TwoSum for additions and an FMA-based
// TwoProduct for scaling give ~48-bit significands on the FP32 pipes.  Doubles
// appear only in single-thread spots (the accept test, record fields).
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff(float x) { return FF{x, 0.0f}; }
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  float e = (a.hi - (s - bb)) + (b.hi - bb);  // exact rounding error of s
  e += a.lo + b.lo;
  const float hi = s + e;
  return FF{hi, e - (hi - s)};
}
__device__ __forceinline__ FF ff_add(FF a, float b) { return ff_add(a, ff(b)); }
__device__ __forceinline__ FF ff_sub(FF a, FF b) { return ff_add(a, FF{-b.hi, -b.lo}); }
__device__ __forceinline__ FF ff_mul(FF a, float b) {
  const float p = a.hi * b;
  float e = fmaf(a.hi, b, -p);  // exact rounding error of p
  e = fmaf(a.lo, b, e);
  const float hi = p + e;
  return FF{hi, e - (hi - p)};
}
__device__ __forceinline__ bool ff_lt(FF a, FF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ double ff_to_d(FF a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }
__device__ __forceinline__ FF ff_from_d(double d) {
  const float hi = static_cast<float>(d);
  return FF{hi, static_cast<float>(d - static_cast<double>(hi))};
}
__device__ __forceinline__ FF shfl_up_ff(FF v, int o) {
  return FF{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

// ---------------------------------------------------------------------------
// kernel arguments and shared scratch

// What one segment leaves for its row's merge.
struct SegRec {
  float m;          // segment max (NaN / +inf: see flags)
  int32_t argmax;   // first index of m in the row
  float z_hi, z_lo; // sum of 2^((l - m) c) over the segment (when the row needs it)
  float theta;      // candidate floor: every finite element >= theta was a candidate
  float kth;        // top-k: the segment's k-th largest value (-inf if it has fewer)
  int32_t ncand;    // listed candidates (<= kSegCap; top-k: the segment's top k)
  int32_t flags;    // kSegBad, kSegOver
  int32_t off;      // merge scratch: offset of this segment's candidates in the pool
  int32_t pad_[3];
};

struct KArgs {
  const void* tgt;
  const void* drf;
  int64_t tgt_seq, tgt_row, drf_seq, drf_row;  // element strides
  const int32_t* tokens;                       // verify [B, K]
  const double* u;                             // verify [B, K+1], sample [B, K]
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* status;
  unsigned long long* tickets;  // counter area: [B] sequences, [nrows] rows, [1] work counter
  spec_row_stat* rows;  // [nrows]
  int32_t* list_idx;    // [nrows * kCap]
  float* list_w;        // [nrows * kCap]
  SegRec* segs;         // [nrows * nseg]
  uint2* seg_cand;      // [nrows * nseg * kSegCap]: (row index, logit bits)
  int B, K, V, R;       // R rows per sequence
  int S, nseg, nrows;   // S elements per segment (a multiple of the vector width)
  uint32_t nseg_m, nseg_s;  // n / nseg == (umulhi(n, m) + n) >> s for 0 <= n < 2^31
  uint32_t rows_m, rows_s;  // the same for rows per sequence (verify: R, sample: K)
  int seg_bytes;        // bytes of one segment buffer in shared memory
  int mode, greedy, top_k, aligned;
  int fused;            // verify with K = 1 whose draft token is drawn in the same call
  const double* u_draft;  // fused: [B] uniforms of the draft draws
  int32_t* out_draft;     // fused: [B] the drawn draft tokens (tokens aliases it)
  const int2* row_map;  // ragged verify: [nrows] {sequence, position | K_b << 16} (NULL: R rows each)
  int need_z;           // segments sum the normaliser (no filter, or top-p without top-k)
  int filt, n0;         // segments list candidates; theta is the n0-th thread maximum
  float top_p, c, temp;
};

struct Slot {  // values published by exchange()
  FF d[kProbes + kWarps + 4];
  int32_t i[kProbes + kWarps + 4];
};

struct alignas(128) Scratch {
  uint64_t bar[2];     // completion of each segment buffer's bulk copy
  int32_t items[4];    // item of iteration k at [k & 3]; nitems = none
  int32_t issued[2];   // a bulk copy is in flight into the buffer
  Slot slot[2];
  // block-level reduction scratch
  float wf[kWarps];
  int32_t wi[kWarps];
  int32_t wi2[kWarps];
  FF wd[kWarps];
  int32_t pcnt[kProbes][kWarps];
  float pmass[kProbes][kWarps];
  FF wtot[kWarps];
  // segment phase
  alignas(16) float tmax[kThreads];  // per-thread maxima (read as float4)
  float theta, kth;
  int32_t seg_n, last;
  int32_t seg_cnt[2];   // candidates of items k with k & 1 == 0, 1
  int32_t run_n[2];     // keys in each half of the running top-k set
  float run_theta[2];   // its k-th value once it holds k keys, else -inf
  // the row being merged
  unsigned long long row_bound;  // largest key a list head left out (0: none)
  FF row_z;
  float row_m, row_theta, row_kth;
  int32_t row_argmax, row_flags, row_over, pool_n;
  FF bd[kProbes + 4];
  int32_t bi[kProbes + 8];
  // candidates of the general path; the draft's kept list in the epilogue
  alignas(16) int32_t cand_idx[kCap];  // segment kernel: kSegCap 64-bit candidate keys
  alignas(8) float cand_val[kCap];    // segment kernel: the running top-k set, 2 x kRunCap keys
};

// Sort keys of the row merge (in the consumed segment buffer, after the pool).
struct SortBuf {
  unsigned long long* skey;  // [kPool]
  uint8_t* segof;            // [kListTable]: the row merge's entry -> segment table
};
static_assert(sizeof(Scratch) <= 8192, "shared scratch grew past its budget");
static_assert(kCap % kThreads == 0 && kPool % kThreads == 0, "lists are split evenly over the threads");
static_assert(kSegCap * 8 <= kCap * 4, "a segment's candidate keys are staged in cand_idx");
static_assert(2 * kRunCap * 8 <= kCap * 4, "the running top-k set lives in cand_val");
static_assert(sizeof(SegRec) % 16 == 0, "segment records are moved as 16-byte words");
static_assert(sizeof(Slot) % sizeof(uint32_t) == 0, "slots are copied as 32-bit words");
static_assert(kThreads * sizeof(SegRec) <= kPool * sizeof(unsigned long long),
              "a tile of segment records is staged in the sort-key buffer");
static_assert(kThreads <= 255, "the row merge's entry table stores segment numbers in one byte");

// ---------------------------------------------------------------------------
// warp / block helpers

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ int warp_incl_scan_i(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += t;
  }
  return v;
}
__device__ __forceinline__ FF warp_incl_scan_ff(FF v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF t = shfl_up_ff(v, o);
    if (lane >= o) v = ff_add(t, v);
  }
  return v;
}

// Exclusive block scan of one float-float per thread (fixed order); *total gets
// the block total.  Uses sm.wd.
__device__ FF block_excl_scan_ff(FF v, FF* total, Scratch& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const FF incl = warp_incl_scan_ff(v, lane);
  FF excl = shfl_up_ff(incl, 1);
  if (lane == 0) excl = ff(0.0f);
  if (lane == 31) sm.wd[warp] = incl;
  __syncthreads();
  FF before = ff(0.0f), tot = ff(0.0f);
  for (int w = 0; w < kWarps; ++w) {
    if (w == warp) before = tot;
    tot = ff_add(tot, sm.wd[w]);
  }
  __syncthreads();
  *total = tot;
  return ff_add(before, excl);
}

// Exclusive block scan of one int per thread; *total gets the block total.
// Uses sm.wi.
__device__ int block_excl_scan_i(int v, int* total, Scratch& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan_i(v, lane);
  if (lane == 31) sm.wi[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += sm.wi[w];
    tot += sm.wi[w];
  }
  __syncthreads();
  *total = tot;
  return before + incl - v;
}

// Iterate a warp's contiguous segment of n elements held as N-element vectors.
// One iteration = 32 consecutive vectors, one per lane.  The loop is
// warp-uniform: f(x, first_elem, nvalid) runs on every lane each iteration
// (nvalid = 0 for lanes past the end, whose x is -inf).  U iterations' loads are
// issued together before any is processed (memory-level parallelism for global
// loads); the iterations themselves, and their order, do not depend on U.
template <int N, int U = 1, typename Load, typename F>
__device__ __forceinline__ void for_warp_segment(int n, int warp, int lane, Load load, F f) {
  const int nvec = (n + N - 1) / N;
  const int vpw = (nvec + kWarps - 1) / kWarps;
  const int vb = min(nvec, warp * vpw), ve = min(nvec, vb + vpw);
  for (int base = vb; base < ve; base += 32 * U) {
    float x[U][N];
    int nvalid[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = base + 32 * u + lane;
      nvalid[u] = 0;
      if (v < ve) {
        load(v, x[u]);
        nvalid[u] = min(N, n - v * N);
      } else {
#pragma unroll
        for (int j = 0; j < N; ++j) x[u][j] = -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + 32 * u < ve) f(x[u], (base + 32 * u + lane) * N, nvalid[u]);
  }
}

// Ordered weights: wl(v, x, nvalid) turns vector v's values x into weights in
// place (entries j >= nvalid must become 0).  Per warp, running (float-float) +=
// per-iteration warp total (float, xor tree) of each lane's per-vector sum
// (float, element order).  warp_ordered_draw repeats exactly this arithmetic,
// so a total and a later scan of the same weights agree bit for bit.
template <int N, int U = 1, typename Load, typename WL>
__device__ FF warp_ordered_total(int n, int warp, int lane, Load load, WL wl) {
  FF running = ff(0.0f);
  for_warp_segment<N, U>(n, warp, lane, load, [&](float (&x)[N], int e0, int nvalid) {
    wl(x, e0, nvalid);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) s += x[j];
    running = ff_add(running, warp_sum_f(s));
  });
  return running;
}

// The scan half: within a warp segment whose ordered total starts at `base`,
// find the smallest element index e with target < base + cumsum(e).  With
// `overflow` (target beyond every total) the last element with positive weight
// is returned instead.  Returns the segment-local element index on all lanes.
template <int N, int U = 1, typename Load, typename WL>
__device__ int warp_ordered_draw(int n, int warp, int lane, Load load, WL wl, FF target, FF base,
                                 bool overflow) {
  FF running = base;
  int found = -1, last_pos = -1;
  bool done = false;
  for_warp_segment<N, U>(n, warp, lane, load, [&](float (&x)[N], int e0, int nvalid) {
    if (done) return;  // warp-uniform
    wl(x, e0, nvalid);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      s += x[j];
      if (x[j] > 0.0f) last_pos = max(last_pos, e0 + j);
    }
    const float it = warp_sum_f(s);
    if (!overflow && ff_lt(target, ff_add(running, it))) {
      const FF incl = warp_incl_scan_ff(ff(s), lane);
      const unsigned hit = __ballot_sync(FULL, ff_lt(target, ff_add(running, incl)));
      int tok = -1;
      if (hit) {
        const int hl = __ffs(hit) - 1;
        if (lane == hl) {
          FF c = ff_add(running, ff_sub(incl, ff(s)));
          int lastp = -1;
          for (int j = 0; j < N; ++j) {
            if (x[j] > 0.0f) {
              lastp = e0 + j;
              c = ff_add(c, x[j]);
              if (ff_lt(target, c)) { tok = e0 + j; break; }
            }
          }
          if (tok < 0) tok = lastp;
        }
        tok = __shfl_sync(FULL, tok, hl);
      } else {  // rounding between the tree and the scan: last positive of the iteration
        int lp = -1;
#pragma unroll
        for (int j = 0; j < N; ++j)
          if (x[j] > 0.0f) lp = e0 + j;
        tok = warp_max_i(lp);
      }
      found = tok;
      done = true;
    }
    running = ff_add(running, it);
  });
  if (!done) found = warp_max_i(last_pos);
  return found;
}

// ---------------------------------------------------------------------------
// block exchange.  Thread 0 (or one lane) fills sm.slot[C.ph]; exchange() is a
// block barrier after which every thread may read that slot, until the next
// exchange().  Slots alternate, so the next writer never races a late reader.
// The selection code below is written against this interface; here every
// reduction is within one CTA (cs = 1, rank = 0).

struct Local {
  static constexpr int cs = 1, rank = 0;
  int ph = 0;
  __device__ Slot& mine(Scratch& sm) { return sm.slot[ph]; }
  __device__ const Slot* exchange(Scratch& sm) {
    const int p = ph;
    __syncthreads();
    ph ^= 1;
    return &sm.slot[p];
  }
};

// ---------------------------------------------------------------------------
// bitonic sorts of 64-bit keys held in registers (descending).  Key i sits in
// thread i / R, slot i % R: exchanges at distance j < R stay in a thread, at
// R <= j < 32 R go through lane shuffles, and only the wider ones (block sort)
// through shared memory, stored slot-major so a warp's accesses are
// conflict-free.

__device__ __forceinline__ void cmp_desc(unsigned long long& a, unsigned long long& b, bool desc) {
  const bool sw = desc ? (a < b) : (a > b);
  const unsigned long long x = sw ? b : a, y = sw ? a : b;
  a = x;
  b = y;
}

// One in-thread stage (k, J) for the keys of thread t (J < R, so slot r pairs
// with slot r | J; J is a compile-time constant so the keys stay in registers).
template <int R, int J>
__device__ __forceinline__ void sort_stage_regs_j(unsigned long long (&key)[R], int t, int k) {
#pragma unroll
  for (int r = 0; r < R; ++r)
    if ((r & J) == 0) cmp_desc(key[r], key[r | J], ((t * R + r) & k) == 0);
}
template <int R>
__device__ __forceinline__ void sort_stage_regs(unsigned long long (&key)[R], int t, int k, int j) {
  if (j == 1) {
    if constexpr (R > 1) sort_stage_regs_j<R, 1>(key, t, k);
  } else if (j == 2) {
    if constexpr (R > 2) sort_stage_regs_j<R, 2>(key, t, k);
  } else if (j == 4) {
    if constexpr (R > 4) sort_stage_regs_j<R, 4>(key, t, k);
  }
  static_assert(R == 1 || R == 2 || R == 4 || R == 8, "keys per thread: 1, 2, 4 or 8");
}
template <int R>
__device__ __forceinline__ void sort_stage_lanes(unsigned long long (&key)[R], int t, int k, int j) {
  const int lx = j / R;
  const bool lower = (t & lx) == 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const unsigned long long o = __shfl_xor_sync(FULL, key[r], lx);
    const bool keep_max = (((t * R + r) & k) == 0) == lower;
    key[r] = keep_max ? (key[r] > o ? key[r] : o) : (key[r] < o ? key[r] : o);
  }
}

// kThreads * R keys over the whole block; xbuf holds kThreads * R keys.
template <int R>
__device__ void block_sort_keys_desc(unsigned long long (&key)[R], unsigned long long* xbuf) {
  const int t = threadIdx.x;
  for (int k = 2; k <= kThreads * R; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < R) {
        sort_stage_regs<R>(key, t, k, j);
      } else if (j < 32 * R) {
        sort_stage_lanes<R>(key, t, k, j);
      } else {
        const int tx = j / R;
        const bool lower = (t & tx) == 0;
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r) xbuf[r * kThreads + t] = key[r];
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const unsigned long long o = xbuf[r * kThreads + (t ^ tx)];
          const bool keep_max = (((t * R + r) & k) == 0) == lower;
          key[r] = keep_max ? (key[r] > o ? key[r] : o) : (key[r] < o ? key[r] : o);
        }
      }
    }
  __syncthreads();
}

// Float-float sum over a warp (xor butterfly: every lane gets the same total).
__device__ __forceinline__ FF warp_sum_ff(FF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = ff_add(v, FF{__shfl_xor_sync(FULL, v.hi, o), __shfl_xor_sync(FULL, v.lo, o)});
  return v;
}

// Sort key (value desc, index asc) of a logit: larger keys first.
__device__ __forceinline__ unsigned long long sort_key(float v, int idx);

// ---------------------------------------------------------------------------
// per-row state

struct RowInfo {
  int b, t, is_target, job;
  int kb, first, nr;  // verify: the sequence's draft length, first row and row count
  int64_t row_off;  // element offset of the row from its tensor base
  int tok;          // draft token at this row (verify, t < K), else -1
};

template <typename E>
struct RowCtx {
  const E* g;   // row in global memory
  const E* sl;  // the data the passes read: the chunk in shared memory, or the row
  int s0, L;    // first row index held in sl, and length
  float m, c;
  int gsrc;     // sl is the row in global memory (general path of a row merge)
  int aligned;  // global row start is 16-byte aligned
};

// The kept set as a prefix of the (logit desc, index asc) order:
// x is kept iff l > tv, or l == tv and x <= ti.
struct Cut {
  float tv;
  int ti;
  __device__ bool keep(float l, int x) const { return l > tv || (l == tv && x <= ti); }
};
__device__ __forceinline__ Cut cut_all() { return Cut{-INFINITY, INT_MAX}; }

template <typename E>
__device__ __forceinline__ auto row_loader(const RowCtx<E>& rc) {
  return [&rc](int v, float (&x)[Fmt<E>::N]) {
    if (rc.gsrc) Fmt<E>::load_row(rc.sl, v, rc.L, rc.aligned != 0, x);
    else Fmt<E>::load(rc.sl, v, x);
  };
}

// ---- probe pass: counts / masses of elements >= each threshold ----------------
// thr[0] > thr[1] > ... > thr[np-1]; restricted to `rcut` when `restricted`.
// The CTA's totals are returned in cnt_out / mass_out (all threads).
template <typename E>
__device__ void probe_pass(const RowCtx<E>& rc, Scratch& sm, Local& C, const float (&thr)[kProbes], int np,
                           bool with_mass, bool restricted, Cut rcut, int (&cnt_out)[kProbes],
                           FF (&mass_out)[kProbes]) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int cnt[kProbes];
  float mass[kProbes];
#pragma unroll
  for (int j = 0; j < kProbes; ++j) { cnt[j] = 0; mass[j] = 0.0f; }
  const float lowest = thr[np - 1];
  for_warp_segment<N, 2>(rc.L, warp, lane, row_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
#pragma unroll
    for (int j = 0; j < N; ++j) {
      if (j < nvalid && x[j] >= lowest) {
        if (restricted && !rcut.keep(x[j], rc.s0 + e0 + j)) continue;
        const float w = with_mass ? wexp(x[j], rc.m, rc.c) : 0.0f;
#pragma unroll
        for (int p = 0; p < kProbes; ++p)
          if (p < np && x[j] >= thr[p]) { cnt[p] += 1; mass[p] += w; }
      }
    }
  });
#pragma unroll
  for (int p = 0; p < kProbes; ++p) {
    cnt[p] = warp_sum_i(cnt[p]);
    mass[p] = warp_sum_f(mass[p]);
    if (lane == 0) { sm.pcnt[p][warp] = cnt[p]; sm.pmass[p][warp] = mass[p]; }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Slot& s = C.mine(sm);
    for (int p = 0; p < np; ++p) {
      int ct = 0;
      FF ms = ff(0.0f);
      for (int w = 0; w < kWarps; ++w) { ct += sm.pcnt[p][w]; ms = ff_add(ms, sm.pmass[p][w]); }
      s.i[p] = ct;
      s.d[p] = ms;
    }
  }
  const Slot* mir = C.exchange(sm);
  if (threadIdx.x == 0) {
    for (int p = 0; p < np; ++p) { sm.bi[p] = 0; sm.bd[p] = ff(0.0f); }
    for (int r = 0; r < C.cs; ++r) {
      const Slot* s = (&mir[r]);
      for (int p = 0; p < np; ++p) { sm.bi[p] += s->i[p]; sm.bd[p] = ff_add(sm.bd[p], s->d[p]); }
    }
  }
  __syncthreads();
  for (int p = 0; p < kProbes; ++p) {
    cnt_out[p] = (p < np) ? sm.bi[p] : 0;
    mass_out[p] = (p < np) ? sm.bd[p] : ff(0.0f);
  }
  __syncthreads();
}

// ---- count per warp of elements satisfying pred ------------------------------
template <typename E, typename P>
__device__ int warp_count(const RowCtx<E>& rc, int warp, int lane, P pred) {
  constexpr int N = Fmt<E>::N;
  int c = 0;
  for_warp_segment<N, 2>(rc.L, warp, lane, row_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (j < nvalid && pred(x[j], rc.s0 + e0 + j)) ++c;
  });
  return warp_sum_i(c);
}

// ---- ordered compaction of elements satisfying pred (index order) ------------
// emit(pos, l, x) runs for the pos-th selected element of this CTA's slice.
// Returns this CTA's count.
template <typename E, typename P, typename Emit>
__device__ int cta_ordered_compact(const RowCtx<E>& rc, Scratch& sm, P pred, Emit emit) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wc = warp_count<E>(rc, warp, lane, pred);
  if (lane == 0) sm.wi[warp] = wc;
  __syncthreads();
  int off = 0, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) off += sm.wi[w];
    total += sm.wi[w];
  }
  __syncthreads();
  int running = off;
  for_warp_segment<N, 2>(rc.L, warp, lane, row_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
    int c = 0;
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (j < nvalid && pred(x[j], rc.s0 + e0 + j)) ++c;
    const int incl = warp_incl_scan_i(c, lane);
    int pos = running + incl - c;
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (j < nvalid && pred(x[j], rc.s0 + e0 + j)) emit(pos++, x[j], rc.s0 + e0 + j);
    running += __shfl_sync(FULL, incl, 31);
  });
  return total;
}

// ---- helpers over the gathered candidate list --------------------------------

__device__ __forceinline__ unsigned long long sort_key(float v, int idx) {
  return (static_cast<unsigned long long>(okey32(v)) << 32) | (0xffffffffu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ float skey_val(unsigned long long k) {
  return okey32_val(static_cast<uint32_t>(k >> 32));
}
__device__ __forceinline__ int skey_idx(unsigned long long k) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
}

// Ordered draw over n list entries (index order), weights wf(i) (float, >= 0),
// prefix sums in float-float: smallest i with u*R < cumsum(i); overflow -> last
// positive entry.  Block-wide; returns the entry position on all threads, or -1
// if R == 0.
template <typename WF>
__device__ int list_ordered_draw(int n, double u, Scratch& sm, WF wf) {
  constexpr int G = kCap / kThreads;  // n <= kCap: G consecutive entries per thread
  const int b0 = static_cast<int>(threadIdx.x) * G;
  float w[G];
  FF run = ff(0.0f);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    w[g] = (b0 + g < n) ? wf(b0 + g) : 0.0f;
    run = ff_add(run, w[g]);
  }
  FF total;
  const FF excl = block_excl_scan_ff(run, &total, sm);
  if (threadIdx.x == 0) {
    sm.bi[0] = INT_MAX;
    sm.bi[1] = -1;
    sm.bd[0] = ff_from_d(u * ff_to_d(total));
  }
  __syncthreads();
  int r = -1;
  if (total.hi > 0.0f) {
    const FF target = sm.bd[0];
    FF c = excl;
    int lastpos = -1;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const FF before = c;
      c = ff_add(c, w[g]);
      if (w[g] > 0.0f) {
        lastpos = b0 + g;
        if (ff_lt(target, c) && !ff_lt(target, before)) atomicMin(&sm.bi[0], b0 + g);
      }
    }
    if (lastpos >= 0) atomicMax(&sm.bi[1], lastpos);
    __syncthreads();
    r = (sm.bi[0] != INT_MAX) ? sm.bi[0] : sm.bi[1];
  }
  __syncthreads();
  return r;
}

// Bracket [lo, hi) over data keys: pred(lo) holds, pred(hi) fails; counts and
// masses are of the elements with key >= lo (resp. >= hi), restricted to rcut.
struct Bracket {
  uint32_t lo, hi;
  int cnt_lo, cnt_hi;
  FF mass_lo, mass_hi;
};

// The CTA's candidates sit at cand_*[0 .. n) in index order; make them visible
// to the whole CTA and return n.
__device__ int rank0_collect(Scratch& sm, Local& C, int n) {
  C.exchange(sm);
  return n;
}

// ---- exact cut ----------------------------------------------------------------


// Narrow `br` until cnt_lo <= cap (sortable on chip) or hi == lo + 1 (one key
// value).  pred = (mass_mode ? mass >= need_mass : count >= need_cnt).  Unless
// `probed` (a first pass already probed near the max), the first probes sit at
// m - W*scale; later ones split [lo, hi) evenly in key space.
template <typename E>
__device__ Bracket bracket_search(const RowCtx<E>& rc, Scratch& sm, Local& C, bool mass_mode, int need_cnt,
                                  FF need_mass, float scale, bool restricted, Cut rcut, Bracket br,
                                  bool probed, int cap) {
  const float W[kProbes] = {0.5f, 1.f, 2.f, 3.f, 4.f, 6.f, 8.f, 16.f};
  for (int pass = probed ? 1 : 0; pass < kMaxPasses; ++pass) {
    if (br.cnt_lo <= cap || br.hi - br.lo <= 1) break;
    uint32_t keys[kProbes];  // ascending, strictly inside (lo, hi)
    int np = 0;
    const uint32_t span = br.hi - br.lo - 1;
    if (span <= kProbes) {
      for (uint32_t k = br.lo + 1; k < br.hi; ++k) keys[np++] = k;
    } else if (pass == 0) {
      uint32_t prev = br.lo;
      for (int j = kProbes - 1; j >= 0; --j) {  // widest window first -> ascending keys
        const float t = Fmt<E>::round_to_grid(rc.m - W[j] * scale);
        uint32_t k = (t == t && t > -INFINITY) ? Fmt<E>::key(t) : prev + 1;
        if (k <= prev) k = prev + 1;
        if (k >= br.hi) break;
        keys[np++] = k;
        prev = k;
      }
    } else {
      for (int j = 1; j <= kProbes; ++j) {
        const uint32_t k =
            br.lo + static_cast<uint32_t>((static_cast<uint64_t>(span + 1) * static_cast<uint64_t>(j)) / (kProbes + 1));
        if (k > br.lo && k < br.hi && (np == 0 || k > keys[np - 1])) keys[np++] = k;
      }
    }
    if (np == 0) break;
    float thr[kProbes];
#pragma unroll
    for (int j = 0; j < kProbes; ++j) thr[j] = (j < np) ? Fmt<E>::val(keys[np - 1 - j]) : 0.0f;
    int cnt[kProbes];
    FF mass[kProbes];
    probe_pass<E>(rc, sm, C, thr, np, mass_mode, restricted, rcut, cnt, mass);
    // thr[j] is keys[np-1-j]: walk from the largest key down
    int first_true = -1;
    for (int j = 0; j < np; ++j) {
      const bool ok = mass_mode ? !ff_lt(mass[j], need_mass) : (cnt[j] >= need_cnt);
      if (ok) { first_true = j; break; }
    }
    if (first_true >= 0) {
      br.lo = keys[np - 1 - first_true];
      br.cnt_lo = cnt[first_true];
      br.mass_lo = mass[first_true];
      if (first_true > 0) {
        br.hi = keys[np - first_true];
        br.cnt_hi = cnt[first_true - 1];
        br.mass_hi = mass[first_true - 1];
      }
    } else {
      br.hi = keys[0];
      br.cnt_hi = cnt[np - 1];
      br.mass_hi = mass[np - 1];
    }
  }
  return br;
}

// Gather every element >= lo_val (and kept by rcut) into the candidate
// list, in index order; returns the count on every thread.
template <typename E>
__device__ int gather_candidates(const RowCtx<E>& rc, Scratch& sm, Local& C, float lo_val, bool restricted,
                                 Cut rcut) {
  auto pred = [&](float l, int x) { return l >= lo_val && (!restricted || rcut.keep(l, x)); };
  const int n = cta_ordered_compact<E>(rc, sm, pred, [&](int pos, float l, int x) {
    if (pos < kCap) { sm.cand_idx[pos] = x; sm.cand_val[pos] = l; }
  });
  return rank0_collect(sm, C, n);
}

// The whole CTA: sort n candidates (idx[], val[], index order) by (logit desc,
// index asc), keep the first need_k (need_k > 0), then the shortest prefix whose
// mass reaches top_p * Z (Z = the kept top-k mass, or z_for_p without top-k).
// Weights are 2^((l - m) c).  Returns in out: the cut (value, index), the kept
// count, Z_f (mass of the kept prefix), the mass of the whole sorted list, and
// whether the top-p crossing was reached within the list.
struct CutResult {
  float tv;
  int ti;
  int nkeep;
  FF zf;
  FF total;
  int reached;
};

__device__ CutResult sort_and_cut(float m, float c, const int32_t* idx, const float* val, int n, SortBuf sb,
                                  int need_k, float top_p, FF z_for_p, Scratch& sm) {
  constexpr int GMAX = kPool / kThreads;
  unsigned long long* skey = sb.skey;
  // sort in registers (zero keys pad, and sort last), then lay the keys out
  // in order for the prefix and the cut
  if (n <= 2 * kThreads) {
    unsigned long long key[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = threadIdx.x * 2 + r;
      key[r] = (i < n) ? sort_key(val[i], idx[i]) : 0ull;
    }
    block_sort_keys_desc<2>(key, skey);
#pragma unroll
    for (int r = 0; r < 2; ++r) skey[threadIdx.x * 2 + r] = key[r];
  } else if (n <= 4 * kThreads) {
    unsigned long long key[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = threadIdx.x * 4 + r;
      key[r] = (i < n) ? sort_key(val[i], idx[i]) : 0ull;
    }
    block_sort_keys_desc<4>(key, skey);
#pragma unroll
    for (int r = 0; r < 4; ++r) skey[threadIdx.x * 4 + r] = key[r];
  } else {
    unsigned long long key[kPool / kThreads];
#pragma unroll
    for (int r = 0; r < kPool / kThreads; ++r) {
      const int i = threadIdx.x * (kPool / kThreads) + r;
      key[r] = (i < n) ? sort_key(val[i], idx[i]) : 0ull;
    }
    block_sort_keys_desc<kPool / kThreads>(key, skey);
#pragma unroll
    for (int r = 0; r < kPool / kThreads; ++r) skey[threadIdx.x * (kPool / kThreads) + r] = key[r];
  }
  __syncthreads();
  const int nk = (need_k > 0) ? min(need_k, n) : n;
  // inclusive prefix of the weights in sorted order: G consecutive entries per
  // thread, kept in registers
  const int G = max(1, (nk + kThreads - 1) / kThreads);
  const int b0 = threadIdx.x * G;
  FF pre[GMAX];
  FF run = ff(0.0f);
#pragma unroll
  for (int g = 0; g < GMAX; ++g) {
    const int i = b0 + g;
    if (g < G && i < nk) run = ff_add(run, wexp(skey_val(skey[i]), m, c));
    pre[g] = run;
  }
  FF total;
  const FF excl = block_excl_scan_ff(run, &total, sm);
  if (threadIdx.x == 0) sm.bi[2] = INT_MAX;
  __syncthreads();
  int cut = nk - 1;
  int reached = 1;
  if (top_p < 1.0f) {
    const FF zk = (need_k > 0) ? total : z_for_p;
    const FF need = ff_mul(zk, top_p);
    bool hit = false;
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
      const int i = b0 + g;
      if (!hit && g < G && i < nk && !ff_lt(ff_add(excl, pre[g]), need)) {
        atomicMin(&sm.bi[2], i);
        hit = true;
      }
    }
    __syncthreads();
    if (sm.bi[2] != INT_MAX) cut = sm.bi[2];
    else reached = 0;  // the list's mass stays below top_p * Z
  }
  // Z_f = the prefix at the cut, published by the thread that holds it
  if (threadIdx.x == cut / G) {
    FF z = ff(0.0f);
#pragma unroll
    for (int g = 0; g < GMAX; ++g)
      if (g == cut - b0) z = ff_add(excl, pre[g]);
    sm.bd[2] = z;
  }
  __syncthreads();
  CutResult r;
  r.tv = skey_val(skey[cut]);
  r.ti = skey_idx(skey[cut]);
  r.nkeep = cut + 1;
  r.zf = sm.bd[2];
  r.total = total;
  r.reached = reached;
  __syncthreads();
  return r;
}

// Tie cut: index of the c-th (1-based) element equal to tie_val (and kept by
// rcut), in index order over the row.  Same value on every thread.
template <typename E>
__device__ int tie_locate(const RowCtx<E>& rc, Scratch& sm, Local& C, float tie_val, int c, bool restricted,
                          Cut rcut) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto pred = [&](float l, int x) { return l == tie_val && (!restricted || rcut.keep(l, x)); };
  const int wc = warp_count<E>(rc, warp, lane, pred);
  if (lane == 0) sm.wi[warp] = wc;
  __syncthreads();
  if (threadIdx.x == 0) {
    Slot& s = C.mine(sm);
    for (int w = 0; w < kWarps; ++w) s.i[1 + w] = sm.wi[w];
  }
  const Slot* mir = C.exchange(sm);
  if (threadIdx.x == 0) {
    int acc = 0, fr = -1, fw = -1, kth = 0;
    for (int r = 0; r < C.cs && fr < 0; ++r)
      for (int w = 0; w < kWarps; ++w) {
        const int cw = (&mir[r])->i[1 + w];
        if (acc + cw >= c) { fr = r; fw = w; kth = c - acc; break; }
        acc += cw;
      }
    sm.bi[0] = fr;
    sm.bi[1] = fw;
    sm.bi[2] = kth;
  }
  __syncthreads();
  const int fr = sm.bi[0], fw = sm.bi[1], kth = sm.bi[2];
  __syncthreads();
  if (C.rank == fr && warp == fw) {
    int running = 0, found = -1;
    for_warp_segment<N, 2>(rc.L, warp, lane, row_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < N; ++j)
        if (j < nvalid && pred(x[j], rc.s0 + e0 + j)) ++cnt;
      const int incl = warp_incl_scan_i(cnt, lane);
      const int before = running + incl - cnt;
      if (before < kth && before + cnt >= kth) {
        int k = before;
        for (int j = 0; j < N; ++j)
          if (j < nvalid && pred(x[j], rc.s0 + e0 + j)) {
            if (++k == kth) { found = rc.s0 + e0 + j; break; }
          }
      }
      running += __shfl_sync(FULL, incl, 31);
    });
    found = warp_max_i(found);
    if (lane == 0) C.mine(sm).i[0] = found;
  }
  mir = C.exchange(sm);
  if (threadIdx.x == 0) sm.bi[3] = (fr >= 0) ? mir[fr].i[0] : INT_MAX;
  __syncthreads();
  const int idx = sm.bi[3];
  __syncthreads();
  return idx;
}

// Count and mass of the elements kept by `cut` over the row (same on every thread);
// with write_list and a kept set that fits kCap, the kept set is written in index
// order to lidx / lw.
template <typename E>
__device__ void kept_pass(const RowCtx<E>& rc, Scratch& sm, Local& C, Cut cut, bool write_list, int32_t* lidx,
                          float* lw, int* nkeep, FF* zf, int* list_len) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto pred = [&](float l, int x) { return cut.keep(l, x); };
  auto wl = [&](float (&x)[N], int e0, int nvalid) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      x[j] = (j < nvalid && cut.keep(x[j], rc.s0 + e0 + j)) ? wexp(x[j], rc.m, rc.c) : 0.0f;
  };
  const FF wt = warp_ordered_total<N>(rc.L, warp, lane, row_loader(rc), wl);
  const int wc = warp_count<E>(rc, warp, lane, pred);
  if (lane == 0) { sm.wtot[warp] = wt; sm.wi2[warp] = wc; }
  __syncthreads();
  if (threadIdx.x == 0) {
    Slot& s = C.mine(sm);
    FF t = ff(0.0f);
    int ct = 0;
    for (int w = 0; w < kWarps; ++w) { t = ff_add(t, sm.wtot[w]); ct += sm.wi2[w]; }
    s.d[0] = t;
    s.i[0] = ct;
  }
  const Slot* mir = C.exchange(sm);
  if (threadIdx.x == 0) {
    FF z = ff(0.0f);
    int total = 0, off = 0;
    for (int r = 0; r < C.cs; ++r) {
      const Slot* s = (&mir[r]);
      z = ff_add(z, s->d[0]);
      if (r < C.rank) off += s->i[0];
      total += s->i[0];
    }
    sm.bd[0] = z;
    sm.bi[0] = total;
    sm.bi[1] = off;
  }
  __syncthreads();
  const int total = sm.bi[0], off = sm.bi[1];
  *nkeep = total;
  *zf = sm.bd[0];
  *list_len = (write_list && total <= kCap) ? total : -1;
  __syncthreads();
  if (write_list && total <= kCap) {
    cta_ordered_compact<E>(rc, sm, pred, [&](int pos, float l, int x) {
      lidx[off + pos] = x;
      lw[off + pos] = wexp(l, rc.m, rc.c);
    });
  }
}

// ---------------------------------------------------------------------------

// n / d for 0 <= n < 2^31 with the host's multiplier and shift for d
__device__ __forceinline__ int fast_div(int n, uint32_t m, uint32_t s) {
  return static_cast<int>((__umulhi(static_cast<uint32_t>(n), m) + static_cast<uint32_t>(n)) >> s);
}

// The sequence of a verify row: R rows per sequence, or (ragged calls) the
// host's per-row table {b, position | K_b << 16}; a sequence's rows are its
// K_b + 1 target rows, then (sampling) its K_b draft rows.
struct SeqRows {
  int b, first, nr, kb;
};
template <bool RAG>
__device__ __forceinline__ SeqRows seq_of_row(const KArgs& a, int row) {
  SeqRows q;
  if constexpr (RAG) {
    const int2 e = __ldg(&a.row_map[row]);
    q.b = e.x;
    q.kb = e.y >> 16;
    q.first = row - (e.y & 0xffff);
    q.nr = a.greedy ? q.kb + 1 : 2 * q.kb + 1;
  } else {
    q.b = fast_div(row, a.rows_m, a.rows_s);
    q.first = q.b * a.R;
    q.nr = a.R;
    q.kb = a.K;
  }
  return q;
}

template <bool RAG>
__device__ RowInfo decode_job(const KArgs& a, int job) {
  RowInfo ri;
  ri.job = job;
  ri.tok = -1;
  if (a.mode == kModeVerify) {
    const SeqRows q = seq_of_row<RAG>(a, job);
    ri.b = q.b;
    ri.kb = q.kb;
    ri.first = q.first;
    ri.nr = q.nr;
    const int r = job - q.first;
    ri.is_target = r <= q.kb;
    ri.t = ri.is_target ? r : r - (q.kb + 1);
    ri.row_off = ri.is_target ? static_cast<int64_t>(ri.b) * a.tgt_seq + static_cast<int64_t>(ri.t) * a.tgt_row
                              : static_cast<int64_t>(ri.b) * a.drf_seq + static_cast<int64_t>(ri.t) * a.drf_row;
  } else {
    ri.b = job / a.K;
    ri.t = job % a.K;
    ri.kb = a.K;
    ri.first = ri.b * a.K;
    ri.nr = a.K;
    ri.is_target = 0;
    ri.row_off = static_cast<int64_t>(ri.b) * a.drf_seq + static_cast<int64_t>(ri.t) * a.drf_row;
  }
  return ri;
}

__device__ void set_status(const KArgs& a, int code) {
  if (a.status) atomicCAS(a.status, 0, code);
}

// ---------------------------------------------------------------------------
// final draw from full rows in global memory (no stored kept list): one CTA
// (the one that completes the sequence), over [0, V).  Residual weights
// max(0, tgt(x) - drf(x)) or, without `resid`, target weights.  Returns the token,
// or -1 if the weights sum to zero.

template <typename E>
__device__ int global_rows_draw(const KArgs& a, const E* gt, const E* gd, float mt, float md, Cut ct, Cut cd,
                                float izt, float izd, bool resid, double u, Scratch& sm) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int V = a.V;
  const bool vec = a.aligned != 0;
  // loads write the weights directly; the value array doubles as weight storage
  auto load = [&](int v, float (&x)[N]) {
    float xt[N], xd[N];
    const int e0 = v * N;
    if (vec && e0 + N <= V) {
      Fmt<E>::load_global(gt, v, xt);
      if (resid) Fmt<E>::load_global(gd, v, xd);
    } else {
#pragma unroll
      for (int j = 0; j < N; ++j) {
        xt[j] = (e0 + j < V) ? Fmt<E>::at_global(gt, e0 + j) : -INFINITY;
        xd[j] = (resid && e0 + j < V) ? Fmt<E>::at_global(gd, e0 + j) : -INFINITY;
      }
    }
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const int xi = e0 + j;
      const float wt = ct.keep(xt[j], xi) ? wexp(xt[j], mt, a.c) : 0.0f;
      if (resid) {
        const float wd = cd.keep(xd[j], xi) ? wexp(xd[j], md, a.c) : 0.0f;
        x[j] = fmaxf(0.0f, wt * izt - wd * izd);
      } else {
        x[j] = wt;
      }
    }
  };
  auto wl = [&](float (&x)[N], int, int nvalid) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (j >= nvalid) x[j] = 0.0f;
  };
  const FF wt = warp_ordered_total<N, 4>(V, warp, lane, load, wl);
  if (lane == 0) sm.wtot[warp] = wt;
  __syncthreads();
  if (threadIdx.x == 0) {
    FF total = ff(0.0f);
    for (int w = 0; w < kWarps; ++w) total = ff_add(total, sm.wtot[w]);
    const FF target = ff_from_d(u * ff_to_d(total));
    int fw = -1, lw = 0;
    FF base = ff(0.0f), cum = ff(0.0f);
    for (int w = 0; w < kWarps; ++w) {
      const FF t = sm.wtot[w];
      if (t.hi > 0.0f) lw = w;
      const FF next = ff_add(cum, t);
      if (fw < 0 && ff_lt(target, next)) { fw = w; base = cum; }
      cum = next;
    }
    const int overflow = fw < 0;
    if (overflow) fw = lw;
    sm.bi[0] = (total.hi > 0.0f) ? fw : -1;
    sm.bi[1] = overflow;
    sm.bd[0] = target;
    sm.bd[1] = base;
    sm.bi[2] = -1;
  }
  __syncthreads();
  const int fw = sm.bi[0];
  const bool overflow = sm.bi[1] != 0;
  const FF target = sm.bd[0], base = sm.bd[1];
  if (fw >= 0 && warp == fw) {
    const int e = warp_ordered_draw<N, 4>(V, warp, lane, load, wl, target, base, overflow);
    if (lane == 0) sm.bi[2] = e;
  }
  __syncthreads();
  const int tok = (fw >= 0) ? sm.bi[2] : -1;
  __syncthreads();
  return tok;
}

// ---------------------------------------------------------------------------
// verify epilogue: the CTA that completes sequence b

// Accept test of a fused call's draft token d (K = 1): the token was drawn by
// the draft row of the same call, so its probabilities under both adjusted
// rows are computed here, with the arithmetic of the row records.
template <typename E>
__device__ __noinline__ bool fused_accept(const KArgs& a, int b, int d, const spec_row_stat& rt,
                                          const spec_row_stat& rd, double u) {
  const E* gt = static_cast<const E*>(a.tgt) + static_cast<int64_t>(b) * a.tgt_seq;
  const E* gd = static_cast<const E*>(a.drf) + static_cast<int64_t>(b) * a.drf_seq;
  auto prob = [&](const E* g, const spec_row_stat& r) -> double {
    if (d < 0 || d >= a.V) return 0.0;
    const float l = Fmt<E>::at_global(g, d);
    const Cut c{__ldcg(&r.tau_val), __ldcg(&r.tau_idx)};
    if (!(c.keep(l, d) && l > -INFINITY)) return 0.0;
    return static_cast<double>(wexp(l, __ldcg(&r.m), a.c)) / __ldcg(&r.zf);
  };
  return u * prob(gd, rd) < prob(gt, rt);
}

template <typename E>
// K = this sequence's draft length (ragged: K_b <= a.K); token, uniform and
// output arrays keep the call's strides (a.K, a.K + 1), and the final draw
// takes uniform column K.
__device__ void verify_epilogue(const KArgs& a, int b, int K, int first, Scratch& sm) {
  const int KS = a.K;  // strides of the [B, K] and [B, K + 1] arrays
  const spec_row_stat* recs = a.rows + first;
  const int R = a.greedy ? K + 1 : 2 * K + 1;
  int32_t* out = a.out_tokens + static_cast<int64_t>(b) * (KS + 1);
  const int tid = threadIdx.x;
  // all row records in parallel, in one round of loads: the flags, and the
  // accept tests (one per thread; the flags decide afterwards whether they count)
  if (tid == 0) { sm.bi[12] = 0; sm.bi[13] = K; }
  __syncthreads();
  int myfl = 0;
  for (int r = tid; r < R; r += kThreads) myfl |= __ldcg(&recs[r].flags);
  {
    for (int t = tid; t < K; t += kThreads) {
      const int d = a.fused ? __ldcg(&a.out_draft[b]) : a.tokens[static_cast<int64_t>(b) * KS + t];
      bool acc;
      if (a.greedy) {
        acc = (d == __ldcg(&recs[t].argmax));
      } else if (a.fused) {
        acc = fused_accept<E>(a, b, d, recs[t], recs[K + 1 + t], a.u[static_cast<int64_t>(b) * (KS + 1) + t]);
      } else {
        // keep d_t with probability min(1, tgt/drf):  u * drf < tgt
        const double pt = __ldcg(&recs[t].p_tok);
        const double pd = __ldcg(&recs[K + 1 + t].p_tok);
        acc = a.u[static_cast<int64_t>(b) * (KS + 1) + t] * pd < pt;
      }
      if (!acc) atomicMin(&sm.bi[13], t);  // the first rejection wins
    }
  }
  if (myfl) atomicOr(&sm.bi[12], myfl);
  __syncthreads();
  const int fl = sm.bi[12], n = sm.bi[13];
  __syncthreads();
  if (fl) {
    for (int t = tid; t <= KS; t += kThreads) out[t] = -1;
    if (tid == 0) {
      a.out_n[b] = -1;
      set_status(a, (fl & kFlagToken) ? SPEC_ERR_TOKEN_RANGE
                                      : (fl & kFlagTimeout) ? SPEC_ERR_TIMEOUT : SPEC_ERR_NONFINITE);
    }
    return;
  }
  for (int t = tid; t <= KS; t += kThreads)
    out[t] = (t < n) ? (a.fused ? __ldcg(&a.out_draft[b]) : a.tokens[static_cast<int64_t>(b) * KS + t]) : -1;
  int token;
  if (a.greedy) {
    token = __ldcg(&recs[n].argmax);
  } else {
    const double u = a.u[static_cast<int64_t>(b) * (KS + 1) + K];
    const int rt = n, rd = K + 1 + n;
    const bool resid = n < K;
    const double zt = __ldcg(&recs[rt].zf);
    const double zd = resid ? __ldcg(&recs[rd].zf) : 1.0;
    const int lt = __ldcg(&recs[rt].list_len);
    const int ld = resid ? __ldcg(&recs[rd].list_len) : 0;
    const int64_t job_t = static_cast<int64_t>(first) + rt, job_d = static_cast<int64_t>(first) + rd;
    if (lt >= 0 && ld >= 0) {
      // kept sets stored: residual over the target's kept list (index order)
      const int32_t* ti = a.list_idx + job_t * kCap;
      const float* tw = a.list_w + job_t * kCap;
      // the draft's kept list goes to shared memory (the candidate arrays are free now)
      if (resid) {
        const int32_t* di = a.list_idx + job_d * kCap;
        const float* dw = a.list_w + job_d * kCap;
        for (int i = tid; i < ld; i += kThreads) { sm.cand_idx[i] = __ldcg(&di[i]); sm.cand_val[i] = __ldcg(&dw[i]); }
        __syncthreads();
      }
      auto drf_w = [&](int x) -> float {
        int lo = 0, hi = ld;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (sm.cand_idx[mid] < x) lo = mid + 1; else hi = mid;
        }
        return (lo < ld && sm.cand_idx[lo] == x) ? sm.cand_val[lo] : 0.0f;
      };
      // residual max(0, tgt - drf) with the same float arithmetic as the full-row draw
      const float izt = 1.0f / static_cast<float>(zt), izd = 1.0f / static_cast<float>(zd);
      int pos = -1;
      if (resid)
        pos = list_ordered_draw(lt, u, sm, [&](int i) {
          return fmaxf(0.0f, __ldcg(&tw[i]) * izt - drf_w(__ldcg(&ti[i])) * izd);
        });
      if (pos < 0)  // bonus row, or zero residual mass: the target row itself
        pos = list_ordered_draw(lt, u, sm, [&](int i) { return __ldcg(&tw[i]); });
      token = (pos >= 0) ? __ldcg(&ti[pos]) : -1;
    } else {
      const E* gt = static_cast<const E*>(a.tgt) + (static_cast<int64_t>(b) * a.tgt_seq + static_cast<int64_t>(rt) * a.tgt_row);
      const E* gd = resid ? static_cast<const E*>(a.drf) +
                                (static_cast<int64_t>(b) * a.drf_seq + static_cast<int64_t>(n) * a.drf_row)
                          : gt;
      const float mt = __ldcg(&recs[rt].m), md = resid ? __ldcg(&recs[rd].m) : 0.0f;
      const Cut ct{__ldcg(&recs[rt].tau_val), __ldcg(&recs[rt].tau_idx)};
      const Cut cd = resid ? Cut{__ldcg(&recs[rd].tau_val), __ldcg(&recs[rd].tau_idx)} : cut_all();
      const float izt = 1.0f / static_cast<float>(zt), izd = 1.0f / static_cast<float>(zd);
      token = -1;
      if (resid) token = global_rows_draw<E>(a, gt, gd, mt, md, ct, cd, izt, izd, true, u, sm);
      if (token < 0) token = global_rows_draw<E>(a, gt, gt, mt, mt, ct, ct, izt, izt, false, u, sm);
    }
  }
  if (tid == 0) {
    out[n] = token;
    a.out_n[b] = n;
  }
}


// ---------------------------------------------------------------------------
// row merge, run by the CTA that finishes a row's last chunk

template <typename E>
__device__ void general_cut(const KArgs& a, const RowCtx<E>& rg, Scratch& sm, Local& C, SortBuf sb, FF z,
                            Cut* cut_out, FF* zf_out, int* list_len_out, int32_t* lidx, float* lw) {
  // exact selection over the whole row in global memory (rg.gsrc): top-k by count,
  // then top-p by mass within it; ends in an on-chip sort or a tie cut by index
  const bool use_k = a.top_k > 0 && a.top_k < a.V;
  const bool use_p = a.top_p < 1.0f;
  Cut cut = cut_all();
  FF zf = z, zk = z;
  int list_len = -1;
  bool sorted = false, restricted = false, final_tie = false;
  Cut kcut = cut_all();
  CutResult res;
  int gathered = 0;
  auto fresh = [&](int cnt_all, FF mass_all) {
    Bracket br;
    br.lo = Fmt<E>::key(-INFINITY);
    br.hi = Fmt<E>::key(rg.m) + 1;
    br.cnt_lo = cnt_all;
    br.mass_lo = mass_all;
    br.cnt_hi = 0;
    br.mass_hi = ff(0.0f);
    return br;
  };
  if (use_k) {
    Bracket br = bracket_search<E>(rg, sm, C, false, a.top_k, ff(0.0f), 1.0f, false, cut_all(),
                                   fresh(a.V, ff(0.0f)), false, kCap);
    if (br.cnt_lo <= kCap) {
      gathered = gather_candidates<E>(rg, sm, C, Fmt<E>::val(br.lo), false, cut_all());
      res = sort_and_cut(rg.m, rg.c, sm.cand_idx, sm.cand_val, gathered, sb, a.top_k, use_p ? a.top_p : 1.0f,
                         ff(0.0f), sm);
      sorted = true;
    } else {
      const float tv = Fmt<E>::val(br.lo);
      kcut = Cut{tv, tie_locate<E>(rg, sm, C, tv, a.top_k - br.cnt_hi, false, cut_all())};
      restricted = true;
      if (!use_p) { cut = kcut; final_tie = true; }
    }
  }
  if (use_p && !sorted) {
    int cnt_all = a.V;
    if (restricted) {
      int ll;
      kept_pass<E>(rg, sm, C, kcut, false, nullptr, nullptr, &cnt_all, &zk, &ll);
    }
    const FF need = ff_mul(zk, a.top_p);
    const Bracket br = bracket_search<E>(rg, sm, C, true, 0, need, a.temp, restricted, kcut,
                                         fresh(cnt_all, zk), false, kCap);
    if (br.cnt_lo <= kCap) {
      gathered = gather_candidates<E>(rg, sm, C, Fmt<E>::val(br.lo), restricted, kcut);
      res = sort_and_cut(rg.m, rg.c, sm.cand_idx, sm.cand_val, gathered, sb, 0, a.top_p, zk, sm);
      sorted = true;
    } else {
      const float tv = Fmt<E>::val(br.lo);
      const float w = wexp(tv, rg.m, rg.c);
      const int ties = br.cnt_lo - br.cnt_hi;
      int c = ties;
      if (w > 0.0f) {  // smallest c with mass_hi + c * w >= need
        const FF rem = ff_sub(need, br.mass_hi);
        const float k = ceilf((rem.hi + rem.lo) / w);
        c = static_cast<int>(fminf(fmaxf(k, 1.0f), static_cast<float>(ties)));
      }
      cut = Cut{tv, tie_locate<E>(rg, sm, C, tv, c, restricted, kcut)};
      final_tie = true;
    }
  }
  if (sorted) {
    cut = Cut{res.tv, res.ti};
    zf = res.zf;
    // the kept list = the gathered candidates (index order) kept by the cut
    if (res.nkeep <= kCap) {
      constexpr int G = kCap / kThreads;  // gathered <= kCap: G consecutive entries per thread
      const int b0 = static_cast<int>(threadIdx.x) * G;
      int cnt = 0;
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (b0 + g < gathered && cut.keep(sm.cand_val[b0 + g], sm.cand_idx[b0 + g])) ++cnt;
      int tot;
      int pos = block_excl_scan_i(cnt, &tot, sm);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int i = b0 + g;
        if (i < gathered && cut.keep(sm.cand_val[i], sm.cand_idx[i])) {
          lidx[pos] = sm.cand_idx[i];
          lw[pos] = wexp(sm.cand_val[i], rg.m, rg.c);
          ++pos;
        }
      }
      list_len = tot;
      __syncthreads();
    }
  }
  if (final_tie) {
    int nk;
    kept_pass<E>(rg, sm, C, cut, true, lidx, lw, &nk, &zf, &list_len);
  }
  *cut_out = cut;
  *zf_out = zf;
  *list_len_out = list_len;
}

// Top-k streaming floor: sort the pool's keys (in a free ring slot), take the k-th
// candidate (value, index) as the floor theta, and keep exactly the pool entries
// at or above it, in their (index) order.  Later chunks only need elements above
// theta's value: their ties at that value have larger indices.
// ---------------------------------------------------------------------------
// row merge, run by the CTA that finishes a row's last segment

// Kept set (the sorted prefix skey[0, n)) written in index order: each entry's
// position is the number of kept entries with a smaller index.
__device__ void write_kept_by_index(const unsigned long long* skey, int n, float m, float c, int32_t* lidx,
                                    float* lw, Scratch& sm) {
  constexpr int G = kCap / kThreads;  // entries per thread: threadIdx.x + g * kThreads
  int32_t* kidx = sm.cand_idx;        // the indices, unpacked once
  for (int i = threadIdx.x; i < n; i += kThreads) kidx[i] = skey_idx(skey[i]);
  __syncthreads();
  // each thread ranks all its entries in one pass over the indices, four at a time
  int xi[G], pos[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int i = threadIdx.x + g * kThreads;
    xi[g] = (i < n) ? kidx[i] : INT_MIN;
    pos[g] = 0;
  }
  const int4* k4 = reinterpret_cast<const int4*>(kidx);
  const int n4 = n >> 2;
  for (int j = 0; j < n4; ++j) {
    const int4 v = k4[j];
#pragma unroll
    for (int g = 0; g < G; ++g)
      pos[g] += (v.x < xi[g]) + (v.y < xi[g]) + (v.z < xi[g]) + (v.w < xi[g]);
  }
  for (int j = n4 << 2; j < n; ++j) {
    const int v = kidx[j];
#pragma unroll
    for (int g = 0; g < G; ++g) pos[g] += (v < xi[g]) ? 1 : 0;
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int i = threadIdx.x + g * kThreads;
    if (i < n) {
      lidx[pos[g]] = xi[g];
      lw[pos[g]] = wexp(skey_val(skey[i]), m, c);
    }
  }
  __syncthreads();
}

// Fold the row's segment records into sm.row_*: max, first argmax, normaliser
// (each segment's sum rescaled to the row max, float-float, fixed order),
// flags, the largest theta and per-segment k-th value; then gather the first
// `lim` entries of every segment's list (sorted: value desc, index asc) into
// the pool, and in sm.row_bound the largest key left out of a list (0: none).
// Top-k keeps only entries >= max(kfloor, every segment's k-th value): both
// bound the row's k-th value from below.
// Records are staged a tile at a time in the sort-key buffer and folded by
// warp 0, 32 at a time.
__device__ void row_merge(const KArgs& a, int row, Scratch& sm, SortBuf sb, int32_t* pidx, float* pval, int lim,
                          float kfloor) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  SegRec* stage = reinterpret_cast<SegRec*>(sb.skey);
  const SegRec* recs = a.segs + static_cast<int64_t>(row) * a.nseg;
  const int ns = a.nseg;
  float m = -INFINITY, th = -INFINITY, kl = -INFINITY;
  int am = -1, fl = 0, total = 0;
  unsigned long long bound = 0ull;
  FF z = ff(0.0f);
  const uint2* cand = a.seg_cand + static_cast<int64_t>(row) * a.nseg * kSegCap;
  for (int t0 = 0; t0 < ns; t0 += kThreads) {
    const int nt = min(kThreads, ns - t0);
    __syncthreads();
    if (tid < nt) {
      const int4* src = reinterpret_cast<const int4*>(recs + t0 + tid);
      int4* dst = reinterpret_cast<int4*>(stage + tid);
#pragma unroll
      for (int w = 0; w < static_cast<int>(sizeof(SegRec) / 16); ++w) dst[w] = __ldcg(src + w);
    }
    __syncthreads();
    if (warp == 0) {
      for (int c0 = 0; c0 < nt; c0 += 32) {
        const int s = c0 + lane;
        const bool valid = s < nt;
        const int flags = valid ? stage[s].flags : 0;
        const bool good = valid && !(flags & kSegBad);
        const float ms = good ? stage[s].m : -INFINITY;
        const int listed = valid ? stage[s].ncand : 0;
        const int nc = min(listed, lim);
        unsigned long long bk = 0ull;
        if (listed > lim) {  // the first entry this list leaves out
          const uint2 e = __ldcg(cand + static_cast<int64_t>(t0 + s) * kSegCap + lim);
          bk = sort_key(__uint_as_float(e.y), static_cast<int>(e.x));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long ob = __shfl_xor_sync(FULL, bk, o);
          bk = ob > bk ? ob : bk;
        }
        bound = bk > bound ? bk : bound;
        const int incl = warp_incl_scan_i(nc, lane);
        if (valid) stage[s].off = total + incl - nc;
        total += __shfl_sync(FULL, incl, 31);
        fl |= static_cast<int>(__reduce_or_sync(FULL, static_cast<unsigned>(flags)));
        float cm = ms;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(FULL, cm, o));
        if (cm > m) {  // a new row max (uniform): rescale the sum so far
          if (z.hi > 0.0f) z = ff_mul(z, ex2f((m - cm) * a.c));
          m = cm;
          const unsigned hit = __ballot_sync(FULL, good && ms == cm);
          am = __shfl_sync(FULL, valid ? stage[s].argmax : -1, __ffs(hit) - 1);
        }
        FF zs = ff(0.0f);
        if (good && stage[s].z_hi > 0.0f) zs = ff_mul(FF{stage[s].z_hi, stage[s].z_lo}, ex2f((ms - m) * a.c));
        z = ff_add(z, warp_sum_ff(zs));
        float tv = good ? stage[s].theta : -INFINITY, kv = good ? stage[s].kth : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          tv = fmaxf(tv, __shfl_xor_sync(FULL, tv, o));
          kv = fmaxf(kv, __shfl_xor_sync(FULL, kv, o));
        }
        th = fmaxf(th, tv);
        kl = fmaxf(kl, kv);
      }
    }
  }
  if (tid == 0) {
    sm.row_m = m;
    sm.row_argmax = am;
    sm.row_flags = fl;
    sm.row_theta = th;
    sm.row_kth = kl;
    sm.row_bound = bound;
    sm.row_z = z;
    // the pool's segment offsets are staged for one tile only
    sm.row_over = (ns > kThreads) || (fl & kSegOver) || (a.top_k <= 0 && total > kPool);
    sm.pool_n = total;
    sm.seg_n = 0;
  }
  __syncthreads();
  // Gather the pool.  Top-k keeps only entries >= the largest per-segment k-th
  // value: the row's k-th largest is at least that, so no entry below it can
  // be kept.  Entry e of the concatenated lists belongs to the last segment
  // whose offset is <= e.  Each thread issues up to eight loads at once.
  total = sm.pool_n;  // folded by warp 0
  if (a.filt && !sm.row_over && !(sm.row_flags & kSegBad) && total <= kListTable) {
    const float floor_v = (a.top_k > 0) ? fmaxf(sm.row_kth, kfloor) : -INFINITY;
    // entry -> segment table (one byte per entry; ns <= kThreads <= 255)
    uint8_t* segof = sb.segof;
    for (int s = tid; s < ns; s += kThreads)
      for (int i = 0, e = min(stage[s].ncand, lim); i < e; ++i) segof[stage[s].off + i] = static_cast<uint8_t>(s);
    __syncthreads();
    constexpr int U = 8;
    for (int base = 0; base < total; base += kThreads * U) {
      uint2 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = base + u * kThreads + tid;
        v[u] = make_uint2(0u, 0xff800000u);  // -inf: never kept
        if (e < total) {
          const int s = segof[e];
          v[u] = __ldcg(cand + static_cast<int64_t>(s) * kSegCap + (e - stage[s].off));
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float x = __uint_as_float(v[u].y);
        if (x > -INFINITY && x >= floor_v) {
          const int pos = atomicAdd(&sm.seg_n, 1);
          if (pos < kPool) {
            pidx[pos] = static_cast<int32_t>(v[u].x);
            pval[pos] = x;
          }
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      sm.pool_n = sm.seg_n;
      if (sm.seg_n > kPool) sm.row_over = 1;
    }
  } else if (a.filt && tid == 0) {
    sm.row_over = 1;  // more listed entries than the table holds
  }
  __syncthreads();
}

// Row end: exact cut from the pool (or the general path), record, draw.
// The end of a row once its cut is known: the draw of a sampled row (and of
// the draft row of a fused call) from the kept list, or by a scan of the row
// when none is stored, then the row record with the draft token's adjusted
// probability (its own logit read back).  The whole CTA.
template <typename E>
__device__ void row_tail(const KArgs& a, const RowInfo& ri, const E* grow, Scratch& sm, float m, int argmax, bool bad,
                         Cut cut, FF zf, int list_len) {
  const int tid = threadIdx.x;
  spec_row_stat* rec = a.rows + ri.job;
  int32_t* lidx = a.list_idx + static_cast<int64_t>(ri.job) * kCap;
  float* lw = a.list_w + static_cast<int64_t>(ri.job) * kCap;
  // sample mode (and the draft row of a fused call): draw this row's token
  const bool draws = a.mode == kModeSample || (a.fused && !ri.is_target);
  if (draws) {
    const double u = a.greedy ? 0.0 : a.fused ? a.u_draft[ri.b] : a.u[static_cast<int64_t>(ri.b) * a.K + ri.t];
    int tok;
    if (bad) {
      tok = -1;
    } else if (a.greedy) {
      tok = argmax;
    } else if (list_len >= 0) {
      __syncthreads();
      const int pos = list_ordered_draw(list_len, u, sm, [&](int i) { return __ldcg(&lw[i]); });
      tok = (pos >= 0) ? __ldcg(&lidx[pos]) : -1;
    } else {
      tok = global_rows_draw<E>(a, grow, grow, m, m, cut, cut, 1.0f, 1.0f, false, u, sm);
    }
    if (tid == 0) {
      if (a.fused) a.out_draft[ri.b] = tok;
      else a.out_tokens[static_cast<int64_t>(ri.b) * a.K + ri.t] = tok;
      rec->token = tok;
    }
  }

  // row record
  if (tid == 0) {
    int flags = 0;
    if (bad) flags |= kFlagNonfinite;
    double p_tok = 0.0;
    if (a.mode == kModeVerify && ri.t < ri.kb && !a.fused) {  // fused: the epilogue computes it
      const int d = a.tokens[static_cast<int64_t>(ri.b) * a.K + ri.t];
      if (d < 0 || d >= a.V) {
        flags |= kFlagToken;
      } else if (!bad && !a.greedy) {
        const float ld = Fmt<E>::at_global(grow, d);
        // same weight as the kept list and the normaliser use
        if (cut.keep(ld, d) && ld > -INFINITY) p_tok = static_cast<double>(wexp(ld, m, a.c)) / ff_to_d(zf);
      }
    }
    rec->zf = ff_to_d(zf);
    rec->p_tok = p_tok;
    rec->m = m;
    rec->tau_val = cut.tv;
    rec->tau_idx = cut.ti;
    rec->argmax = argmax;
    rec->list_len = list_len;
    rec->flags = flags;
    if (a.mode == kModeSample && bad) set_status(a, SPEC_ERR_NONFINITE);
  }
}

template <typename E>
__device__ void row_finish(const KArgs& a, const RowInfo& ri, const E* grow, Scratch& sm, Local& C, SortBuf sb,
                           int32_t* pool_idx, float* pool_val) {
  // first the pool of every segment list's head: as many entries as a 256-key
  // (top-k) or 512-key (top-p: the nucleus may be long) register sort holds
  const int row = ri.job;
  const int ns = a.nseg;
  int lim = (a.top_k > 0) ? min(a.top_k, max(4, 256 / ns)) : max(4, 512 / ns);
  // top-k through a running set: a few lists of k keys each, taken whole
  if (lim >= kSegCap || (a.top_k > 0 && a.top_k <= kRunCap)) lim = INT_MAX;
  row_merge(a, row, sm, sb, pool_idx, pool_val, lim, -INFINITY);
  const float m = sm.row_m;
  const int argmax = sm.row_argmax;
  const int fl = sm.row_flags;
  // NaN / +inf in a segment, or no finite value in the row
  const bool bad = (fl & kSegBad) || !(m > -INFINITY);
  const FF z = sm.row_z;
  bool over = sm.row_over != 0;
  int total = sm.pool_n;
  unsigned long long bound = sm.row_bound;
  const float theta = sm.row_theta;
  __syncthreads();

  int32_t* lidx = a.list_idx + static_cast<int64_t>(ri.job) * kCap;
  float* lw = a.list_w + static_cast<int64_t>(ri.job) * kCap;
  const bool use_k = a.top_k > 0 && a.top_k < a.V;
  const bool use_p = a.top_p < 1.0f;
  RowCtx<E> rg;
  rg.g = grow;
  rg.sl = grow;
  rg.s0 = 0;
  rg.L = a.V;
  rg.m = m;
  rg.c = a.c;
  rg.gsrc = 1;
  rg.aligned = a.aligned;

  Cut cut = cut_all();
  FF zf = z;
  int list_len = -1;
  if (!bad && !a.greedy && (use_k || use_p)) {
    bool done = false;
    float head_kth = -INFINITY;
    for (int attempt = 0; attempt < 2 && !done; ++attempt) {
      if (attempt == 1) {  // the heads did not settle the cut: every listed entry
        if (lim == INT_MAX) break;
        row_merge(a, row, sm, sb, pool_idx, pool_val, INT_MAX, head_kth);
        over = sm.row_over != 0;
        total = sm.pool_n;
        bound = sm.row_bound;
        __syncthreads();
      }
      if (over || total <= 0) continue;
      const CutResult res = sort_and_cut(m, a.c, pool_idx, pool_val, total, sb, use_k ? a.top_k : 0,
                                         use_p ? a.top_p : 1.0f, z, sm);
      // Exact when no element outside the pool can be kept.  Every element
      // left out of a list's head has a key <= bound; every element left out of
      // a list lies below its segment's k-th value (top-k: the pool's k-th key
      // must exceed bound), or below the segment's candidate floor (top-p: the
      // cut must be reached within the pool, at or above every floor, and
      // above bound).
      bool exact;
      if (use_k) {
        // the head pool's k-th value bounds the row's k-th value from below
        if (total >= a.top_k) head_kth = skey_val(sb.skey[a.top_k - 1]);
        exact = bound == 0ull || (total >= a.top_k && sb.skey[a.top_k - 1] > bound);
      } else {
        exact = res.reached && theta <= res.tv && (bound == 0ull || sort_key(res.tv, res.ti) > bound);
      }
      if (exact) {
        cut = Cut{res.tv, res.ti};
        zf = res.zf;
        if (res.nkeep <= kCap) {
          write_kept_by_index(sb.skey, res.nkeep, m, a.c, lidx, lw, sm);
          list_len = res.nkeep;
        }
        done = true;
      }
      __syncthreads();
    }
    if (!done) general_cut<E>(a, rg, sm, C, sb, z, &cut, &zf, &list_len, lidx, lw);
  }

  row_tail<E>(a, ri, grow, sm, m, argmax, bad, cut, zf, list_len);
}

// ---------------------------------------------------------------------------
// segment phase helpers

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Streaming 16-byte load: read once, so no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4& q, int w) {
  return w == 0 ? q.x : w == 1 ? q.y : w == 2 ? q.z : q.w;
}

template <typename E>
struct Seg;

template <>
struct Seg<uint16_t> {  // bf16 bits, 8 per vector
  static constexpr int N = 8;
  __device__ static float get(const uint4& q, int i) {
    const uint32_t w = word_of(q, i >> 1);
    return (i & 1) ? __uint_as_float(w & 0xffff0000u) : __uint_as_float(w << 16);
  }
  __device__ static uint4 neg_inf() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }
  // vector v with only its first n elements read (tail, or a row start that is
  // not 16-byte aligned); the rest are -inf
  __device__ static uint4 load_some(const uint16_t* g, int v, int n) {
    const unsigned short* s = reinterpret_cast<const unsigned short*>(g) + static_cast<int64_t>(v) * 8;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (2 * i < n) ? __ldg(s + 2 * i) : 0xff80u;
      const uint32_t hi = (2 * i + 1 < n) ? __ldg(s + 2 * i + 1) : 0xff80u;
      w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static float pw_max(uint32_t w) { return max_nan(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); }
  // Bit i set when element i is >= f (ordered compare: NaN never passes), on
  // packed pairs.  f must lie on the bf16 grid.
  __device__ static uint32_t ge_mask(const uint4& q, float f) {
    const uint32_t fb = __float_as_uint(f) >> 16;
    const uint32_t tw = fb | (fb << 16);
    __nv_bfloat162 t;
    memcpy(&t, &tw, 4);
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t x = word_of(q, w);
      __nv_bfloat162 xv;
      memcpy(&xv, &x, 4);
      const uint32_t r = __hge2_mask(xv, t);
      m |= ((r & 1u) | ((r >> 15) & 2u)) << (2 * w);
    }
    return m;
  }
  // the compare value of a threshold: bf16 grid values and keys' floors stay
  // the same set under truncation; -inf becomes the lowest finite value, so
  // that -inf elements never pass
  __device__ static float grid_floor(float t) {
    return __uint_as_float(__float_as_uint(fmaxf(t, -3.402823466e38f)) & 0xffff0000u);
  }
  // NaN-propagating max of NV vectors, on packed pairs; pw[j] keeps vector j's
  // packed maximum (pw_max gives its value)
  template <int NV>
  __device__ static float lane_max(const uint4 (&q)[NV], uint32_t (&pw)[NV]) {
    uint32_t w[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      __nv_bfloat162 a, b, c, d;
      memcpy(&a, &q[j].x, 4);
      memcpy(&b, &q[j].y, 4);
      memcpy(&c, &q[j].z, 4);
      memcpy(&d, &q[j].w, 4);
      const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
      memcpy(&w[j], &m, 4);
      pw[j] = w[j];
    }
#pragma unroll
    for (int j = 1; j < NV; ++j) {
      __nv_bfloat162 a, b;
      memcpy(&a, &w[0], 4);
      memcpy(&b, &w[j], 4);
      const __nv_bfloat162 m = __hmax2_nan(a, b);
      memcpy(&w[0], &m, 4);
    }
    return max_nan(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xffff0000u));
  }
  // Sum of 2^((x - g) c) over the NV vectors' elements (g: their max, finite),
  // the weight function's arithmetic (x - g, then times c, rounded to
  // nearest) on packed f32 pairs
  template <int NV>
  __device__ static float zsum(const uint4 (&q)[NV], float g, float c) {
    uint64_t gg, cc, s = 0ull;
    asm("mov.b64 %0, {%1, %1};" : "=l"(gg) : "f"(g));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t x = word_of(q[j], w);
        uint64_t p, d;
        asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "r"(x << 16), "r"(x & 0xffff0000u));
        asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(p), "l"(gg));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(d), "l"(cc));
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
        asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(ex2f(lo)), "f"(ex2f(hi)));
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(s), "l"(p));
      }
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(s));
    return lo + hi;
  }
  // NaN-propagating max of the vector, on packed pairs
  __device__ static float vmax(const uint4& q) {
    __nv_bfloat162 a, b, c, d;
    memcpy(&a, &q.x, 4);
    memcpy(&b, &q.y, 4);
    memcpy(&c, &q.z, 4);
    memcpy(&d, &q.w, 4);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    uint32_t mw;
    memcpy(&mw, &m, 4);
    return max_nan(__uint_as_float(mw << 16), __uint_as_float(mw & 0xffff0000u));
  }
};

template <>
struct Seg<float> {  // 4 per vector
  static constexpr int N = 4;
  __device__ static float get(const uint4& q, int i) { return __uint_as_float(word_of(q, i)); }
  __device__ static uint4 neg_inf() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
  __device__ static uint4 load_some(const float* g, int v, int n) {
    const float* s = g + static_cast<int64_t>(v) * 4;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = (i < n) ? __float_as_uint(__ldg(s + i)) : 0xff800000u;
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ static float vmax(const uint4& q) {
    return max_nan(max_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                   max_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
  }
  __device__ static uint32_t ge_mask(const uint4& q, float f) {
    return (__uint_as_float(q.x) >= f ? 1u : 0u) | (__uint_as_float(q.y) >= f ? 2u : 0u) |
           (__uint_as_float(q.z) >= f ? 4u : 0u) | (__uint_as_float(q.w) >= f ? 8u : 0u);
  }
  __device__ static float grid_floor(float t) { return fmaxf(t, -3.402823466e38f); }
  template <int NV>
  __device__ static float lane_max(const uint4 (&q)[NV], uint32_t (&pw)[NV]) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const float v = vmax(q[j]);
      pw[j] = __float_as_uint(v);
      m = max_nan(m, v);
    }
    return m;
  }
  __device__ static float pw_max(uint32_t w) { return __uint_as_float(w); }
};

// Bitonic sort of one value per lane, descending across the warp.
__device__ __forceinline__ float warp_sort_desc(float v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(FULL, v, j);
      const bool desc = (lane & k) == 0, lower = (lane & j) == 0;
      v = (desc == lower) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

// Entries of the descending list s[0, 32) that are >= v (> v when strict).
__device__ __forceinline__ int count_at_least(const float* s, float v, bool strict) {
  int pos = 0;
#pragma unroll
  for (int step = 32; step > 0; step >>= 1) {
    if (pos + step <= 32) {
      const float x = s[pos + step - 1];
      if (strict ? (x > v) : (x >= v)) pos += step;
    }
  }
  return pos;
}

// ---------------------------------------------------------------------------
// Counters in the workspace's counter area: every call finds them at zero and
// leaves them at zero -- the arrival that completes a counter resets it, once
// no other arrival of the call can touch it.

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// ---------------------------------------------------------------------------
// The two launches of a call.
//
// spec_seg_kernel: a persistent grid over items (item = row * nseg + segment);
// CTA b takes items b, b + grid, b + 2 grid, ...  Each CTA owns two segment
// buffers in shared memory that bulk copies fill two items ahead, so one copy is
// in flight while an item is processed.  Per item: maxima, then (one barrier)
// argmax, normaliser and the candidate floor, then (a second) the candidates,
// then (a third) warp 0 writes the segment's list and record while the other
// warps start the next item.
//
// spec_row_kernel: one CTA per row merges the row's segment records and lists,
// cuts, records the row and -- for the last row of a sequence to finish, found
// by a counter -- runs the sequence's accept tests and final draw.


// Source of an item: row = item / nseg, then the row's place (decode_job's
// mapping) with the divisions done by multiply-high.
template <typename E, bool RAG>
__device__ __forceinline__ const E* item_src(const KArgs& a, int item, int* s0, int* L) {
  const int row = fast_div(item, a.nseg_m, a.nseg_s);
  const int seg = item - row * a.nseg;
  int64_t off;
  bool tgt;
  if (a.mode == kModeVerify) {
    const SeqRows q = seq_of_row<RAG>(a, row);
    const int b = q.b, r = row - q.first;
    tgt = r <= q.kb;
    off = tgt ? static_cast<int64_t>(b) * a.tgt_seq + static_cast<int64_t>(r) * a.tgt_row
              : static_cast<int64_t>(b) * a.drf_seq + static_cast<int64_t>(r - (q.kb + 1)) * a.drf_row;
  } else {
    const int b = fast_div(row, a.rows_m, a.rows_s), t = row - b * a.K;
    tgt = false;
    off = static_cast<int64_t>(b) * a.drf_seq + static_cast<int64_t>(t) * a.drf_row;
  }
  *s0 = seg * a.S;
  *L = min(a.S, a.V - *s0);
  return static_cast<const E*>(tgt ? a.tgt : a.drf) + off + *s0;
}

// Thread 0: start the bulk copy of an item's 16-byte-aligned part into a
// segment buffer (one arrival with its byte count; a zero count completes the
// phase at once).
template <typename E, bool RAG>
__device__ __forceinline__ void item_issue(const KArgs& a, int item, void* segbuf, uint64_t* bar) {
  int s0, L;
  const E* g = item_src<E, RAG>(a, item, &s0, &L);
  const uint32_t bytes = static_cast<uint32_t>(L) * sizeof(E) & ~15u;
  mbar_expect_tx(bar, bytes);
  if (bytes > 0) bulk_copy_g2s(segbuf, g, bytes, bar);
}

// Vector v of an item: from the segment buffer when staged, else from global
// memory (rows not 16-byte aligned, or after a lost copy); the partial tail
// vector from global memory; -inf past the end.
template <typename E>
__device__ __forceinline__ uint4 item_vec(const E* g, int L, bool staged, bool aligned, const uint4* seg, int v) {
  constexpr int N = Seg<E>::N;
  if (v < L / N) {
    if (staged) return seg[v];
    if (aligned) return ld_stream(reinterpret_cast<const uint4*>(g) + v);
  }
  if (v * N < L) return Seg<E>::load_some(g, v, min(N, L - v * N));
  return Seg<E>::neg_inf();
}

// RAG: a ragged call (rows found through the host's per-row table)
template <typename E, bool RAG>
__global__ void __launch_bounds__(kThreads, 4) spec_seg_kernel(const KArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Scratch& sm = *reinterpret_cast<Scratch*>(smem_raw);
  unsigned char* bufs = smem_raw + sizeof(Scratch);
  constexpr int N = Seg<E>::N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nitems = a.nrows * a.nseg;
  // this CTA's items: one contiguous range, so it meets a row's segments in order
  const int beg = static_cast<int>(static_cast<int64_t>(blockIdx.x) * nitems / gridDim.x);
  const int end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * nitems / gridDim.x);
  unsigned long long* ckey = reinterpret_cast<unsigned long long*>(sm.cand_idx);  // an item's candidate keys
  unsigned long long* run = reinterpret_cast<unsigned long long*>(sm.cand_val);   // two halves of kRunCap keys
  // top-k with a running set: the CTA keeps the top k keys of the row segments
  // it has met so far; once it holds k, its k-th value is a floor for the row's
  // k-th value, and later segments of the row only collect elements >= it
  const bool stream_k = a.filt && a.top_k > 0 && a.top_k <= kRunCap;

  // a bulk copy needs 16-byte-aligned rows; a copy that misses its bounded wait
  // switches the CTA to plain loads (the stray copy is awaited before exit)
  bool staged = a.aligned != 0;
  bool issued0 = false, issued1 = false, stray0 = false, stray1 = false;
  uint32_t ph0 = 0, ph1 = 0;
  if (tid == 0) {
    mbar_init(&sm.bar[0], 1);
    mbar_init(&sm.bar[1], 1);
    fence_mbar_init();
    sm.seg_cnt[0] = sm.seg_cnt[1] = 0;
    sm.run_n[0] = sm.run_n[1] = 0;
    sm.run_theta[0] = sm.run_theta[1] = -INFINITY;
  }
  __syncthreads();
  if (staged) {
    issued0 = beg < end;
    issued1 = beg + 1 < end;
    if (tid == 0) {
      if (issued0) item_issue<E, RAG>(a, beg, bufs, &sm.bar[0]);
      if (issued1) item_issue<E, RAG>(a, beg + 1, bufs + a.seg_bytes, &sm.bar[1]);
    }
  }

  int k = 0, rp = 0, prev_row = -1;  // rp: the half of run[] holding the running set
  for (int cur = beg; cur < end; ++cur, ++k) {
    const int p = k & 1;
    const int row = fast_div(cur, a.nseg_m, a.nseg_s);
    const bool new_run = row != prev_row;
    prev_row = row;
    const bool run_ends = cur + 1 >= end || fast_div(cur + 1, a.nseg_m, a.nseg_s) != row;
    int s0, L;
    const E* g = item_src<E, RAG>(a, cur, &s0, &L);
    const uint4* seg = reinterpret_cast<const uint4*>(bufs + p * a.seg_bytes);

    // ---- wait for this item's copy
    const bool issued = p ? issued1 : issued0;
    bool lost = false;
    if (issued) {
      uint32_t& ph = p ? ph1 : ph0;
      lost = !mbar_wait_bounded(&sm.bar[p], ph);
      ph ^= 1u;
      if (lost) { if (p) stray1 = true; else stray0 = true; }
    }
    const bool from_smem = issued && !lost;
    const int nv = L / N;  // vectors wholly inside the item
    auto vec = [&](int j) -> uint4 {
      const int v = j * kThreads + tid;
      if (from_smem && v < nv) return seg[v];
      return item_vec<E>(g, L, false, a.aligned != 0, seg, v);
    };
    // the running floor, when the set already holds k keys of this row
    const float rfloor = (stream_k && !new_run) ? sm.run_theta[rp] : -INFINITY;
    const bool steady = rfloor > -INFINITY;

    // ---- pass 1: per-vector and per-thread maxima (NaN-propagating); with a
    // running floor, the elements >= it are collected in the same pass
    float vm[kNV];
    float tm = -INFINITY;
#pragma unroll
    for (int j = 0; j < kNV; ++j) {
      vm[j] = Seg<E>::vmax(vec(j));
      tm = max_nan(tm, vm[j]);
    }
    if (steady && tm >= rfloor) {
      uint32_t mask = 0;
#pragma unroll
      for (int j = 0; j < kNV; ++j)
        if (vm[j] >= rfloor) mask |= 1u << j;
      while (mask) {
        const int j = __ffs(mask) - 1;
        mask &= mask - 1;
        const uint4 q = vec(j);
#pragma unroll
        for (int i = 0; i < N; ++i) {
          const float x = Seg<E>::get(q, i);
          if (x >= rfloor) {
            const int pos = atomicAdd(&sm.seg_cnt[p], 1);
            if (pos < kSegCap) ckey[pos] = sort_key(x, s0 + (j * kThreads + tid) * N + i);
          }
        }
      }
    }
    float wm = tm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = max_nan(wm, __shfl_xor_sync(FULL, wm, o));
    if (lane == 0) sm.wf[warp] = wm;
    const float srt = (a.filt && !steady) ? warp_sort_desc(tm, lane) : 0.0f;
    if (a.filt && !steady) sm.tmax[tid] = srt;  // each warp's maxima, descending
    if (tid == 0) sm.run_theta[rp ^ 1] = -INFINITY;  // set by this item's merge when it holds k keys
    if (__syncthreads_or(lost)) staged = false;  // S1
    // item k counts candidates in seg_cnt[k & 1]; every thread read the other
    // counter (item k - 1's) before this barrier, so it can be cleared now
    if (tid == 0) sm.seg_cnt[p ^ 1] = 0;
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) ms = max_nan(ms, sm.wf[w]);
    const bool bad = !(ms == ms) || ms == INFINITY;
    const bool live = !bad && ms > -INFINITY;  // some finite value

    // ---- first argmax: the first vector whose maximum is ms, then its first element
    int am = INT_MAX;
    if (live && tm == ms) {
      int jj = 0;
#pragma unroll
      for (int j = kNV - 1; j >= 0; --j)
        if (vm[j] == ms) jj = j;
      const uint4 q = vec(jj);
#pragma unroll
      for (int i = N - 1; i >= 0; --i)
        if (Seg<E>::get(q, i) == ms) am = (jj * kThreads + tid) * N + i;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = min(am, __shfl_xor_sync(FULL, am, o));
    if (lane == 0) sm.wi[warp] = am;

    // ---- normaliser relative to the segment max: pairwise within the thread,
    // float-float across threads
    if (a.need_z && live) {
      float sv[kNV];
#pragma unroll
      for (int j = 0; j < kNV; ++j) {
        const uint4 q = vec(j);
        float w[N];
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = wexp(Seg<E>::get(q, i), ms, a.c);
#pragma unroll
        for (int h = N / 2; h > 0; h >>= 1)
#pragma unroll
          for (int i = 0; i < h; ++i) w[i] += w[i + h];
        sv[j] = w[0];
      }
#pragma unroll
      for (int h = 1; h < kNV; h <<= 1)
#pragma unroll
        for (int j = 0; j + h < kNV; j += 2 * h) sv[j] += sv[j + h];
      const FF wz = warp_sum_ff(ff(sv[0]));
      if (lane == 0) sm.wd[warp] = wz;
    }

    // ---- without a running floor: the candidate floor is the n0-th largest
    // thread maximum.  Ranks order the kThreads maxima by (value desc, warp,
    // position in the warp's sorted list); exactly one thread has rank n0 - 1.
    const bool cands = a.filt && live && a.n0 <= kThreads && !steady;
    float theta = rfloor;
    if (a.filt && !steady) {
      if (cands) {
        int rank = lane;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
          if (w != warp) rank += count_at_least(sm.tmax + w * 32, srt, w > warp);
        if (rank == a.n0 - 1) sm.theta = srt;
      }
      __syncthreads();  // S2
      theta = sm.theta;
      // every finite element >= theta, from the vectors whose maximum reaches it
      if (cands && tm >= theta) {
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < kNV; ++j)
          if (vm[j] >= theta) mask |= 1u << j;
        while (mask) {
          const int j = __ffs(mask) - 1;
          mask &= mask - 1;
          const uint4 q = vec(j);
#pragma unroll
          for (int i = 0; i < N; ++i) {
            const float x = Seg<E>::get(q, i);
            if (x >= theta && x > -INFINITY) {
              const int pos = atomicAdd(&sm.seg_cnt[p], 1);
              if (pos < kSegCap) ckey[pos] = sort_key(x, s0 + (j * kThreads + tid) * N + i);
            }
          }
        }
      }
      __syncthreads();  // S3: the candidates are complete
    }
    const int n = sm.seg_cnt[p];
    const bool collected = cands || (steady && live);
    const bool over = a.filt && live && (!collected || n > kSegCap);
    const bool listed = collected && !over;
    SegRec* rec = a.segs + cur;
    uint2* gc = a.seg_cand + static_cast<int64_t>(cur) * kSegCap;
    int ncand = 0;
    float kth = -INFINITY;

    if (stream_k) {
      // ---- merge the new keys into the running set (sorted desc, at most k):
      // a key's new position is the number of larger keys in both lists
      const int rn = new_run ? 0 : sm.run_n[rp];
      const unsigned long long* src = run + rp * kRunCap;
      unsigned long long* dst = run + (rp ^ 1) * kRunCap;
      const int nn = listed ? n : 0;
      const int K = a.top_k;
      for (int i = tid; i < rn; i += kThreads) {
        const unsigned long long key = src[i];
        int r = i;
        for (int c = 0; c < nn; ++c) r += (ckey[c] > key) ? 1 : 0;
        if (r < K) dst[r] = key;
        if (r == K - 1) sm.run_theta[rp ^ 1] = skey_val(key);
      }
      for (int c = tid; c < nn; c += kThreads) {
        const unsigned long long key = ckey[c];
        int lo = 0, hi = rn;  // larger keys of the sorted running set
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (src[mid] > key) lo = mid + 1; else hi = mid;
        }
        int r = lo;
        for (int q = 0; q < nn; ++q) r += (ckey[q] > key) ? 1 : 0;
        if (r < K) dst[r] = key;
        if (r == K - 1) sm.run_theta[rp ^ 1] = skey_val(key);
      }
      const int new_n = min(K, rn + nn);
      if (tid == 0) sm.run_n[rp ^ 1] = new_n;
      __syncthreads();  // the merged set (and the buffer's last reads) are complete
      rp ^= 1;
      // the run ends here: its top k is the list of this item
      if (run_ends && !over) {
        for (int i = tid; i < new_n; i += kThreads)
          gc[i] = make_uint2(static_cast<uint32_t>(skey_idx(dst[i])), __float_as_uint(skey_val(dst[i])));
        ncand = new_n;
        kth = (new_n >= K) ? sm.run_theta[rp] : -INFINITY;
      }
    } else if (listed) {
      // ---- per-item list in rank order (value desc, index asc): top-k keeps
      // ranks < k, and the candidate of rank k - 1 is the k-th value
      const bool use_k = a.top_k > 0;
      const int keep = use_k ? min(n, a.top_k) : n;
      for (int c = tid; c < n; c += kThreads) {
        const unsigned long long key = ckey[c];
        int rank = 0;
#pragma unroll 4
        for (int q = 0; q < n; ++q) rank += (ckey[q] > key) ? 1 : 0;
        if (rank < keep) gc[rank] = make_uint2(static_cast<uint32_t>(skey_idx(key)), __float_as_uint(skey_val(key)));
        if (use_k && rank == a.top_k - 1) rec->kth = skey_val(key);
      }
      ncand = keep;
    }

    // ---- refill the buffer with the item two ahead, once every read of it is
    // done: the merge barrier (running top-k) or S3 (other filters) followed
    // them; without a filter the argmax and normaliser passes need one here
    if (!a.filt) __syncthreads();
    const int nxt = cur + 2;
    const bool refill = staged && nxt < end;
    if (p) issued1 = refill; else issued0 = refill;
    if (tid == 0 && refill) {
      fence_proxy_async_smem();
      item_issue<E, RAG>(a, nxt, bufs + p * a.seg_bytes, &sm.bar[p]);
    }

    // ---- the segment record (thread 0)
    if (tid == 0) {
      int amin = INT_MAX;
      for (int w = 0; w < kWarps; ++w) amin = min(amin, sm.wi[w]);
      FF z = ff(0.0f);
      if (a.need_z && live)
        for (int w = 0; w < kWarps; ++w) z = ff_add(z, sm.wd[w]);
      rec->m = ms;
      rec->argmax = (amin == INT_MAX) ? -1 : s0 + amin;
      rec->z_hi = z.hi;
      rec->z_lo = z.lo;
      rec->theta = collected ? theta : -INFINITY;
      if (stream_k) rec->kth = kth;
      else if (!(listed && a.top_k > 0 && n >= a.top_k)) rec->kth = -INFINITY;
      rec->ncand = ncand;
      rec->flags = (bad ? kSegBad : 0) | (over ? kSegOver : 0);
    }
  }
  // copies that missed their wait must land before the shared memory is released
  if (stray0) (void)mbar_wait_bounded(&sm.bar[0], ph0 ^ 1u);
  if (stray1) (void)mbar_wait_bounded(&sm.bar[1], ph1 ^ 1u);
  // this CTA is done: the row kernel may be scheduled (it still waits for the
  // whole grid's memory before reading it)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Row merge, cut, record and (verify) the sequence counter and epilogue.
// At most 102 registers (5 CTAs per SM; bf16 rows need that many without
// spilling), fp32 rows 64 (8 per SM: the 1024 rows of a greedy batch of 256
// sequences run in one wave; ptxas moves a few values to the stack).
template <typename E, bool RAG>
__global__ void __launch_bounds__(kThreads, sizeof(E) == 4 ? 8 : 5) spec_row_kernel(const KArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Scratch& sm = *reinterpret_cast<Scratch*>(smem_raw);
  unsigned char* scratch = smem_raw + sizeof(Scratch);
  int32_t* pool_idx = reinterpret_cast<int32_t*>(scratch);
  float* pool_val = reinterpret_cast<float*>(pool_idx + kPool);
  const SortBuf sb{reinterpret_cast<unsigned long long*>(pool_val + kPool),
                   reinterpret_cast<uint8_t*>(pool_val + kPool + 2 * kPool)};
  // launched as a programmatic dependent of the segment kernel: wait until that
  // grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int row = static_cast<int>(blockIdx.x); row < a.nrows; row += static_cast<int>(gridDim.x)) {
    const RowInfo ri = decode_job<RAG>(a, row);
    const E* grow = static_cast<const E*>(ri.is_target ? a.tgt : a.drf) + ri.row_off;
    Local C;
    row_finish<E>(a, ri, grow, sm, C, sb, pool_idx, pool_val);
    // every global write of the row is ordered before the sequence counter
    __syncthreads();
    if (a.mode == kModeVerify) {
      if (threadIdx.x == 0) {
        fence_acq_rel_gpu();
        unsigned long long* tk = &a.tickets[ri.b];
        const bool last = atomicAdd(tk, 1ull) == static_cast<unsigned long long>(ri.nr - 1);
        if (last) {
          *tk = 0ull;  // the sequence's last row: no other arrival of this call
          fence_acq_rel_gpu();
        }
        sm.bi[15] = last ? 1 : 0;
      }
      __syncthreads();
      if (sm.bi[15]) verify_epilogue<E>(a, ri.b, ri.kb, ri.first, sm);
    }
    __syncthreads();
  }
}


// ---------------------------------------------------------------------------
// The one-launch streaming kernel (rows whose starts are 16-byte aligned;
// greedy, top-k with k <= kSK, or top-p alone; ragged batches too).
//
// A persistent grid, four CTAs per SM; CTA c takes rows c, c + G, c + 2G, ...
// in order, so whole sequences complete one after another through the launch
// and the work after a row (its cut and record, and a sequence's accept tests
// and final draw) overlaps the streaming of other rows.  A row never leaves
// its CTA: there is no cross-CTA merge.
//
//   * Each warp owns a ring of kSNS 3-KB buffers that bulk copies fill; a row
//     is walked in warp-stages of kSWV vectors, warp w taking stages w, w + 4,
//     ...  Lane 0 keeps the ring full, running ahead through this warp's
//     stages of its next rows, so a warp waits only for its own copies and
//     never for a row boundary.
//   * Per stage and lane: the max of its six vectors (packed bf16 pairs for
//     bf16) against the running max; only a new max looks at single elements
//     (its first index).
//   * Top-k works on groups: a lane's six vectors of one stage.  A row's top k
//     elements lie in the k groups with the largest maxima (k elements reach
//     the k-th largest group max), so a warp keeps (group max, group) for
//     every group whose max reaches its threshold -- one slot per lane, no
//     element work while streaming.  The threshold starts at the k-th largest
//     vector maximum of the warp's first stage and rises to the k-th largest
//     buffered group max whenever the buffer passes a high-water mark; every
//     such value bounds the row's k-th element from below, so a warp also
//     takes any higher value another warp publishes.
//   * Row end: the k-th largest group max over the whole row, f2 (a radix
//     select over every buffered group); the groups at or above it are read
//     back from the row (one round of loads), their elements >= f2 ranked by
//     one warp in registers (value desc, index asc); the first k, then the
//     top-p prefix within them, are the kept set, written in index order with
//     the row record.  Ties or a buffer too small for a stage send the row to
//     the exact general path.  The CTA that completes a sequence (a counter)
//     runs its accept tests and final draw.
//   * Top-p alone: each lane also sums its groups' weights (the normaliser),
//     and the warps keep their 160 largest groups.  At the row end f2 is the
//     largest group max whose groups' maxima alone weigh top_p * Z; the
//     elements >= f2 of those groups form a pool in the drained ring (the
//     issue cursor stops at the row's end in this mode), cut by counting bf16
//     grid points (else a block sort) and written in index order.

constexpr int kSK = 64;            // largest top-k the streaming kernel collects
constexpr int kSWV = 192;          // vectors per warp-stage (3 KB)
constexpr int kSVPL = kSWV / 32;   // vectors per lane and stage
constexpr int kSNS = 3;            // buffers per warp
constexpr int kSWCap = 256;        // candidate entries per warp
constexpr int kSKeys = 256;        // row-end ranking capacity (keys in the Scratch's candidate arrays)
constexpr int kSGroups = 512;      // top-k row end: groups read back (their first vectors, after the keys)
constexpr int kSPKeep = 160;       // top-p: groups a warp keeps when its buffer is cut
constexpr int kSPHwm = kSWCap - 32; // top-p: buffer entries that trigger the cut (a stage adds <= 32)
constexpr int kSPBuckets = 2048;   // bf16 top-p pool cut: grid points between the floor and the max
constexpr int kSPItems = 5120;     // top-p row end: group vectors read back (after the pool and its keys)
constexpr int kSVShift = 26;       // a buffer entry: first vector of the group | (top-p) its vectors' mask << kSVShift
constexpr size_t kSStage = static_cast<size_t>(kSWV) * 16;
constexpr size_t kSRing = static_cast<size_t>(kWarps) * kSNS * kSStage;
constexpr size_t kSCand = static_cast<size_t>(kWarps) * kSWCap * sizeof(uint2);
static_assert(kCap * sizeof(unsigned long long) <= kSCand, "the general path's sort keys fit the candidate buffers");
static_assert(kListTable <= sizeof(int32_t) * kCap + sizeof(float) * kCap &&
                  kSKeys * sizeof(unsigned long long) + kSGroups * sizeof(int32_t) <=
                      sizeof(int32_t) * kCap + sizeof(float) * kCap,
              "the merge's entry table and the row-end keys fit the Scratch's candidate arrays");
static_assert(kSK <= kSWV && 4 * kSK <= kSWCap && kSK <= 64, "a warp's first stage and buffer hold k candidates");
static_assert(kPool * (2 * sizeof(int32_t) + sizeof(unsigned long long)) + kSPItems * sizeof(int32_t) <= kSRing,
              "the top-p row end's pool, sort keys and vector list fit the drained stage ring");
static_assert(kSVPL <= 32 - kSVShift, "a group's vector mask fits above its first vector");
static_assert(kSPKeep < kSPHwm, "a cut buffer has room for the next stage");
static_assert(kSPBuckets * sizeof(int) <= kPool * sizeof(unsigned long long) && kThreads <= kSPBuckets,
              "the bf16 pool cut's buckets (then the bitmap's run prefixes) fit the sort-key space");

// What a streaming launch keeps besides the max and first argmax.
enum : int { kSMGreedy = 0, kSMTopK = 1, kSMTopP = 2 };

struct alignas(128) StreamHdr {
  uint64_t bar[kWarps * kSNS];  // completion of each warp's buffers
  float wthr[kWarps];           // published warp thresholds of the current row
  float wmax[kWarps];
  int32_t warg[kWarps];
  int32_t wflag[kWarps];        // row end: kSegOver
  int32_t wfill[kWarps];        // entries in each warp's buffer (slots taken by atomics)
  int32_t nlist;                // row end: keys gathered
  int32_t cut;                  // row end: rank of the last kept entry
  FF zf;                        // row end: kept mass
  FF wz[kWarps];                // top-p row end: each warp's normaliser, relative to its max
  int32_t pc[4];                // top-p row end, bf16 pool cut: crossing thread, bucket, count, last index
  uint32_t rbins[48];           // top-k row end: the radix select's three rounds of 16 bins
  float wpart[2 * kWarps];      // top-p row end: the warps' partial masses, by round parity
  int32_t last;                 // this CTA completed the sequence
};

template <int PASS_CAND>
__host__ __device__ constexpr size_t stream_smem_bytes() {
  return sizeof(Scratch) + sizeof(StreamHdr) + kSRing + (PASS_CAND ? kSCand : 0);
}

// Largest t whose set bits lie in the top KB bits such that at least `need`
// of the warp's keys key(0..PER-1) are >= t; 0 when fewer than `need` keys are
// nonzero (a zero key counts for nothing).  Same value on every lane.
template <int PER, int KB, typename KeyOf>
__device__ __forceinline__ uint32_t warp_select_key(KeyOf key_of, int need) {
  // the bits that every nonzero key shares with the largest are set from the
  // start: the result lies between the smallest and the largest key
  uint32_t lo = 0xffffffffu, hi = 0u;
  int nz = 0;
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const uint32_t k = key_of(p);
    if (k) lo = min(lo, k);
    hi = max(hi, k);
    nz += k ? 1 : 0;
  }
  lo = __reduce_min_sync(FULL, lo);
  hi = __reduce_max_sync(FULL, hi);
  if (static_cast<int>(__reduce_add_sync(FULL, static_cast<unsigned>(nz))) < need) return 0u;
  const int top = 31 - __clz(lo ^ hi);  // highest differing bit (-1: all keys equal)
  uint32_t t = (top < 0) ? hi : (hi & ~((2u << top) - 1u));
#pragma unroll 1
  for (int bit = min(top, 31); bit >= 32 - KB; --bit) {
    const uint32_t c = t | (1u << bit);
    int n = 0;
#pragma unroll
    for (int p = 0; p < PER; ++p) n += (key_of(p) >= c) ? 1 : 0;
    if (static_cast<int>(__reduce_add_sync(FULL, static_cast<unsigned>(n))) >= need) t = c;
  }
  return t;
}

// The float a key threshold t compares as: for data on the element grid,
// x >= key_floor(t) iff okey32(x) >= t (bf16 keys compare on their top 16 bits).
__device__ __forceinline__ float key_floor(uint32_t t) { return t ? okey32_val(t) : -INFINITY; }

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

// The k-th largest value of a warp's buffer of n entries (-inf when fewer).
template <typename E>
__device__ __forceinline__ float warp_buffer_kth(const uint2* wc, int n, int k) {
  constexpr int KB = sizeof(E) == 2 ? 16 : 32;
  constexpr int PER = kSWCap / 32;
  const int lane = threadIdx.x & 31;
  uint32_t key[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int i = p * 32 + lane;
    key[p] = (i < n) ? okey32(__uint_as_float(wc[i].y)) : 0u;
  }
  return key_floor(warp_select_key<PER, KB>([&](int p) { return key[p]; }, k));
}

// Drop the buffer entries below f (order kept); returns the new count.
__device__ __forceinline__ int warp_buffer_compact(uint2* wc, int n, float f) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  int out = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    uint2 e = make_uint2(0u, 0u);
    bool keep = false;
    if (i < n) {
      e = wc[i];
      keep = __uint_as_float(e.y) >= f;
    }
    const unsigned km = __ballot_sync(FULL, keep);  // every lane has read its entry
    if (keep) wc[out + __popc(km & lt)] = e;
    out += __popc(km);
  }
  __syncwarp();
  return out;
}

// Slots for `cnt` entries of every lane of a warp from the shared counter
// *fill: one atomic per warp; returns this lane's first slot (entries in lane
// order).
__device__ __forceinline__ int warp_reserve(int* fill, int cnt) {
  const int lane = threadIdx.x & 31;
  const int incl = warp_incl_scan_i(cnt, lane);
  int base = 0;
  if (lane == 31 && incl > 0) base = atomicAdd(fill, incl);
  return __shfl_sync(FULL, base, 31) + incl - cnt;
}

// The largest key threshold t (its set bits in the top KB bits) such that the
// values v[p] of the keys key[p] >= t add up to at least `need` over the
// whole CTA (every thread holds PER keys; zero keys count for nothing); 0 when
// even all of them fall short.  Four key bits a round: each round adds the
// values of the keys that match the bits fixed so far into 16 shared bins by
// their next digit, and every thread walks the bins from the top digit down.
// T = int (counts: the need-th largest key).
// bins: 3 x 16 of T, zero on entry; one block barrier a round; the same value
// on every thread.
template <int PER, int KB, typename T>
__device__ uint32_t block_radix_select(const uint32_t (&key)[PER], const T (&v)[PER], T need, void* bins) {
  T* bn = static_cast<T*>(bins);
  uint32_t t = 0;
  T above = T(0);
  int r = 0;
#pragma unroll 1
  for (int shift = 28; shift >= 32 - KB; shift -= 4, ++r) {
    T* b = bn + (r % 3) * 16;
    const uint32_t hm = (shift == 28) ? 0u : (0xffffffffu << (shift + 4));  // the bits fixed so far
#pragma unroll
    for (int p = 0; p < PER; ++p)
      if (key[p] != 0u && (key[p] & hm) == t) atomicAdd(&b[(key[p] >> shift) & 15u], v[p]);
    __syncthreads();
    // the bins of round r + 2 were read last in round r - 1
    if (threadIdx.x < 16) bn[((r + 2) % 3) * 16 + threadIdx.x] = T(0);
    T acc = above;
    int ds = -1;
#pragma unroll 1
    for (int d = 15; d >= 0; --d) {
      const T x = b[d];
      if (acc + x >= need) {
        ds = d;
        break;
      }
      acc += x;
    }
    if (ds < 0) return 0u;  // the same on every thread
    t |= static_cast<uint32_t>(ds) << shift;
    above = acc;
  }
  return t;
}

// Top-p row end: the largest key threshold t (top KB bits) such that the
// weights wt[p] of the entries whose keys key[p] are >= t add up to at least
// `need` over the whole CTA (every thread holds PER entries; zero keys count
// for nothing); a value <= lo when even all of them fall short.  Every
// nonzero key lies in [lo, hi] (lo > 0): the bits those two share are set from
// the start.  One block barrier a round; the same value on every thread.
// part: 2 * kWarps floats.
template <int PER, int KB>
__device__ uint32_t block_select_mass(const uint32_t (&key)[PER], const float (&wt)[PER], float need, uint32_t lo,
                                      uint32_t hi, float* part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lo >= hi) return lo;
  const int top = 31 - __clz(static_cast<int>(lo ^ hi));  // the first bit they differ in
  uint32_t t = lo & ~((2u << top) - 1u);                 // their shared prefix: <= every key
#pragma unroll 1
  for (int bit = top; bit >= 32 - KB; --bit) {
    const uint32_t c = t | (1u << bit);
    float s = 0.0f;
#pragma unroll
    for (int p = 0; p < PER; ++p) s += (key[p] >= c) ? wt[p] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
    float* pr = part + (bit & 1) * kWarps;  // the round before and after write the other half
    if (lane == 0) pr[warp] = s;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += pr[w];
    if (tot >= need) t = c;
  }
  return t;
}

// The value of a bf16 grid point from its 16-bit order key (okey32 >> 16).
__device__ __forceinline__ float bf16_key_val(uint32_t k16) {
  const uint32_t k = k16 << 16;
  return okey32_val((k & 0x80000000u) ? k : (k | 0xffffu));
}

// bf16 top-p row end: the cut of a pool that holds every element of the row
// >= floor_v (n entries: pidx, pval), by counting instead of sorting.  The
// values lie on the bf16 grid, so a bucket (one grid point) weighs its count
// times the point's weight.  The buckets are walked from the row max down with
// float-float prefix masses to the first at which the mass reaches top_p * Z;
// that bucket's elements are taken in index order until it does.  The kept
// set is written in index order through a bitmap of the row (its position is
// the number of kept indices below it) when it fits the stored list.  Returns
// false, having written nothing, when the values span more than kSPBuckets
// grid points, the row more than 32 * nbm words, or the pool's mass stays
// below top_p * Z.  cnt: kSPBuckets ints; bm: nbm words.  The whole CTA.
__device__ bool pool_bucket_cut(int V, float m, float c, float top_p, FF z, int n, const int32_t* pidx,
                                const float* pval, float floor_v, int* cnt, uint32_t* bm, int nbm, StreamHdr& hd,
                                Scratch& sm, int32_t* lidx, float* lw, Cut* cut, FF* zf, int* list_len) {
  const int tid = threadIdx.x;
  const int khi = static_cast<int>(okey32(m) >> 16), klo = static_cast<int>(okey32(floor_v) >> 16);
  const int R = khi - klo + 1;  // bucket b: grid point khi - b
  const int nw = (V + 31) >> 5;
  if (R < 1 || R > kSPBuckets || nw > nbm) return false;
  for (int b = tid; b < R; b += kThreads) cnt[b] = 0;
  for (int w = tid; w < nw; w += kThreads) bm[w] = 0u;
  if (tid == 0) hd.pc[0] = INT_MAX;
  __syncthreads();
  for (int i = tid; i < n; i += kThreads) atomicAdd(&cnt[khi - static_cast<int>(okey32(pval[i]) >> 16)], 1);
  __syncthreads();
  // each thread a run of buckets, the max first
  const int per = (R + kThreads - 1) / kThreads;
  const int b0 = min(R, tid * per), b1 = min(R, b0 + per);
  FF run = ff(0.0f);
  for (int b = b0; b < b1; ++b) {
    const int k = cnt[b];
    if (k) run = ff_add(run, ff_mul(ff(wexp(bf16_key_val(khi - b), m, c)), static_cast<float>(k)));
  }
  FF total;
  const FF excl = block_excl_scan_ff(run, &total, sm);
  const FF need = ff_mul(z, top_p);
  if (ff_lt(total, need)) return false;  // the same on every thread
  // the first thread whose run reaches need walks it: the bucket, then the
  // elements of that bucket one at a time
  if (!ff_lt(ff_add(excl, run), need)) atomicMin(&hd.pc[0], tid);
  __syncthreads();
  if (tid == hd.pc[0]) {
    FF x = excl;
    int bs = -1, js = 0, blast = -1;
    for (int b = b0; b < b1 && bs < 0; ++b) {
      const int k = cnt[b];
      if (!k) continue;
      blast = b;
      const float w = wexp(bf16_key_val(khi - b), m, c);
      const FF y = ff_add(x, ff_mul(ff(w), static_cast<float>(k)));
      if (!ff_lt(y, need)) {
        bs = b;
        for (js = 0; js < k;) {  // the crossing within the bucket (the whole bucket at most)
          x = ff_add(x, w);
          ++js;
          if (!ff_lt(x, need)) break;
        }
      } else {
        x = y;
      }
    }
    if (bs < 0) {
      // the run's crossing was not met bucket by bucket (a rounding difference
      // from the scan): the whole of its last nonempty bucket (bucket 0, the
      // max, is never empty)
      for (int b = b0 - 1; blast < 0 && b >= 0; --b)
        if (cnt[b]) blast = b;
      bs = blast;
      js = cnt[bs];
    }
    hd.pc[1] = bs;
    hd.pc[2] = js;
    hd.pc[3] = -1;
    hd.zf = x;
  }
  __syncthreads();
  const int bs = hd.pc[1], js = hd.pc[2];
  const float vs = bf16_key_val(khi - bs);
  const bool part = js < cnt[bs];  // the cut bucket is taken in part: rank its elements by index
  for (int i = tid; i < n; i += kThreads) {
    const float v = pval[i];
    const int x = pidx[i];
    bool keep = v > vs;
    if (v == vs) {
      int r = 0;
      if (part)
        for (int q = 0; q < n; ++q) r += (pval[q] == vs && pidx[q] < x) ? 1 : 0;
      keep = r < js;
      if (keep) atomicMax(&hd.pc[3], x);
    }
    if (keep) atomicOr(&bm[x >> 5], 1u << (x & 31));
  }
  __syncthreads();
  // positions: a prefix count of the bitmap, in runs of words per thread
  const int wper = (nw + kThreads - 1) / kThreads;
  const int w0 = min(nw, tid * wper), w1 = min(nw, w0 + wper);
  int pc = 0;
  for (int w = w0; w < w1; ++w) pc += __popc(bm[w]);
  int nkeep;
  const int pre = block_excl_scan_i(pc, &nkeep, sm);
  cnt[tid] = pre;  // the buckets are done with
  __syncthreads();
  if (nkeep <= kCap) {
    for (int i = tid; i < n; i += kThreads) {
      const int x = pidx[i];
      const int w = x >> 5;
      const uint32_t below = bm[w] & ((1u << (x & 31)) - 1u);
      if (!(bm[w] & (1u << (x & 31)))) continue;
      const int t = w / wper;
      int pos = cnt[t] + __popc(below);
      for (int q = t * wper; q < w; ++q) pos += __popc(bm[q]);
      lidx[pos] = x;
      lw[pos] = wexp(pval[i], m, c);
    }
    *list_len = nkeep;
  } else {
    *list_len = -1;
  }
  *cut = Cut{vs, hd.pc[3]};
  *zf = hd.zf;
  __syncthreads();
  return true;
}

// Bitonic sort of 32 R keys held by one warp (key i at lane i / R, slot
// i % R), descending.
template <int R>
__device__ __forceinline__ void warp_sort_keys_desc(unsigned long long (&key)[R]) {
  const int t = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32 * R; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < R) sort_stage_regs<R>(key, t, k, j);
      else sort_stage_lanes<R>(key, t, k, j);
    }
}

// list_ordered_draw for n <= 64 entries, by one warp (two entries a lane, lane
// l holding entries 2l and 2l + 1): the smallest i with u R < cumsum(i), the
// last positive entry on overflow, -1 if R == 0.  Same value on every lane.
template <typename WF>
__device__ int warp_list_draw(int n, double u, WF wf) {
  const int lane = threadIdx.x & 31;
  float w[2];
  FF pre[2];
  FF run = ff(0.0f);
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int i = 2 * lane + g;
    w[g] = (i < n) ? wf(i) : 0.0f;
    run = ff_add(run, w[g]);
    pre[g] = run;
  }
  const FF incl = warp_incl_scan_ff(run, lane);
  const FF excl = ff_sub(incl, run);
  const FF total = FF{__shfl_sync(FULL, incl.hi, 31), __shfl_sync(FULL, incl.lo, 31)};
  if (!(total.hi > 0.0f)) return -1;
  const FF target = ff_from_d(u * ff_to_d(total));
  int first = INT_MAX, last = -1;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int i = 2 * lane + g;
    const FF before = (g == 0) ? excl : ff_add(excl, pre[0]);
    const FF c = ff_add(excl, pre[g]);
    if (w[g] > 0.0f) {
      last = i;
      if (ff_lt(target, c) && !ff_lt(target, before)) first = min(first, i);
    }
  }
  first = static_cast<int>(__reduce_min_sync(FULL, static_cast<unsigned>(first)));
  last = static_cast<int>(__reduce_max_sync(FULL, static_cast<unsigned>(last + 1))) - 1;
  return (first != INT_MAX) ? first : last;
}

// This warp's part of a row: its stages, the row's whole vectors and their
// address (issue cursor of the ring).
struct RowRing {
  int my, nw;
  const uint4* src;
};
// A row of a streaming launch: a ragged call (a per-row table) or not.
__device__ __forceinline__ RowInfo stream_job(const KArgs& a, int row) {
  return a.row_map ? decode_job<true>(a, row) : decode_job<false>(a, row);
}

template <typename E>
__device__ __noinline__ RowRing row_ring(const KArgs& a, int row, int warp) {
  constexpr int N = Seg<E>::N;
  const RowInfo ri = stream_job(a, row);
  RowRing r;
  const int nv = (a.V + N - 1) / N, nst = (nv + kSWV - 1) / kSWV;
  r.my = (nst > warp) ? (nst - warp + kWarps - 1) / kWarps : 0;
  r.nw = a.V / N;
  r.src = reinterpret_cast<const uint4*>(static_cast<const E*>(ri.is_target ? a.tgt : a.drf) + ri.row_off);
  return r;
}

// The row record, the draw of a sampled row, and (rows before a sequence's
// last draft position) the draft token's adjusted probability.  One thread.
// kept: the cut (tv, ti) and mass zf; list_len < 0 when no list is stored.
// wd(d): the weight of token d when it is kept, else 0.
template <typename WD>
__device__ void stream_record(const KArgs& a, const RowInfo& ri, float m, int argmax, bool bad, Cut cut, FF zf,
                              int list_len, int tok, WD wd) {
  spec_row_stat* rec = a.rows + ri.job;
  int flags = bad ? kFlagNonfinite : 0;
  double p_tok = 0.0;
  if (a.mode == kModeVerify && ri.t < ri.kb && !a.fused) {
    const int d = a.tokens[static_cast<int64_t>(ri.b) * a.K + ri.t];
    if (d < 0 || d >= a.V) {
      flags |= kFlagToken;
    } else if (!bad && !a.greedy) {
      const float w = wd(d);
      if (w > 0.0f) p_tok = static_cast<double>(w) / ff_to_d(zf);
    }
  }
  if (a.mode == kModeSample || (a.fused && !ri.is_target)) {
    if (a.fused) a.out_draft[ri.b] = tok;
    else a.out_tokens[static_cast<int64_t>(ri.b) * a.K + ri.t] = tok;
    rec->token = tok;
    if (a.mode == kModeSample && bad) set_status(a, SPEC_ERR_NONFINITE);
  }
  rec->zf = ff_to_d(zf);
  rec->p_tok = p_tok;
  rec->m = m;
  rec->tau_val = cut.tv;
  rec->tau_idx = cut.ti;
  rec->argmax = argmax;
  rec->list_len = list_len;
  rec->flags = flags;
}

// The sequence epilogue of a sampling call whose rows all stored their kept
// lists (the streaming kernel's top-k rows): the records of every row in one
// round of loads, the accept tests, then the two lists the final draw needs
// in one more round, both held in shared memory.  The arithmetic is the
// verify epilogue's.  Falls back to it for lists it does not hold.
// recs: shared scratch for 128 rows (flags, p_tok, zf, list_len).
template <typename E>
__device__ void stream_epilogue(const KArgs& a, int b, int K, int first, Scratch& sm, unsigned char* recs) {
  const int KS = a.K;
  const int R = 2 * K + 1;
  const int tid = threadIdx.x;
  if (R > kThreads) {
    verify_epilogue<E>(a, b, K, first, sm);
    return;
  }
  double* sp = reinterpret_cast<double*>(recs);
  double* sz = sp + kThreads;
  int32_t* sf = reinterpret_cast<int32_t*>(sz + kThreads);
  int32_t* sl = sf + kThreads;
  if (tid < R) {
    const spec_row_stat* r = a.rows + first + tid;
    sp[tid] = __ldcg(&r->p_tok);
    sz[tid] = __ldcg(&r->zf);
    sf[tid] = __ldcg(&r->flags);
    sl[tid] = __ldcg(&r->list_len);
  }
  if (tid == 0) {
    sm.bi[12] = 0;
    sm.bi[13] = K;
  }
  __syncthreads();
  if (tid < R && sf[tid]) atomicOr(&sm.bi[12], sf[tid]);
  // keep d_t with probability min(1, tgt/drf):  u * drf < tgt
  if (tid < K && !(a.u[static_cast<int64_t>(b) * (KS + 1) + tid] * sp[K + 1 + tid] < sp[tid])) atomicMin(&sm.bi[13], tid);
  __syncthreads();
  const int fl = sm.bi[12], n = sm.bi[13];
  const bool resid = n < K;
  const int rt = n, rd = K + 1 + n;
  const int lt = sl[rt], ld = resid ? sl[rd] : 0;
  constexpr int kHalf = kCap / 2;
  if (!fl && (lt < 0 || ld < 0 || lt > kHalf || ld > kHalf)) {
    __syncthreads();
    verify_epilogue<E>(a, b, K, first, sm);
    return;
  }
  int32_t* out = a.out_tokens + static_cast<int64_t>(b) * (KS + 1);
  if (fl) {
    for (int t = tid; t <= KS; t += kThreads) out[t] = -1;
    if (tid == 0) {
      a.out_n[b] = -1;
      set_status(a, (fl & kFlagToken) ? SPEC_ERR_TOKEN_RANGE
                                      : (fl & kFlagTimeout) ? SPEC_ERR_TIMEOUT : SPEC_ERR_NONFINITE);
    }
    return;
  }
  for (int t = tid; t <= KS; t += kThreads) out[t] = (t < n) ? a.tokens[static_cast<int64_t>(b) * KS + t] : -1;
  // the two kept lists (index order) the draw needs
  int32_t* ti = sm.cand_idx;
  float* tw = sm.cand_val;
  int32_t* di = sm.cand_idx + kHalf;
  float* dw = sm.cand_val + kHalf;
  {
    const int64_t jt = static_cast<int64_t>(first) + rt, jd = static_cast<int64_t>(first) + rd;
    for (int i = tid; i < lt + ld; i += kThreads) {
      if (i < lt) {
        ti[i] = __ldcg(&a.list_idx[jt * kCap + i]);
        tw[i] = __ldcg(&a.list_w[jt * kCap + i]);
      } else {
        di[i - lt] = __ldcg(&a.list_idx[jd * kCap + (i - lt)]);
        dw[i - lt] = __ldcg(&a.list_w[jd * kCap + (i - lt)]);
      }
    }
  }
  __syncthreads();
  auto drf_w = [&](int x) -> float {
    int lo = 0, hi = ld;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (di[mid] < x) lo = mid + 1;
      else hi = mid;
    }
    return (lo < ld && di[lo] == x) ? dw[lo] : 0.0f;
  };
  const double u = a.u[static_cast<int64_t>(b) * (KS + 1) + K];
  const float izt = 1.0f / static_cast<float>(sz[rt]), izd = 1.0f / static_cast<float>(resid ? sz[rd] : 1.0);
  auto resid_w = [&](int i) { return fmaxf(0.0f, tw[i] * izt - drf_w(ti[i]) * izd); };
  auto tgt_w = [&](int i) { return tw[i]; };
  if (lt <= 64) {
    // one warp: two entries a lane, no block barriers
    if (threadIdx.x < 32) {
      int pos = resid ? warp_list_draw(lt, u, resid_w) : -1;
      if (pos < 0) pos = warp_list_draw(lt, u, tgt_w);
      if (tid == 0) {
        out[n] = (pos >= 0) ? ti[pos] : -1;
        a.out_n[b] = n;
      }
    }
    return;
  }
  int pos = -1;
  if (resid) pos = list_ordered_draw(lt, u, sm, resid_w);
  if (pos < 0) pos = list_ordered_draw(lt, u, sm, tgt_w);
  if (tid == 0) {
    out[n] = (pos >= 0) ? ti[pos] : -1;
    a.out_n[b] = n;
  }
}

// MODE: kSMGreedy (the max and first argmax alone), kSMTopK (top-k candidate
// groups), kSMTopP (candidate groups and the normaliser; top-p alone).
template <typename E, int MODE>
__global__ void __launch_bounds__(kThreads, 4) spec_stream_kernel(const KArgs a) {
  constexpr bool CAND = MODE != kSMGreedy, TOPP = MODE == kSMTopP;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Scratch& sm = *reinterpret_cast<Scratch*>(smem_raw);
  StreamHdr& hd = *reinterpret_cast<StreamHdr*>(smem_raw + sizeof(Scratch));
  unsigned char* ring = smem_raw + sizeof(Scratch) + sizeof(StreamHdr);
  unsigned char* cand = ring + kSRing;  // CAND: the warps' buffers
  constexpr int N = Seg<E>::N;
  constexpr int KB = sizeof(E) == 2 ? 16 : 32;  // significant key bits of an element
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned char* wring = ring + static_cast<size_t>(warp) * kSNS * kSStage;
  uint64_t* wbar = hd.bar + warp * kSNS;
  uint2* wc = reinterpret_cast<uint2*>(cand) + warp * kSWCap;  // CAND: this warp's buffer
  const int G = static_cast<int>(gridDim.x);
  const int ktop = a.top_k;
  // buffer entries that trigger a cut, and the groups the cut keeps
  const int hwm = TOPP ? kSPHwm : max(kSWCap * 5 / 8, 2 * ktop);
  const int keep = TOPP ? kSPKeep : ktop;
  const int nv = (a.V + N - 1) / N, nw = a.V / N;  // vectors of a row, whole ones

  if (lane == 0) {
    for (int b = 0; b < kSNS; ++b) mbar_init(&wbar[b], 1);
    fence_mbar_init();
  }
  if (tid < kWarps) hd.wthr[tid] = -INFINITY;
  __syncthreads();
  uint32_t phase = 0;   // bit b: parity of buffer b's next completion
  uint32_t pending = 0; // lane 0, bit b: buffer b has a copy whose completion was not seen
  bool staged = true;   // this warp still uses bulk copies
  int bnext = 0;        // buffer of this warp's next stage

  // lane 0's issue cursor: row ir, its stage ik, buffer ib.  Top-p stops at
  // the end of row ilim: its row end works in the drained ring.
  int ir = static_cast<int>(blockIdx.x), ik = 0, ib = 0, inflight = 0;
  int ilim = TOPP ? ir : INT_MAX;
  RowRing ig{0, 0, nullptr};
  if (lane == 0 && ir < a.nrows) ig = row_ring<E>(a, ir, warp);
  auto top_up = [&]() {
    while (staged && inflight < kSNS && ir < a.nrows) {
      if (ik >= ig.my) {
        if (ir >= ilim) break;
        ir += G;
        ik = 0;
        if (ir < a.nrows) ig = row_ring<E>(a, ir, warp);
        continue;
      }
      const int vs = (warp + kWarps * ik) * kSWV;
      const int nb = max(0, min(ig.nw - vs, kSWV));
      mbar_expect_tx(&wbar[ib], static_cast<uint32_t>(nb) * 16u);
      if (nb > 0) bulk_copy_g2s(wring + ib * kSStage, ig.src + vs, static_cast<uint32_t>(nb) * 16u, &wbar[ib]);
      pending |= 1u << ib;
      ib = (ib + 1 == kSNS) ? 0 : ib + 1;
      ++ik;
      ++inflight;
    }
  };
  if (lane == 0) top_up();

  for (int row = static_cast<int>(blockIdx.x); row < a.nrows; row += G) {
    if (TOPP && lane == 0 && ilim < row) {  // the ring is free again: this row's copies
      fence_proxy_async_smem();  // after the last row end's generic accesses to the ring
      ilim = row;
      top_up();
    }
    const RowInfo ri = stream_job(a, row);
    const E* grow = static_cast<const E*>(ri.is_target ? a.tgt : a.drf) + ri.row_off;
    const uint4* gv = reinterpret_cast<const uint4*>(grow);
    const int nst = (nv + kSWV - 1) / kSWV;
    const int my = (nst > warp) ? (nst - warp + kWarps - 1) / kWarps : 0;

    float rmax = -INFINITY;
    int rarg = INT_MAX;
    float zm = -INFINITY;   // TOPP: the lane's normaliser z, relative to zm
    FF z = ff(0.0f);
    float thr = -INFINITY;  // CAND: this warp's threshold (warp-uniform)
    int wn = 0;             // CAND: entries in the warp's buffer
    bool wover = false;     // CAND: the buffer could not take a stage

    for (int k = 0; k < my; ++k) {
      const int b = bnext;
      bnext = (b + 1 == kSNS) ? 0 : b + 1;
      const int vs = (warp + kWarps * k) * kSWV;
      bool from_smem = false;
      if (staged) {
        bool ok = mbar_try_wait(&wbar[b], (phase >> b) & 1u);
        if (!ok) ok = mbar_wait_bounded(&wbar[b], (phase >> b) & 1u);
        from_smem = __all_sync(FULL, ok);
        if (from_smem) {
          phase ^= 1u << b;
          pending &= ~(1u << b);
        } else {  // a copy was lost: this warp reads the rows itself from now on
          staged = false;
          set_status(a, SPEC_ERR_TIMEOUT);
        }
      }
      const uint32_t wbase = smem_addr(wring + b * kSStage);
      // vector j of this lane (vector vs + 32 j + lane of the row)
      auto vec = [&](int j) -> uint4 {
        const int t = j * 32 + lane, v = vs + t;
        if (v < nw) return from_smem ? ld_shared_v4(wbase + static_cast<uint32_t>(t) * 16u) : ld_stream(gv + v);
        if (v < nv) return Seg<E>::load_some(grow, v, a.V - v * N);
        return Seg<E>::neg_inf();
      };
      uint4 q[kSVPL];
      if (from_smem && vs + kSWV <= nw) {
#pragma unroll
        for (int j = 0; j < kSVPL; ++j) q[j] = ld_shared_v4(wbase + static_cast<uint32_t>(j * 32 + lane) * 16u);
      } else {
#pragma unroll
        for (int j = 0; j < kSVPL; ++j) q[j] = vec(j);
      }
      // the lane's max over its vectors (NaN-propagating), and each vector's
      uint32_t pw[kSVPL];
      const float tm = Seg<E>::template lane_max<kSVPL>(q, pw);
      // a new running max: the first element that holds it (the lane meets its
      // elements in index order)
      if (tm > rmax) {
        int jf = kSVPL - 1;
#pragma unroll
        for (int j = kSVPL - 1; j >= 0; --j) jf = (Seg<E>::pw_max(pw[j]) == tm) ? j : jf;
        uint4 x = q[0];
#pragma unroll
        for (int j = 1; j < kSVPL; ++j) x = (j == jf) ? q[j] : x;
        int ef = 0;
#pragma unroll
        for (int i = N - 1; i >= 0; --i) ef = (Seg<E>::get(x, i) == tm) ? i : ef;
        rarg = (vs + jf * 32 + lane) * N + ef;
      }
      rmax = max_nan(rmax, tm);
      if constexpr (TOPP) {
        // the normaliser: the group's sum relative to its max, folded into the
        // lane's (rescaled when the group holds a new max)
        if (tm > -INFINITY) {  // false for NaN: such a row takes the general path
          float s;
          if constexpr (sizeof(E) == 2) {
            s = Seg<E>::template zsum<kSVPL>(q, tm, a.c);
          } else {
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int j = 0; j < kSVPL; ++j)
#pragma unroll
              for (int i = 0; i < N; i += 2) {
                s0 += wexp(Seg<E>::get(q[j], i), tm, a.c);
                s1 += wexp(Seg<E>::get(q[j], i + 1), tm, a.c);
              }
            s = s0 + s1;
          }
          if (tm > zm) {
            z = ff_add(ff_mul(z, wexp(zm, tm, a.c)), s);
            zm = tm;
          } else {
            z = ff_add(z, s * wexp(tm, zm, a.c));
          }
        }
      }

      if constexpr (CAND) {
        if (!wover) {
          // a lane's group: its kSVPL vectors of the stage.  The row's top k
          // elements lie in the k groups with the largest maxima, so the warp
          // keeps (group max, group) for every group whose max reaches its
          // threshold; the elements are picked out at the row end.
          // The first stage: the k-th largest finite vector maximum (at least
          // k elements reach it).
          if (!TOPP && k == 0) {
            const uint32_t t = warp_select_key<kSVPL, KB>(
                [&](int j) {
                  const float v = Seg<E>::pw_max(pw[j]);
                  return (v > -INFINITY && v < INFINITY) ? okey32(v) : 0u;
                },
                ktop);
            thr = fmaxf(thr, key_floor(t));
          }
          float te = thr;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) te = fmaxf(te, reinterpret_cast<volatile float*>(hd.wthr)[w]);
          // a buffer past its high-water mark is cut to its k largest groups
          // first (k group maxima at or above a value: k elements at or above it)
          if (wn >= hwm) {
            te = fmaxf(te, warp_buffer_kth<E>(wc, wn, keep));
            wn = warp_buffer_compact(wc, wn, te);
          }
          const bool hot = tm >= te;  // false for NaN
          const unsigned hb = __ballot_sync(FULL, hot);
          if (hb) {
            const int c = __popc(hb);
            if (wn + c > kSWCap) {
              wover = true;  // ties beyond the buffer: the row takes the general path
            } else {
              if (hot) {
                // top-p: which of the group's vectors reach te (only those can
                // hold an element >= any later floor)
                uint32_t vmk = 0;
                if constexpr (TOPP) {
#pragma unroll
                  for (int j = 0; j < kSVPL; ++j) vmk |= (Seg<E>::pw_max(pw[j]) >= te) ? (1u << j) : 0u;
                }
                wc[wn + __popc(hb & ((1u << lane) - 1u))] =
                    make_uint2(static_cast<uint32_t>(vs + lane) | (vmk << kSVShift), __float_as_uint(tm));
              }
              wn += c;
              __syncwarp();
            }
          }
          if (te > thr) {
            thr = te;
            if (lane == 0) hd.wthr[warp] = thr;
          }
        }
      }
      // the warp is done with the buffer: lane 0 refills the ring
      __syncwarp();
      if (lane == 0) {
        --inflight;
        top_up();
      }
    }

    // ---- row end: max, first argmax (lowest index among the lanes that hold it)
    float wm = rmax;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = max_nan(wm, __shfl_xor_sync(FULL, wm, o));
    int wa = (rmax == wm) ? rarg : INT_MAX;  // false for NaN
    wa = static_cast<int>(__reduce_min_sync(FULL, static_cast<unsigned>(wa)));
    if constexpr (TOPP) {
      // the warp's normaliser relative to its max (float-float butterfly)
      FF wz = (z.hi > 0.0f) ? ff_mul(z, wexp(zm, wm, a.c)) : ff(0.0f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        wz = ff_add(wz, FF{__shfl_xor_sync(FULL, wz.hi, o), __shfl_xor_sync(FULL, wz.lo, o)});
      if (lane == 0) hd.wz[warp] = wz;
    }
    if (lane == 0) {
      hd.wmax[warp] = wm;
      hd.warg[warp] = wa;
      hd.wflag[warp] = wover ? kSegOver : 0;
    }
    if (tid == 0) {
      hd.nlist = 0;
      hd.cut = 0;
    }
    if (CAND && tid < 48) hd.rbins[tid] = 0u;
    __syncthreads();
    float m = -INFINITY, f = -INFINITY;
    int am = INT_MAX, fl = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) m = max_nan(m, hd.wmax[w]);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (hd.wmax[w] == m) am = min(am, hd.warg[w]);
      fl |= hd.wflag[w];
      f = fmaxf(f, hd.wthr[w]);
    }
    const bool bad = !(m == m) || m == INFINITY || !(m > -INFINITY);
    const int argmax = (am == INT_MAX) ? -1 : am;
    __syncthreads();  // the thresholds are read: the next row starts from none
    if (tid < kWarps) hd.wthr[tid] = -INFINITY;

    if constexpr (!CAND) {
      if (tid == 0)
        stream_record(a, ri, m, argmax, bad, cut_all(), ff(0.0f), -1, bad ? -1 : argmax, [](int) { return 0.0f; });
    } else if constexpr (TOPP) {
      // ---- top-p: every element >= f lies in a buffered group.  A tighter
      // floor f2 >= f is the largest group max such that the maxima of the
      // groups at or above it alone weigh at least top_p * Z: at least that
      // mass lies at or above f2, so the nucleus does too.  The elements >= f2
      // of those groups are read back from the row into a pool (the ring is
      // drained), sorted (value desc, index asc) and cut where the prefix mass
      // reaches top_p * Z.
      int32_t* pidx = reinterpret_cast<int32_t*>(ring);
      float* pval = reinterpret_cast<float*>(pidx + kPool);
      unsigned long long* skey = reinterpret_cast<unsigned long long*>(pval + kPool);
      int32_t* gsel = reinterpret_cast<int32_t*>(skey + kPool);
      // the row's normaliser: every warp's sum rescaled to the row max, in warp order
      FF zrow = ff(0.0f);
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        if (hd.wz[w].hi > 0.0f) zrow = ff_add(zrow, ff_mul(hd.wz[w], wexp(hd.wmax[w], m, a.c)));
      bool general = bad || (fl & kSegOver) || !(zrow.hi > 0.0f);
      constexpr int PER = kSWCap / 32;
      uint32_t gkey[PER];
      float gw[PER];
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        const int i = p * 32 + lane;
        const float g0v = (!general && i < wn) ? __uint_as_float(wc[i].y) : -INFINITY;
        const bool in = !general && i < wn && g0v >= f;
        gkey[p] = in ? okey32(g0v) : 0u;
        gw[p] = in ? wexp(g0v, m, a.c) : 0.0f;
      }
      float f2 = f;
      if (!general) {  // block-uniform
        // a small margin: the float sums of the weights may round up.  A
        // bisection (bins of masses would take contended float atomics)
        const float need = zrow.hi * a.top_p * (1.0f + 0x1p-10f);
        f2 = fmaxf(f, key_floor(block_select_mass<PER, KB>(gkey, gw, need, okey32(f), okey32(m), hd.wpart)));
      }
      // the marked vectors of the groups >= f2, listed
      {
        int cnt = 0;
#pragma unroll
        for (int p = 0; p < PER; ++p)
          if (gkey[p] != 0u && okey32_val(gkey[p]) >= f2) cnt += __popc(wc[p * 32 + lane].x >> kSVShift);
        int pos = warp_reserve(&hd.cut, cnt);
#pragma unroll
        for (int p = 0; p < PER; ++p)
          if (gkey[p] != 0u && okey32_val(gkey[p]) >= f2) {
            const uint32_t e = wc[p * 32 + lane].x;
            const int v0 = static_cast<int>(e & ((1u << kSVShift) - 1u));
            for (uint32_t b = e >> kSVShift; b; b &= b - 1, ++pos)
              if (pos < kSPItems) gsel[pos] = v0 + (__ffs(b) - 1) * 32;
          }
      }
      __syncthreads();
      general = general || hd.cut > kSPItems;
      if (!general) {
        const int ni = hd.cut;
        const float tf = Seg<E>::grid_floor(f2);
        // item = (group, vector of the group); the loads of a round go out together
        constexpr int R = 8;
        for (int base = 0; base < ni; base += R * kThreads) {
          uint4 x[R];
          int vv[R];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int it = base + r * kThreads + tid;
            vv[r] = -1;
            x[r] = Seg<E>::neg_inf();
            if (it < ni) {
              const int v = gsel[it];
              vv[r] = v;
              if (v < nw) x[r] = ld_stream(gv + v);
              else if (v < nv) x[r] = Seg<E>::load_some(grow, v, a.V - v * N);
            }
          }
          uint32_t mk[R];
          int cnt = 0;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            mk[r] = (vv[r] >= 0) ? Seg<E>::ge_mask(x[r], tf) : 0u;
            cnt += __popc(mk[r]);
          }
          int pos = warp_reserve(&hd.nlist, cnt);
#pragma unroll
          for (int r = 0; r < R; ++r)
            for (uint32_t b = mk[r]; b; b &= b - 1, ++pos) {
              const int i = __ffs(b) - 1;
              if (pos < kPool) {
                pidx[pos] = vv[r] * N + i;
                pval[pos] = Seg<E>::get(x[r], i);
              }
            }
        }
      }
      __syncthreads();
      const int n = hd.nlist;
      general = general || n > kPool || n < 1;
      if (!general) {
        int32_t* lidx = a.list_idx + static_cast<int64_t>(row) * kCap;
        float* lw = a.list_w + static_cast<int64_t>(row) * kCap;
        Cut kc = cut_all();
        FF kz = zrow;
        int list_len = -1;
        bool done = false;
        if constexpr (sizeof(E) == 2) {
          // bf16: by counting (the ring past the pool holds the buckets and the bitmap)
          int* cnt = reinterpret_cast<int*>(skey);
          uint32_t* bm = reinterpret_cast<uint32_t*>(gsel);
          constexpr int kBm = static_cast<int>((kSRing - 2 * kPool * sizeof(int32_t) - kPool * sizeof(unsigned long long)) /
                                               sizeof(uint32_t));
          done = pool_bucket_cut(a.V, m, a.c, a.top_p, zrow, n, pidx, pval, Seg<E>::grid_floor(f2), cnt, bm, kBm, hd,
                                 sm, lidx, lw, &kc, &kz, &list_len);
        }
        if (!done) {
          const CutResult res = sort_and_cut(m, a.c, pidx, pval, n, SortBuf{skey, nullptr}, 0, a.top_p, zrow, sm);
          if (res.reached) {
            if (res.nkeep <= kCap) {
              write_kept_by_index(skey, res.nkeep, m, a.c, lidx, lw, sm);
              list_len = res.nkeep;
            }
            kc = Cut{res.tv, res.ti};
            kz = res.zf;
            done = true;
          }
        }
        if (done) row_tail<E>(a, ri, grow, sm, m, argmax, false, kc, kz, list_len);
        else general = true;  // the pool's mass stays below top_p * Z
        __syncthreads();
      }
      if (general) {
        // the exact general path, with the row's max, argmax and normaliser
        if (tid == 0) {
          SegRec* rec = a.segs + row;
          rec->m = m;
          rec->argmax = argmax;
          rec->z_hi = zrow.hi;
          rec->z_lo = zrow.lo;
          rec->theta = -INFINITY;
          rec->kth = -INFINITY;
          rec->ncand = 0;
          rec->flags = (bad ? kSegBad : 0) | kSegOver;
        }
        __syncthreads();
        Local C;
        const SortBuf sb{reinterpret_cast<unsigned long long*>(cand), reinterpret_cast<uint8_t*>(sm.cand_idx)};
        row_finish<E>(a, ri, grow, sm, C, sb, reinterpret_cast<int32_t*>(cand), reinterpret_cast<float*>(cand));
      }
    } else {
      // ---- top-k: the groups whose max is >= f hold every element >= f; their
      // elements >= f are read back from the row (the copies are gone) and
      // ranked (value desc, index asc)
      unsigned long long* keys = reinterpret_cast<unsigned long long*>(sm.cand_idx);
      int32_t* gsel = reinterpret_cast<int32_t*>(keys + kSKeys);
      bool general = bad || (fl & kSegOver);
      // every group whose max is >= f is buffered, so the k-th largest
      // buffered group max is the row's: a tighter floor f2 (at least k groups,
      // so k elements, reach it); then the groups >= f2 are listed
      constexpr int PER = kSWCap / 32;
      uint32_t gkey[PER];
      int gone[PER];
#pragma unroll
      for (int p = 0; p < PER; ++p) {
        const int i = p * 32 + lane;
        const float g = (!general && i < wn) ? __uint_as_float(wc[i].y) : -INFINITY;
        const bool in = !general && i < wn && g >= f;
        gkey[p] = in ? okey32(g) : 0u;
        gone[p] = in ? 1 : 0;
      }
      float f2 = f;
      if (!general) f2 = fmaxf(f, key_floor(block_radix_select<PER, KB, int>(gkey, gone, ktop, hd.rbins)));
      {
        int cnt = 0;
#pragma unroll
        for (int p = 0; p < PER; ++p) cnt += (gkey[p] != 0u && okey32_val(gkey[p]) >= f2) ? 1 : 0;
        int pos = warp_reserve(&hd.cut, cnt);
#pragma unroll
        for (int p = 0; p < PER; ++p)
          if (gkey[p] != 0u && okey32_val(gkey[p]) >= f2) {
            if (pos < kSGroups) gsel[pos] = static_cast<int>(wc[p * 32 + lane].x);
            ++pos;
          }
      }
      __syncthreads();
      if (!general) {
        f = f2;
        const int ng2 = (hd.cut <= kSGroups) ? hd.cut : 0;  // more: the general path (no keys)
        const float tf = Seg<E>::grid_floor(f);
        // item = (group, vector of the group); the loads of a round go out together
        constexpr int R = 4;
        for (int base = 0; base < ng2 * kSVPL; base += R * kThreads) {
          uint4 x[R];
          int vv[R];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int it = base + r * kThreads + tid;
            vv[r] = -1;
            x[r] = Seg<E>::neg_inf();
            if (it < ng2 * kSVPL) {
              const int g = it / kSVPL, j = it - g * kSVPL;
              const int v = gsel[g] + j * 32;
              vv[r] = v;
              if (v < nw) x[r] = ld_stream(gv + v);
              else if (v < nv) x[r] = Seg<E>::load_some(grow, v, a.V - v * N);
            }
          }
          uint32_t mk[R];
          int cnt = 0;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            mk[r] = (vv[r] >= 0) ? Seg<E>::ge_mask(x[r], tf) : 0u;
            cnt += __popc(mk[r]);
          }
          int pos = warp_reserve(&hd.nlist, cnt);
#pragma unroll
          for (int r = 0; r < R; ++r)
            for (uint32_t b = mk[r]; b; b &= b - 1, ++pos) {
              const int i = __ffs(b) - 1;
              if (pos < kSKeys) keys[pos] = sort_key(Seg<E>::get(x[r], i), vv[r] * N + i);
            }
        }
      }
      __syncthreads();
      const int n = hd.nlist;
      general = general || n > kSKeys || n < 1;
      // warp 0 alone: sort the keys (value desc, index asc) in registers, cut
      // top-k then top-p with float-float prefix masses, sort the kept set by
      // index, write it with the record, and draw a sampled row's token
      if (!general) {
        if (warp == 0) {
          unsigned long long key[2];
          if (n <= 64) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int i = 2 * lane + r;
              key[r] = (i < n) ? keys[i] : 0ull;  // zero keys sort last
            }
            warp_sort_keys_desc<2>(key);
          } else {
            // up to 256 keys: sorted eight a lane, then the first 64 two a lane
            unsigned long long k8[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const int i = 8 * lane + r;
              k8[r] = (i < n) ? keys[i] : 0ull;
            }
            warp_sort_keys_desc<8>(k8);
            __syncwarp();
            if (lane < 8) {
#pragma unroll
              for (int r = 0; r < 8; ++r) keys[8 * lane + r] = k8[r];
            }
            __syncwarp();
#pragma unroll
            for (int r = 0; r < 2; ++r) key[r] = keys[2 * lane + r];
          }
          const int kk = min(ktop, n);
          float w2[2];
          FF pre[2];
          FF run = ff(0.0f);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int i = 2 * lane + g;
            w2[g] = (i < kk) ? wexp(skey_val(key[g]), m, a.c) : 0.0f;
            run = ff_add(run, w2[g]);
            pre[g] = run;
          }
          const FF incl = warp_incl_scan_ff(run, lane);
          const FF excl = ff_sub(incl, run);
          const FF total = FF{__shfl_sync(FULL, incl.hi, 31), __shfl_sync(FULL, incl.lo, 31)};
          int cut = kk - 1;
          if (a.top_p < 1.0f) {
            const FF need = ff_mul(total, a.top_p);
            int first = INT_MAX;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const int i = 2 * lane + g;
              if (i < kk && !ff_lt(ff_add(excl, pre[g]), need)) first = min(first, i);
            }
            first = static_cast<int>(__reduce_min_sync(FULL, static_cast<unsigned>(first)));
            if (first != INT_MAX) cut = first;
          }
          const int nkeep = cut + 1;
          // the kept mass and the cut key, from the lane that holds the cut
          const int hl = cut >> 1;
          const FF zc = ff_add(excl, pre[cut & 1]);
          const FF zf = FF{__shfl_sync(FULL, zc.hi, hl), __shfl_sync(FULL, zc.lo, hl)};
          const unsigned long long ck = __shfl_sync(FULL, (cut & 1) ? key[1] : key[0], hl);
          const Cut kc{skey_val(ck), skey_idx(ck)};
          // the kept set by index: (index asc) as a descending sort of its complement
          unsigned long long ik[2];
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int i = 2 * lane + g;
            ik[g] = (i < nkeep) ? ((static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(skey_idx(key[g]))) << 32) |
                                   __float_as_uint(w2[g]))
                                : 0ull;
          }
          warp_sort_keys_desc<2>(ik);
          int32_t* lidx = a.list_idx + static_cast<int64_t>(row) * kCap;
          float* lw = a.list_w + static_cast<int64_t>(row) * kCap;
          int32_t* sidx = sm.cand_idx;  // the keys are in registers: the list, for the draw
          float* sw = sm.cand_val;
          __syncwarp();
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int p = 2 * lane + g;
            if (p < nkeep) {
              const int xi = static_cast<int>(0xffffffffu - static_cast<uint32_t>(ik[g] >> 32));
              const float xw = __uint_as_float(static_cast<uint32_t>(ik[g]));
              lidx[p] = xi;
              lw[p] = xw;
              sidx[p] = xi;
              sw[p] = xw;
            }
          }
          __syncwarp();
          int tok = -1;
          if (a.mode == kModeSample || (a.fused && !ri.is_target)) {
            const double u = a.fused ? a.u_draft[ri.b] : a.u[static_cast<int64_t>(ri.b) * a.K + ri.t];
            const int pos = warp_list_draw(nkeep, u, [&](int i) { return sw[i]; });
            tok = (pos >= 0) ? sidx[pos] : -1;
          }
          // the kept weight of a token: a search of the kept list (index order)
          auto wd = [&](int d) {
            int lo = 0, hi = nkeep;
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (sidx[mid] < d) lo = mid + 1;
              else hi = mid;
            }
            return (lo < nkeep && sidx[lo] == d) ? sw[lo] : 0.0f;
          };
          if (lane == 0) stream_record(a, ri, m, argmax, false, kc, zf, nkeep, tok, wd);
        }
      } else {
        // the exact general path: the row's record says what the stream could
        // not settle (a non-finite row, or a buffer too small for its ties)
        if (tid == 0) {
          SegRec* rec = a.segs + row;
          rec->m = m;
          rec->argmax = argmax;
          rec->z_hi = 0.0f;
          rec->z_lo = 0.0f;
          rec->theta = -INFINITY;
          rec->kth = -INFINITY;
          rec->ncand = 0;
          rec->flags = (bad ? kSegBad : 0) | kSegOver;
        }
        __syncthreads();
        // with the record flagged, the merge gathers no pool (the pool arrays
        // are never touched) and the general path sorts at most kCap keys in
        // the candidate buffers
        Local C;
        const SortBuf sb{reinterpret_cast<unsigned long long*>(cand), reinterpret_cast<uint8_t*>(sm.cand_idx)};
        row_finish<E>(a, ri, grow, sm, C, sb, reinterpret_cast<int32_t*>(cand), reinterpret_cast<float*>(cand));
      }
    }

    // ---- the CTA that completes the sequence runs its epilogue
    __syncthreads();  // every global write of the row is ordered before the sequence counter
    if (a.mode == kModeVerify) {
      if (tid == 0) {
        fence_acq_rel_gpu();
        unsigned long long* tk = &a.tickets[ri.b];
        const bool last = atomicAdd(tk, 1ull) == static_cast<unsigned long long>(ri.nr - 1);
        if (last) {
          *tk = 0ull;  // the sequence's last row: no other arrival of this call
          fence_acq_rel_gpu();
        }
        hd.last = last ? 1 : 0;
      }
      __syncthreads();
      if (hd.last) {
        if (CAND && !a.fused) stream_epilogue<E>(a, ri.b, ri.kb, ri.first, sm, cand);
        else verify_epilogue<E>(a, ri.b, ri.kb, ri.first, sm);
      }
    }
    __syncthreads();  // the Scratch and the candidate buffers are free again
  }
  // copies whose completion was never seen (only after a lost one) must land
  // before the shared memory is released
  if (lane == 0)
    for (int b = 0; b < kSNS; ++b)
      if (pending & (1u << b)) (void)mbar_wait_bounded(&wbar[b], (phase >> b) & 1u);
}

}  // namespace
