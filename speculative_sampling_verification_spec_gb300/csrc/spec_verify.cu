// spec_verify.cu -- speculative-sampling verification on GB300 (sm_103a).
//
// Operation: "Speculative Decoding" (roadtointelligence.com), section "Draft,
// then verify", steps 1-4; filters before rejection sampling per the
// paperlayer.ai summary of "Accelerating Large Language Model Decoding with
// Speculative Sampling", section "Speculative Sampling"; greedy as argmax per
// the FDE Interviews breakdown of that paper, section "01 The paper in one
// minute".
//
// Design (one launch per call):
//   * Every vocabulary row the method reads is one job.  A job runs on a
//     thread-block cluster of CS CTAs; CTA r holds elements [r*S, r*S + S) of
//     the row in shared memory, brought in by bulk asynchronous copies
//     (cp.async.bulk + mbarrier) in up to four stages, scanned for the max as
//     the stages land.  The row is read from HBM once; every later pass reads
//     shared memory.
//   * Row statistics (max, argmax, normaliser) and the top-k / top-p cut are
//     reduced across the cluster through distributed shared memory.  Every CTA
//     reduces the published per-CTA values in rank order, so all CTAs hold
//     bit-identical results and take identical branches.
//   * The cut is exact: an 8-probe bracket search over the order-preserving
//     key of the logits narrows [lo, hi) until the elements >= lo fit the
//     on-chip sort (<= kCap, by (logit desc, index asc)), or until the bracket
//     holds a single key value, whose tie group is cut by index.
//   * Each row writes a record (normaliser, cut, draft-token probability, the
//     kept set in index order when it fits) to the caller's workspace.  The
//     last cluster of a sequence to finish (atomic ticket, no spinning) runs
//     the accept tests and the one final draw for that sequence.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "spec_verify.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 512;       // on-chip sort capacity == stored kept-list capacity
constexpr int kWarpCap = kCap / 8;  // first-pass candidate list per warp (8 warps)
constexpr int kProbes = 8;      // thresholds evaluated per probe pass
constexpr int kStages = 4;      // bulk-copy stages per slice
constexpr int kMaxCluster = 8;  // portable cluster size
constexpr int kMaxPasses = 40;  // bound on probe passes (16-bit keys need <= 6, 32-bit <= 11)
constexpr unsigned FULL = 0xffffffffu;

constexpr int kFlagNonfinite = 1, kFlagToken = 2, kFlagTimeout = 4;

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
// Bounded wait on phase 0 of a stage barrier: gives up after ~2 s of wall time
// (and after a hard iteration cap), so a lost copy cannot hang the GPU.
__device__ bool mbar_wait_bounded(uint64_t* bar) {
  if (mbar_try_wait(bar, 0)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < 100000u; ++it) {
    if (mbar_try_wait(bar, 0)) return true;
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
__device__ __forceinline__ float wexp(float l, float m, float c) { return exp2f((l - m) * c); }

// ---------------------------------------------------------------------------
// float-float ("double-single") sums.  GB300 runs FP64 at a small fraction of
// its FP32 rate, so running totals, prefix sums and cluster reductions keep a
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
__device__ __forceinline__ FF shfl_ff(FF v, int src) {
  return FF{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// ---------------------------------------------------------------------------
// kernel arguments and shared scratch

struct KArgs {
  const void* tgt;
  const void* drf;
  int64_t tgt_seq, tgt_row, drf_seq, drf_row;  // element strides
  const int32_t* tokens;                       // verify [B, K]
  const double* u;                             // verify [B, K+1], sample [B, K]
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* status;
  unsigned long long* tickets;  // [B]: (call tag << 32) | rows finished
  uint32_t tag;                 // nonzero, distinct for consecutive calls
  spec_row_stat* rows;  // [B * R]
  int32_t* list_idx;    // [B * R * kCap]
  float* list_w;        // [B * R * kCap]
  int B, K, V, R, S;    // R rows per sequence, S slice elements per CTA
  int mode, greedy, top_k, aligned;
  float top_p, c, temp;
};

struct Slot {  // per-CTA values published to the cluster
  FF d[kProbes + kWarps + 4];
  int32_t i[kProbes + kWarps + 4];
};

struct alignas(128) Scratch {
  uint64_t bar[kStages];
  Slot slot[2];
  Slot mirror[kMaxCluster];  // local copy of every rank's slot after an exchange
  // block-level reduction scratch
  float wf[kWarps];
  int32_t wi[kWarps];
  int32_t wi2[kWarps];
  FF wd[kWarps];
  int32_t pcnt[kProbes][kWarps];
  float pmass[kProbes][kWarps];
  FF wtot[kWarps];
  // values broadcast to the whole CTA by thread 0
  float m;
  int32_t argmax, bad, abort_;
  FF bd[kProbes + 4];
  int32_t bi[kProbes + 8];
  // candidates: this CTA's, and on rank 0 the cluster's gathered list
  int32_t cand_idx[kCap];
  float cand_val[kCap];
};

// Rank 0's sort buffers live in its slice buffer: on the path that sorts, the
// slice is no longer read once the candidates are gathered.
struct SortBuf {
  unsigned long long* skey;  // [kCap]
  FF* scan;                  // [kCap]
};
constexpr size_t kSortBufBytes = kCap * (sizeof(unsigned long long) + sizeof(FF));
// scratch + a 64 KB slice must leave room for three CTAs in an SM's 228 KB
static_assert(sizeof(Scratch) <= 8192, "shared scratch grew past its budget");
static_assert(sizeof(Slot) % sizeof(uint32_t) == 0, "slots are copied as 32-bit words");

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
// cluster exchange.  Thread 0 (or one lane) fills sm.slot[C.ph] first;
// exchange() is a cluster barrier (release/acquire), after which all threads copy
// every rank's slot of that phase into the local mirror at once -- one round of
// distributed-shared-memory loads instead of a serial chain -- and return it.
// Slots alternate between two buffers, so a rank may overwrite its slot for the
// next exchange while others still copy the previous one.  The mirror stays
// valid until the next exchange().  Every thread tracks the phase itself.

struct Cluster {
  cg::cluster_group cl;
  int cs, rank, ph;
  __device__ Cluster() : cl(cg::this_cluster()), ph(0) {
    cs = static_cast<int>(cl.num_blocks());
    rank = static_cast<int>(cl.block_rank());
  }
  __device__ Slot& mine(Scratch& sm) { return sm.slot[ph]; }
  __device__ const Slot* exchange(Scratch& sm) {
    const int p = ph;
    cl.sync();
    ph ^= 1;
    constexpr int W = static_cast<int>(sizeof(Slot) / sizeof(uint32_t));
    for (int i = threadIdx.x; i < cs * W; i += kThreads) {
      const int r = i / W, o = i - r * W;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(cl.map_shared_rank(&sm.slot[p], r));
      reinterpret_cast<uint32_t*>(&sm.mirror[r])[o] = src[o];
    }
    __syncthreads();
    return sm.mirror;
  }
};

// ---------------------------------------------------------------------------
// per-row state

struct RowInfo {
  int b, t, is_target, job;
  int64_t row_off;  // element offset of the row from its tensor base
  int tok;          // draft token at this row (verify, t < K), else -1
};

template <typename E>
struct RowCtx {
  const E* g;   // row in global memory
  const E* sl;  // this CTA's slice in shared memory
  int s0, L;    // slice start (row index) and length
  float m, c;
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
__device__ __forceinline__ auto smem_loader(const RowCtx<E>& rc) {
  return [&rc](int v, float (&x)[Fmt<E>::N]) { Fmt<E>::load(rc.sl, v, x); };
}

// ---- load + max/argmax/non-finite scan --------------------------------------
template <typename E>
__device__ void load_and_scan(const KArgs& a, const RowCtx<E>& rc, E* sl, Scratch& sm, Cluster& C) {
  constexpr int N = Fmt<E>::N;
  const int tid = threadIdx.x;
  float best = -INFINITY;
  int best_idx = INT_MAX;
  int bad = 0, abort_ = 0;

  auto scan_vec = [&](int v) {  // vector v of the slice
    bool nan;
    const float vm = Fmt<E>::vec_max(sl, v, nan);
    bad |= nan;
    if (vm > best) {  // rare: the running max rises O(log n) times per thread
      float x[N];
      Fmt<E>::load(sl, v, x);
      best = vm;
#pragma unroll
      for (int j = N - 1; j >= 0; --j)
        if (x[j] == vm) best_idx = rc.s0 + v * N + j;
    }
  };

  const int64_t bytes = static_cast<int64_t>(rc.L) * sizeof(E);
  const int64_t bulk = a.aligned ? (bytes & ~int64_t(15)) : 0;
  int nst = 0;
  int64_t chunk = 0;
  if (bulk > 0) {
    nst = static_cast<int>((bulk / 16 < kStages ? bulk / 16 : int64_t(kStages)));
    chunk = ((bulk / nst) + 15) & ~int64_t(15);
    nst = static_cast<int>((bulk + chunk - 1) / chunk);
    if (tid == 0) {
      for (int s = 0; s < nst; ++s) mbar_init(&sm.bar[s], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      const char* src = reinterpret_cast<const char*>(rc.g + rc.s0);
      char* dst = reinterpret_cast<char*>(sl);
      for (int s = 0; s < nst; ++s) {
        const int64_t off = s * chunk;
        const uint32_t sz = static_cast<uint32_t>((chunk < bulk - off ? chunk : bulk - off));
        mbar_expect_tx(&sm.bar[s], sz);
        bulk_copy_g2s(dst + off, src + off, sz, &sm.bar[s]);
      }
    }
  }
  // elements past the bulk part (unaligned rows, or a ragged tail) by plain loads
  const int e_tail = static_cast<int>(bulk / static_cast<int64_t>(sizeof(E)));
  for (int e = e_tail + tid; e < rc.L; e += kThreads) sl[e] = rc.g[rc.s0 + e];

  for (int s = 0; s < nst; ++s) {
    if (!mbar_wait_bounded(&sm.bar[s])) abort_ = 1;
    const int v0 = static_cast<int>((s * chunk) / 16);
    const int v1 = static_cast<int>((bulk < (s + 1) * chunk ? bulk : (s + 1) * chunk) / 16);
    for (int v = v0 + tid; v < v1; v += kThreads) scan_vec(v);
  }
  __syncthreads();  // tail stores visible
  for (int e = e_tail + tid; e < rc.L; e += kThreads) {
    const float x = Fmt<E>::at(sl, e);
    bad |= (x != x);
    if (x > best) { best = x; best_idx = rc.s0 + e; }
  }

  // reduce (max value, lowest index), bad, abort
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(FULL, best, o);
    const int oi = __shfl_xor_sync(FULL, best_idx, o);
    if (ov > best || (ov == best && oi < best_idx)) { best = ov; best_idx = oi; }
    bad |= __shfl_xor_sync(FULL, bad, o);
    abort_ |= __shfl_xor_sync(FULL, abort_, o);
  }
  if (lane == 0) { sm.wf[warp] = best; sm.wi[warp] = best_idx; sm.wi2[warp] = bad | (abort_ << 1); }
  __syncthreads();
  if (tid == 0) {
    float bv = -INFINITY;
    int bi = INT_MAX, fl = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (sm.wf[w] > bv || (sm.wf[w] == bv && sm.wi[w] < bi)) { bv = sm.wf[w]; bi = sm.wi[w]; }
      fl |= sm.wi2[w];
    }
    Slot& s = C.mine(sm);
    s.d[0] = ff(bv);
    s.i[0] = bi;
    s.i[1] = fl;
  }
  const Slot* mir = C.exchange(sm);
  if (tid == 0) {
    float bv = -INFINITY;
    int bi = INT_MAX, fl = 0;
    for (int r = 0; r < C.cs; ++r) {
      const Slot* s = (&mir[r]);
      const float v = s->d[0].hi;
      const int i = s->i[0];
      if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
      fl |= s->i[1];
    }
    sm.m = bv;
    sm.argmax = bi;
    sm.bad = (fl & 1) || !(bv < INFINITY) || bi == INT_MAX;  // NaN, +inf, or no finite logit
    sm.abort_ = (fl >> 1) & 1;
  }
  __syncthreads();
}

// ---- cluster-wide ordered total of weights over the resident row -------------
// Leaves per-(rank, warp) totals in the mirror (d[1 + w] of each rank), for a
// following cluster_ordered_draw with the same weights and no exchange between.
template <typename E, typename WF>
__device__ FF cluster_weight_total(const RowCtx<E>& rc, Scratch& sm, Cluster& C, WF wf) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto wl = [&](float (&x)[N], int e0, int nvalid) {
#pragma unroll
    for (int j = 0; j < N; ++j) x[j] = (j < nvalid) ? wf(x[j], rc.s0 + e0 + j) : 0.0f;
  };
  const FF wt = warp_ordered_total<N>(rc.L, warp, lane, smem_loader(rc), wl);
  if (lane == 0) sm.wtot[warp] = wt;
  __syncthreads();
  if (threadIdx.x == 0) {
    Slot& s = C.mine(sm);
    FF tot = ff(0.0f);
    for (int w = 0; w < kWarps; ++w) {
      s.d[1 + w] = sm.wtot[w];
      tot = ff_add(tot, sm.wtot[w]);
    }
    s.d[0] = tot;
  }
  const Slot* mir = C.exchange(sm);
  if (threadIdx.x == 0) {
    FF z = ff(0.0f);
    for (int r = 0; r < C.cs; ++r) z = ff_add(z, mir[r].d[0]);
    sm.bd[0] = z;
  }
  __syncthreads();
  const FF z = sm.bd[0];
  __syncthreads();
  return z;
}

// Ordered draw over the cluster-resident row with the weights of the preceding
// cluster_weight_total (its totals still in the mirror).  The finding warp writes the token through
// `emit(token)`.
template <typename E, typename WF, typename Emit>
__device__ void cluster_ordered_draw(const RowCtx<E>& rc, Scratch& sm, Cluster& C, double u, WF wf,
                                     Emit emit) {
  const Slot* mir = sm.mirror;
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    FF total = ff(0.0f);
    for (int r = 0; r < C.cs; ++r)
      for (int w = 0; w < kWarps; ++w) total = ff_add(total, mir[r].d[1 + w]);
    const FF target = ff_from_d(u * ff_to_d(total));
    int fr = -1, fw = -1, lr = 0, lw = 0;
    FF base = ff(0.0f), cum = ff(0.0f);
    for (int r = 0; r < C.cs && fr < 0; ++r)
      for (int w = 0; w < kWarps; ++w) {
        const FF t = mir[r].d[1 + w];
        if (t.hi > 0.0f) { lr = r; lw = w; }
        const FF next = ff_add(cum, t);
        if (ff_lt(target, next)) { fr = r; fw = w; base = cum; break; }
        cum = next;
      }
    const int overflow = fr < 0;
    if (overflow) { fr = lr; fw = lw; }
    sm.bi[0] = fr;
    sm.bi[1] = fw;
    sm.bi[2] = overflow;
    sm.bd[0] = target;
    sm.bd[1] = base;
  }
  __syncthreads();
  const int fr = sm.bi[0], fw = sm.bi[1];
  const bool overflow = sm.bi[2] != 0;
  const FF target = sm.bd[0], base = sm.bd[1];
  __syncthreads();
  if (C.rank == fr && warp == fw) {
    auto wl = [&](float (&x)[N], int e0, int nvalid) {
#pragma unroll
      for (int j = 0; j < N; ++j) x[j] = (j < nvalid) ? wf(x[j], rc.s0 + e0 + j) : 0.0f;
    };
    const int e = warp_ordered_draw<N>(rc.L, warp, lane, smem_loader(rc), wl, target, base, overflow);
    if (lane == 0) emit(e >= 0 ? rc.s0 + e : -1);
  }
}

// ---- probe pass: counts / masses of elements >= each threshold ----------------
// thr[0] > thr[1] > ... > thr[np-1]; restricted to `rcut` when `restricted`.
// Cluster totals are returned in cnt_out / mass_out (all threads).
template <typename E>
__device__ void probe_pass(const RowCtx<E>& rc, Scratch& sm, Cluster& C, const float (&thr)[kProbes], int np,
                           bool with_mass, bool restricted, Cut rcut, int (&cnt_out)[kProbes],
                           FF (&mass_out)[kProbes]) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int cnt[kProbes];
  float mass[kProbes];
#pragma unroll
  for (int j = 0; j < kProbes; ++j) { cnt[j] = 0; mass[j] = 0.0f; }
  const float lowest = thr[np - 1];
  for_warp_segment<N>(rc.L, warp, lane, smem_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
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
  for_warp_segment<N>(rc.L, warp, lane, smem_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
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
  for_warp_segment<N>(rc.L, warp, lane, smem_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
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

// ---- rank-0 helpers over the gathered candidate list -------------------------

// Bitonic sort of skey[0..P) descending (P a power of two <= kCap).
__device__ void bitonic_sort_desc(unsigned long long* skey, int P) {
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = skey[i], y = skey[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) { skey[i] = y; skey[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
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
  const int i0 = 2 * threadIdx.x, i1 = i0 + 1;  // n <= kCap = 2 * kThreads
  const float w0 = (i0 < n) ? wf(i0) : 0.0f;
  const float w1 = (i1 < n) ? wf(i1) : 0.0f;
  FF total;
  const FF excl = block_excl_scan_ff(ff_add(ff(w0), w1), &total, sm);
  if (threadIdx.x == 0) {
    sm.bi[0] = INT_MAX;
    sm.bi[1] = -1;
    sm.bd[0] = ff_from_d(u * ff_to_d(total));
  }
  __syncthreads();
  int r = -1;
  if (total.hi > 0.0f) {
    const FF target = sm.bd[0];
    const FF c0 = ff_add(excl, w0), c1 = ff_add(c0, w1);
    if (w0 > 0.0f && ff_lt(target, c0) && !ff_lt(target, excl)) atomicMin(&sm.bi[0], i0);
    if (w1 > 0.0f && ff_lt(target, c1) && !ff_lt(target, c0)) atomicMin(&sm.bi[0], i1);
    if (w1 > 0.0f) atomicMax(&sm.bi[1], i1);
    else if (w0 > 0.0f) atomicMax(&sm.bi[1], i0);
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

// ---- first pass ---------------------------------------------------------------
// One sweep over the resident slice after the max is known.  It computes the
// normaliser (when needed: no filter, or top-p without top-k), the counts and
// masses of the elements above each of the first probe thresholds, and, per
// warp, the index-ordered list of elements above the lowest threshold (up to
// kWarpCap; more sets `overflow`).  One cluster exchange publishes everything.

struct PassA {
  FF z;
  int cnt[kProbes];
  FF mass[kProbes];
  int overflow;
};

// First probe thresholds: m - W*scale on the data grid, strictly descending.
template <typename E>
__device__ int first_probes(float m, float scale, float (&thr)[kProbes]) {
  const float W[kProbes] = {0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f, 8.f};
  int np = 0;
  uint32_t prev = Fmt<E>::key(m) + 1;
  const uint32_t kmin = Fmt<E>::key(-INFINITY);
  for (int j = 0; j < kProbes; ++j) {
    const float t = Fmt<E>::round_to_grid(m - W[j] * scale);
    if (!(t == t) || !(t > -INFINITY)) break;
    uint32_t k = Fmt<E>::key(t);
    if (k >= prev) k = prev - 1;
    if (k <= kmin) break;
    thr[np++] = Fmt<E>::val(k);
    prev = k;
  }
  for (int j = np; j < kProbes; ++j) thr[j] = -INFINITY;
  return np;
}

template <typename E>
__device__ void first_pass(const RowCtx<E>& rc, Scratch& sm, Cluster& C, bool need_z, bool filtered,
                           bool with_mass, const float (&thr)[kProbes], int np, PassA& out) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int cnt[kProbes];
  float mass[kProbes];
#pragma unroll
  for (int p = 0; p < kProbes; ++p) { cnt[p] = 0; mass[p] = 0.0f; }
  const float lowest = (filtered && np > 0) ? thr[np - 1] : INFINITY;
  FF running = ff(0.0f);
  int lcount = 0;  // warp-uniform list length
  int32_t* widx = sm.cand_idx + warp * kWarpCap;
  float* wval = sm.cand_val + warp * kWarpCap;
  for_warp_segment<N>(rc.L, warp, lane, smem_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
    if (need_z) {  // same arithmetic as warp_ordered_total with weights wexp
      float s = 0.0f;
#pragma unroll
      for (int j = 0; j < N; ++j) s += (j < nvalid) ? wexp(x[j], rc.m, rc.c) : 0.0f;
      running = ff_add(running, warp_sum_f(s));
    }
    int c = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) c += (j < nvalid && x[j] >= lowest) ? 1 : 0;
    if (__any_sync(FULL, c != 0)) {
#pragma unroll
      for (int j = 0; j < N; ++j) {
        if (j < nvalid && x[j] >= lowest) {
          const float w = with_mass ? wexp(x[j], rc.m, rc.c) : 0.0f;
#pragma unroll
          for (int p = 0; p < kProbes; ++p)
            if (p < np && x[j] >= thr[p]) { cnt[p] += 1; mass[p] += w; }
        }
      }
      const int incl = warp_incl_scan_i(c, lane);
      int pos = lcount + incl - c;
#pragma unroll
      for (int j = 0; j < N; ++j) {
        if (j < nvalid && x[j] >= lowest) {
          if (pos < kWarpCap) { widx[pos] = rc.s0 + e0 + j; wval[pos] = x[j]; }
          ++pos;
        }
      }
      lcount += __shfl_sync(FULL, incl, 31);
    }
  });
#pragma unroll
  for (int p = 0; p < kProbes; ++p) {
    cnt[p] = warp_sum_i(cnt[p]);
    mass[p] = warp_sum_f(mass[p]);
    if (lane == 0) { sm.pcnt[p][warp] = cnt[p]; sm.pmass[p][warp] = mass[p]; }
  }
  if (lane == 0) {
    sm.wtot[warp] = running;
    sm.wi2[warp] = min(lcount, kWarpCap);
    sm.wi[warp] = lcount > kWarpCap;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Slot& s = C.mine(sm);
    FF z = ff(0.0f);
    int of = 0;
    for (int w = 0; w < kWarps; ++w) {
      s.d[1 + w] = sm.wtot[w];
      z = ff_add(z, sm.wtot[w]);
      of |= sm.wi[w];
    }
    s.d[0] = z;
    for (int p = 0; p < kProbes; ++p) {
      int ct = 0;
      FF ms = ff(0.0f);
      for (int w = 0; w < kWarps; ++w) { ct += sm.pcnt[p][w]; ms = ff_add(ms, sm.pmass[p][w]); }
      s.i[p] = ct;
      s.d[1 + kWarps + p] = ms;
    }
    s.i[kProbes] = of;
  }
  const Slot* mir = C.exchange(sm);
  // thread 0 reduces the mirror in rank order; the whole CTA reads the result
  if (threadIdx.x == 0) {
    FF z = ff(0.0f);
    int of = 0;
    for (int r = 0; r < C.cs; ++r) { z = ff_add(z, mir[r].d[0]); of |= mir[r].i[kProbes]; }
    for (int p = 0; p < kProbes; ++p) {
      int ct = 0;
      FF ms = ff(0.0f);
      for (int r = 0; r < C.cs; ++r) { ct += mir[r].i[p]; ms = ff_add(ms, mir[r].d[1 + kWarps + p]); }
      sm.bi[p] = ct;
      sm.bd[p] = ms;
    }
    sm.bd[kProbes] = z;
    sm.bi[kProbes] = of;
  }
  __syncthreads();
  out.z = sm.bd[kProbes];
  out.overflow = sm.bi[kProbes];
  for (int p = 0; p < kProbes; ++p) { out.cnt[p] = sm.bi[p]; out.mass[p] = sm.bd[p]; }
  __syncthreads();
}

// Bracket implied by the first pass's probes (same update rule as bracket_search).
template <typename E>
__device__ Bracket bracket_from_probes(float m, const float (&thr)[kProbes], int np, const PassA& pa,
                                       bool mass_mode, int need_cnt, FF need_mass, int cnt_all,
                                       FF mass_all, int* first_true_out) {
  Bracket br;
  br.lo = Fmt<E>::key(-INFINITY);
  br.hi = Fmt<E>::key(m) + 1;
  br.cnt_lo = cnt_all;
  br.mass_lo = mass_all;
  br.cnt_hi = 0;
  br.mass_hi = ff(0.0f);
  int ft = -1;
  for (int j = 0; j < np; ++j) {  // thr[0] is the largest threshold
    const bool ok = mass_mode ? !ff_lt(pa.mass[j], need_mass) : (pa.cnt[j] >= need_cnt);
    if (ok) { ft = j; break; }
  }
  if (ft >= 0) {
    br.lo = Fmt<E>::key(thr[ft]);
    br.cnt_lo = pa.cnt[ft];
    br.mass_lo = pa.mass[ft];
    if (ft > 0) {
      br.hi = Fmt<E>::key(thr[ft - 1]);
      br.cnt_hi = pa.cnt[ft - 1];
      br.mass_hi = pa.mass[ft - 1];
    }
  } else if (np > 0) {
    br.hi = Fmt<E>::key(thr[np - 1]);
    br.cnt_hi = pa.cnt[np - 1];
    br.mass_hi = pa.mass[np - 1];
  }
  *first_true_out = ft;
  return br;
}

// After a CTA has its candidates at cand_*[0 .. n) in index order: publish n,
// and rank 0 appends the other ranks' lists after its own in one flat round of
// remote loads.  Returns the cluster count on every CTA.
__device__ int rank0_collect(Scratch& sm, Cluster& C, int n) {
  if (threadIdx.x == 0) C.mine(sm).i[0] = n;
  const Slot* mir = C.exchange(sm);
  int off[kMaxCluster + 1];
  off[0] = 0;
  for (int r = 0; r < C.cs; ++r) off[r + 1] = off[r] + mir[r].i[0];
  const int total = off[C.cs];
  if (C.rank == 0) {
    for (int j = n + threadIdx.x; j < min(total, kCap); j += kThreads) {
      int r = 1;
      while (r + 1 < C.cs && j >= off[r + 1]) ++r;
      const int i = j - off[r];
      sm.cand_idx[j] = C.cl.map_shared_rank(sm.cand_idx, r)[i];
      sm.cand_val[j] = C.cl.map_shared_rank(sm.cand_val, r)[i];
    }
  }
  __syncthreads();
  return total;
}

// Candidates from the first pass's warp lists: keep entries >= lo_val, compact
// them (warp order = index order) to the front, and collect them on rank 0.
__device__ int lists_gather(Scratch& sm, Cluster& C, float lo_val) {
  const int j0 = 2 * threadIdx.x, j1 = j0 + 1;  // 2 * kThreads == kCap slots
  const int f0 = (j0 % kWarpCap) < sm.wi2[j0 / kWarpCap] && sm.cand_val[j0] >= lo_val;
  const int f1 = (j1 % kWarpCap) < sm.wi2[j1 / kWarpCap] && sm.cand_val[j1] >= lo_val;
  const int32_t i0 = sm.cand_idx[j0], i1 = sm.cand_idx[j1];
  const float v0 = sm.cand_val[j0], v1 = sm.cand_val[j1];
  int tot;
  const int pos = block_excl_scan_i(f0 + f1, &tot, sm);
  if (f0) { sm.cand_idx[pos] = i0; sm.cand_val[pos] = v0; }
  if (f1) { sm.cand_idx[pos + f0] = i1; sm.cand_val[pos + f0] = v1; }
  __syncthreads();
  return rank0_collect(sm, C, tot);
}

// ---- exact cut ----------------------------------------------------------------


// Narrow `br` until cnt_lo <= kCap (sortable on chip) or hi == lo + 1 (one key
// value).  pred = (mass_mode ? mass >= need_mass : count >= need_cnt).  Unless
// `probed` (a first pass already probed near the max), the first probes sit at
// m - W*scale; later ones split [lo, hi) evenly in key space.
template <typename E>
__device__ Bracket bracket_search(const RowCtx<E>& rc, Scratch& sm, Cluster& C, bool mass_mode, int need_cnt,
                                  FF need_mass, float scale, bool restricted, Cut rcut, Bracket br,
                                  bool probed) {
  const float W[kProbes] = {0.5f, 1.f, 2.f, 3.f, 4.f, 6.f, 8.f, 16.f};
  for (int pass = probed ? 1 : 0; pass < kMaxPasses; ++pass) {
    if (br.cnt_lo <= kCap || br.hi - br.lo <= 1) break;
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

// Gather every element >= lo_val (and kept by rcut) into rank 0's candidate
// list, in index order; returns the cluster count on every CTA.
template <typename E>
__device__ int gather_candidates(const RowCtx<E>& rc, Scratch& sm, Cluster& C, float lo_val, bool restricted,
                                 Cut rcut) {
  auto pred = [&](float l, int x) { return l >= lo_val && (!restricted || rcut.keep(l, x)); };
  const int n = cta_ordered_compact<E>(rc, sm, pred, [&](int pos, float l, int x) {
    if (pos < kCap) { sm.cand_idx[pos] = x; sm.cand_val[pos] = l; }
  });
  return rank0_collect(sm, C, n);
}

// Rank 0 (all its threads): sort the n gathered candidates by (logit desc, index
// asc), keep the first need_k (need_k > 0), then the shortest prefix whose mass
// reaches top_p * Z (Z = the kept top-k mass, or z_for_p without top-k).
// Leaves Z_f in sm.bd[0], the cut value in sm.bd[1], the kept count in sm.bi[0],
// the cut index in sm.bi[1] and the gathered count in sm.bi[7].
template <typename E>
__device__ void rank0_sort_and_cut(const RowCtx<E>& rc, Scratch& sm, SortBuf sb, int n, int need_k, float top_p,
                                   FF z_for_p) {
  unsigned long long* skey = sb.skey;
  FF* scan = sb.scan;
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = threadIdx.x; i < P; i += kThreads)
    skey[i] = (i < n) ? ((static_cast<unsigned long long>(okey32(sm.cand_val[i])) << 32) |
                            (0xffffffffu - static_cast<uint32_t>(sm.cand_idx[i])))
                         : 0ull;
  __syncthreads();
  bitonic_sort_desc(skey, P);
  const int nk = (need_k > 0) ? min(need_k, n) : n;
  const int i0 = 2 * threadIdx.x, i1 = i0 + 1;
  const float w0 = (i0 < nk) ? wexp(skey_val(skey[i0]), rc.m, rc.c) : 0.0f;
  const float w1 = (i1 < nk) ? wexp(skey_val(skey[i1]), rc.m, rc.c) : 0.0f;
  FF total;
  const FF excl = block_excl_scan_ff(ff_add(ff(w0), w1), &total, sm);
  if (i0 < nk) scan[i0] = ff_add(excl, w0);
  if (i1 < nk) scan[i1] = ff_add(ff_add(excl, w0), w1);
  if (threadIdx.x == 0) sm.bi[2] = INT_MAX;
  __syncthreads();
  int cut = nk - 1;
  if (top_p < 1.0f) {
    const FF zk = (need_k > 0) ? total : z_for_p;
    const FF need = ff_mul(zk, top_p);
    if (i0 < nk && !ff_lt(scan[i0], need)) atomicMin(&sm.bi[2], i0);
    if (i1 < nk && !ff_lt(scan[i1], need)) atomicMin(&sm.bi[2], i1);
    __syncthreads();
    if (sm.bi[2] != INT_MAX) cut = sm.bi[2];  // otherwise rounding: keep all nk
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    sm.bd[0] = scan[cut];
    sm.bd[1] = ff(skey_val(skey[cut]));
    sm.bi[0] = cut + 1;
    sm.bi[1] = skey_idx(skey[cut]);
    sm.bi[7] = n;  // gathered count (the kept list is filtered from these)
  }
  __syncthreads();
}

// Tie cut: index of the c-th (1-based) element equal to tie_val (and kept by
// rcut), in index order across the cluster.  Same value on every CTA.
template <typename E>
__device__ int tie_locate(const RowCtx<E>& rc, Scratch& sm, Cluster& C, float tie_val, int c, bool restricted,
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
    for_warp_segment<N>(rc.L, warp, lane, smem_loader(rc), [&](float (&x)[N], int e0, int nvalid) {
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

// Count and mass of the elements kept by `cut`, cluster-wide (same on every CTA);
// with write_list and a kept set that fits kCap, the kept set is written in index
// order to lidx / lw.
template <typename E>
__device__ void kept_pass(const RowCtx<E>& rc, Scratch& sm, Cluster& C, Cut cut, bool write_list, int32_t* lidx,
                          float* lw, int* nkeep, FF* zf, int* list_len) {
  constexpr int N = Fmt<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto pred = [&](float l, int x) { return cut.keep(l, x); };
  auto wl = [&](float (&x)[N], int e0, int nvalid) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      x[j] = (j < nvalid && cut.keep(x[j], rc.s0 + e0 + j)) ? wexp(x[j], rc.m, rc.c) : 0.0f;
  };
  const FF wt = warp_ordered_total<N>(rc.L, warp, lane, smem_loader(rc), wl);
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

__device__ RowInfo decode_job(const KArgs& a, int job) {
  RowInfo ri;
  ri.job = job;
  ri.tok = -1;
  if (a.mode == kModeVerify) {
    ri.b = job / a.R;
    const int r = job % a.R;
    ri.is_target = r <= a.K;
    ri.t = ri.is_target ? r : r - (a.K + 1);
    ri.row_off = ri.is_target ? static_cast<int64_t>(ri.b) * a.tgt_seq + static_cast<int64_t>(ri.t) * a.tgt_row
                              : static_cast<int64_t>(ri.b) * a.drf_seq + static_cast<int64_t>(ri.t) * a.drf_row;
    if (ri.t < a.K) ri.tok = a.tokens[static_cast<int64_t>(ri.b) * a.K + ri.t];
  } else {
    ri.b = job / a.K;
    ri.t = job % a.K;
    ri.is_target = 0;
    ri.row_off = static_cast<int64_t>(ri.b) * a.drf_seq + static_cast<int64_t>(ri.t) * a.drf_row;
  }
  return ri;
}

__device__ void set_status(const KArgs& a, int code) {
  if (a.status) atomicCAS(a.status, 0, code);
}

// ---------------------------------------------------------------------------
// final draw from full rows in global memory (no stored kept list): the rank-0
// CTA of the sequence's last cluster alone, over [0, V).  Residual weights
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
// verify epilogue: the rank-0 CTA of the last cluster of sequence b

template <typename E>
__device__ void verify_epilogue(const KArgs& a, int b, Scratch& sm) {
  const int K = a.K, R = a.R;
  const spec_row_stat* recs = a.rows + static_cast<int64_t>(b) * R;
  int32_t* out = a.out_tokens + static_cast<int64_t>(b) * (K + 1);
  const int tid = threadIdx.x;
  // all row records in parallel: flags, then the first rejection (one test per thread)
  if (tid == 0) { sm.bi[12] = 0; sm.bi[13] = K; }
  __syncthreads();
  int myfl = 0;
  for (int r = tid; r < R; r += kThreads) myfl |= __ldcg(&recs[r].flags);
  if (myfl) atomicOr(&sm.bi[12], myfl);
  __syncthreads();
  if (sm.bi[12] == 0) {
    for (int t = tid; t < K; t += kThreads) {
      const int d = a.tokens[static_cast<int64_t>(b) * K + t];
      bool acc;
      if (a.greedy) {
        acc = (d == __ldcg(&recs[t].argmax));
      } else {
        // keep d_t with probability min(1, tgt/drf):  u * drf < tgt
        const double pt = __ldcg(&recs[t].p_tok);
        const double pd = __ldcg(&recs[K + 1 + t].p_tok);
        acc = a.u[static_cast<int64_t>(b) * (K + 1) + t] * pd < pt;
      }
      if (!acc) atomicMin(&sm.bi[13], t);  // the first rejection wins
    }
  }
  __syncthreads();
  const int fl = sm.bi[12], n = sm.bi[13];
  __syncthreads();
  if (fl) {
    for (int t = tid; t <= K; t += kThreads) out[t] = -1;
    if (tid == 0) {
      a.out_n[b] = -1;
      set_status(a, (fl & kFlagToken) ? SPEC_ERR_TOKEN_RANGE
                                      : (fl & kFlagTimeout) ? SPEC_ERR_TIMEOUT : SPEC_ERR_NONFINITE);
    }
    return;
  }
  for (int t = tid; t <= K; t += kThreads) out[t] = (t < n) ? a.tokens[static_cast<int64_t>(b) * K + t] : -1;
  int token;
  if (a.greedy) {
    token = __ldcg(&recs[n].argmax);
  } else {
    const double u = a.u[static_cast<int64_t>(b) * (K + 1) + K];
    const int rt = n, rd = K + 1 + n;
    const bool resid = n < K;
    const double zt = __ldcg(&recs[rt].zf);
    const double zd = resid ? __ldcg(&recs[rd].zf) : 1.0;
    const int lt = __ldcg(&recs[rt].list_len);
    const int ld = resid ? __ldcg(&recs[rd].list_len) : 0;
    const int64_t job_t = static_cast<int64_t>(b) * R + rt, job_d = static_cast<int64_t>(b) * R + rd;
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
// the kernel: one cluster per row

template <typename E>
__global__ void __launch_bounds__(kThreads, 3) spec_rows_kernel(const KArgs a) {
  Cluster C;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Scratch& sm = *reinterpret_cast<Scratch*>(smem_raw);
  E* sl = reinterpret_cast<E*>(smem_raw + sizeof(Scratch));
  const SortBuf sb{reinterpret_cast<unsigned long long*>(sl),
                   reinterpret_cast<FF*>(reinterpret_cast<unsigned char*>(sl) + kCap * sizeof(unsigned long long))};
  const int tid = threadIdx.x;
  const int job = static_cast<int>(blockIdx.x) / C.cs;
  const RowInfo ri = decode_job(a, job);

  RowCtx<E> rc;
  rc.g = static_cast<const E*>(ri.is_target ? a.tgt : a.drf) + ri.row_off;
  rc.sl = sl;
  rc.s0 = C.rank * a.S;
  rc.L = min(a.S, a.V - rc.s0);
  rc.c = a.c;
  rc.m = 0.0f;

  load_and_scan<E>(a, rc, sl, sm, C);
  rc.m = sm.m;
  const bool abort_ = sm.abort_ != 0;
  const bool bad = (sm.bad != 0) || abort_;
  const int argmax = sm.argmax;

  spec_row_stat* rec = a.rows + job;
  int32_t* lidx = a.list_idx + static_cast<int64_t>(job) * kCap;
  float* lw = a.list_w + static_cast<int64_t>(job) * kCap;
  const bool use_k = a.top_k > 0 && a.top_k < a.V;
  const bool use_p = a.top_p < 1.0f;

  Cut cut = cut_all();
  FF zf = ff(1.0f);
  int list_len = -1;
  bool rank0_list = false;  // kept list sits in rank 0's candidate arrays

  if (!bad && !a.greedy) {
    // first pass: normaliser (no filter, or top-p without top-k), first probes and
    // candidate lists (top-k by count, else top-p by mass)
    const bool need_z = !use_k;
    const bool filtered = use_k || use_p;
    const bool mass_mode = !use_k;
    float thr[kProbes];
    const int np = filtered ? first_probes<E>(rc.m, use_k ? 1.0f : a.temp, thr) : 0;
    PassA pa;
    first_pass<E>(rc, sm, C, need_z, filtered, filtered && mass_mode, thr, np, pa);
    if (!filtered) {
      zf = pa.z;
    } else {
      FF zk = pa.z;
      bool restricted = false, final_tie = false;
      Cut kcut = cut_all();
      if (use_k) {
        // stage A: top-k by count
        int ft;
        Bracket br = bracket_from_probes<E>(rc.m, thr, np, pa, false, a.top_k, ff(0.0f), a.V, ff(0.0f), &ft);
        int n = -1;
        if (ft >= 0 && br.cnt_lo <= kCap && !pa.overflow) {
          n = lists_gather(sm, C, Fmt<E>::val(br.lo));
        } else {
          br = bracket_search<E>(rc, sm, C, false, a.top_k, ff(0.0f), 1.0f, false, cut_all(), br, np > 0);
          if (br.cnt_lo <= kCap) n = gather_candidates<E>(rc, sm, C, Fmt<E>::val(br.lo), false, cut_all());
        }
        if (n >= 0) {
          if (C.rank == 0) rank0_sort_and_cut<E>(rc, sm, sb, n, a.top_k, use_p ? a.top_p : 1.0f, ff(0.0f));
          rank0_list = true;
        } else {
          const float tv = Fmt<E>::val(br.lo);
          const int ti = tie_locate<E>(rc, sm, C, tv, a.top_k - br.cnt_hi, false, cut_all());
          kcut = Cut{tv, ti};
          restricted = true;
          if (!use_p) { cut = kcut; final_tie = true; }
        }
      }
      if (use_p && !rank0_list) {
        // stage B: top-p by mass, within the top-k set when stage A ended in a tie cut
        Bracket br;
        int ft = -1;
        if (restricted) {
          int nk, ll;
          kept_pass<E>(rc, sm, C, kcut, false, nullptr, nullptr, &nk, &zk, &ll);
          br.lo = Fmt<E>::key(-INFINITY);
          br.hi = Fmt<E>::key(rc.m) + 1;
          br.cnt_lo = nk;
          br.mass_lo = zk;
          br.cnt_hi = 0;
          br.mass_hi = ff(0.0f);
        } else {
          br = bracket_from_probes<E>(rc.m, thr, np, pa, true, 0, ff_mul(zk, a.top_p), a.V, zk, &ft);
        }
        const FF need = ff_mul(zk, a.top_p);
        int n = -1;
        if (!restricted && ft >= 0 && br.cnt_lo <= kCap && !pa.overflow) {
          n = lists_gather(sm, C, Fmt<E>::val(br.lo));
        } else {
          br = bracket_search<E>(rc, sm, C, true, 0, need, a.temp, restricted, kcut, br, !restricted && np > 0);
          if (br.cnt_lo <= kCap) n = gather_candidates<E>(rc, sm, C, Fmt<E>::val(br.lo), restricted, kcut);
        }
        if (n >= 0) {
          if (C.rank == 0) rank0_sort_and_cut<E>(rc, sm, sb, n, 0, a.top_p, zk);
          rank0_list = true;
        } else {
          const float tv = Fmt<E>::val(br.lo);
          const float w = wexp(tv, rc.m, rc.c);
          const int ties = br.cnt_lo - br.cnt_hi;
          int c = ties;
          if (w > 0.0f) {  // smallest c with mass_hi + c * w >= need
            const FF rem = ff_sub(need, br.mass_hi);
            const float k = ceilf((rem.hi + rem.lo) / w);
            c = static_cast<int>(fminf(fmaxf(k, 1.0f), static_cast<float>(ties)));
          }
          const int ti = tie_locate<E>(rc, sm, C, tv, c, restricted, kcut);
          cut = Cut{tv, ti};
          final_tie = true;
        }
      }
      if (final_tie) {
        int nk;
        kept_pass<E>(rc, sm, C, cut, true, lidx, lw, &nk, &zf, &list_len);
      }
    }
  }

  // rank 0: the kept list = gathered candidates (index order) kept by the cut
  if (rank0_list && C.rank == 0) {
    cut = Cut{sm.bd[1].hi, sm.bi[1]};
    zf = sm.bd[0];
    list_len = sm.bi[0];
    const int gathered = sm.bi[7];
    const int i0 = 2 * tid, i1 = i0 + 1;
    const int f0 = (i0 < gathered) && cut.keep(sm.cand_val[i0], sm.cand_idx[i0]);
    const int f1 = (i1 < gathered) && cut.keep(sm.cand_val[i1], sm.cand_idx[i1]);
    int tot;
    const int pos = block_excl_scan_i(f0 + f1, &tot, sm);
    if (f0) { lidx[pos] = sm.cand_idx[i0]; lw[pos] = wexp(sm.cand_val[i0], rc.m, rc.c); }
    if (f1) { lidx[pos + f0] = sm.cand_idx[i1]; lw[pos + f0] = wexp(sm.cand_val[i1], rc.m, rc.c); }
    __syncthreads();
  }

  // sample mode: draw the token of this row
  if (a.mode == kModeSample) {
    const double u = a.greedy ? 0.0 : a.u[static_cast<int64_t>(ri.b) * a.K + ri.t];
    int32_t* outp = a.out_tokens + static_cast<int64_t>(ri.b) * a.K + ri.t;
    if (bad || a.greedy) {
      if (C.rank == 0 && tid == 0) {
        const int tok = bad ? -1 : argmax;
        *outp = tok;
        rec->token = tok;
      }
    } else if (rank0_list || list_len >= 0) {
      // kept list stored: draw over it (rank 0)
      if (!rank0_list) { __threadfence(); }
      C.cl.sync();  // lists written by every CTA are visible after the barrier
      if (C.rank == 0) {
        const int pos = list_ordered_draw(list_len, u, sm, [&](int i) { return __ldcg(&lw[i]); });
        if (tid == 0) {
          const int tok = (pos >= 0) ? __ldcg(&lidx[pos]) : -1;
          *outp = tok;
          rec->token = tok;
        }
      }
    } else {
      // no stored list: ordered draw over the resident row
      auto wk = [&](float l, int x) { return cut.keep(l, x) ? wexp(l, rc.m, rc.c) : 0.0f; };
      // unfiltered rows: the totals of the normaliser pass are still in the mirror
      if (use_k || use_p) (void)cluster_weight_total<E>(rc, sm, C, wk);
      cluster_ordered_draw<E>(rc, sm, C, u, wk, [&](int tok) {
        *outp = tok;
        rec->token = tok;
      });
    }
  }

  // row record (rank 0)
  if (C.rank == 0 && tid == 0) {
    int flags = 0;
    if (bad) flags |= abort_ ? kFlagTimeout : kFlagNonfinite;
    double p_tok = 0.0;
    if (a.mode == kModeVerify && ri.t < a.K) {
      const int d = ri.tok;
      if (d < 0 || d >= a.V) {
        flags |= kFlagToken;
      } else if (!bad && !a.greedy) {
        const float ld = Fmt<E>::at_global(rc.g, d);
        // same weight as the kept list and the normaliser use
        if (cut.keep(ld, d) && ld > -INFINITY) p_tok = static_cast<double>(wexp(ld, rc.m, rc.c)) / ff_to_d(zf);
      }
    }
    rec->zf = ff_to_d(zf);
    rec->p_tok = p_tok;
    rec->m = rc.m;
    rec->tau_val = cut.tv;
    rec->tau_idx = cut.ti;
    rec->argmax = argmax;
    rec->list_len = list_len;
    rec->flags = flags;
    if (a.mode == kModeSample && (flags & ~kFlagToken)) set_status(a, abort_ ? SPEC_ERR_TIMEOUT : SPEC_ERR_NONFINITE);
  }

  // every global write of this cluster is ordered before the sequence ticket, and
  // no CTA leaves while another may still read its shared memory
  __threadfence();
  C.cl.sync();

  if (a.mode == kModeVerify && C.rank == 0) {
    if (tid == 0) {
      // Tagged ticket: a value left by an earlier call (other tag) counts as zero,
      // so the workspace never needs re-zeroing.  Lock-free: a failed CAS means
      // another row of this sequence finished, so at most R - 1 retries.
      unsigned long long* tk = &a.tickets[ri.b];
      const unsigned long long tag = static_cast<unsigned long long>(a.tag) << 32;
      unsigned long long cur = atomicAdd(tk, 0ull), next;
      for (int tries = 0; tries <= a.R; ++tries) {
        next = ((cur & 0xffffffff00000000ull) == tag) ? cur + 1 : (tag | 1ull);
        const unsigned long long seen = atomicCAS(tk, cur, next);
        if (seen == cur) break;
        cur = seen;
      }
      sm.bi[15] = (next == (tag | static_cast<unsigned long long>(a.R)));
      __threadfence();
    }
    __syncthreads();
    if (sm.bi[15]) verify_epilogue<E>(a, ri.b, sm);
  }
}

}  // namespace

// ===========================================================================
// host side

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint32_t> g_tag{0};

uint32_t next_tag() {
  uint32_t t;
  do { t = g_tag.fetch_add(1, std::memory_order_relaxed) + 1; } while (t == 0);
  return t;
}

struct DevInfo {
  int sms = 0;
  int max_smem = 0;
  size_t smem_set[2] = {0, 0};  // dynamic smem attribute already set, per kernel
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
  int esize = 0, R = 0, CS = 1, S = 0, aligned = 0;
  int64_t nrows = 0;
  size_t smem = 0;
  size_t off_tickets = 0, off_rows = 0, off_lidx = 0, off_lw = 0, ws_bytes = 0;
};

bool finite_positive(float x) { return x > 0.0f && x < INFINITY; }

// Validates the parameters shared by both entry points and sizes the workspace.
// Cluster/slice choice needs the device; with `need_device` false only sizes are
// computed (used by the *_workspace_size queries, which then do not touch CUDA).
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
  if (pl->nrows > (int64_t(1) << 27)) return SPEC_ERR_INVALID_ARG;
  pl->off_tickets = 0;
  pl->off_rows = round_up(static_cast<size_t>(p->B) * 8, 256);
  pl->off_lidx = pl->off_rows + round_up(static_cast<size_t>(pl->nrows) * sizeof(spec_row_stat), 256);
  pl->off_lw = pl->off_lidx + round_up(static_cast<size_t>(pl->nrows) * kCap * 4, 256);
  pl->ws_bytes = pl->off_lw + round_up(static_cast<size_t>(pl->nrows) * kCap * 4, 256);
  return SPEC_OK;
}

// Slice and cluster size: ~64 KB of row per CTA (three CTAs per SM), smaller
// slices while there are fewer than two CTAs per SM, at most 8 CTAs per row.
spec_status plan_launch(const spec_params* p, const DevInfo& di, Plan* pl) {
  const int64_t row_bytes = static_cast<int64_t>(p->V) * pl->esize;
  int64_t target = 65536;
  const int64_t jobs = pl->nrows;
  while (target > 8192 && jobs * std::min<int64_t>(kMaxCluster, (row_bytes + target - 1) / target) <
                              2 * static_cast<int64_t>(di.sms))
    target /= 2;
  int cs = static_cast<int>(std::min<int64_t>(kMaxCluster, std::max<int64_t>(1, (row_bytes + target - 1) / target)));
  for (;;) {
    int64_t S = (static_cast<int64_t>(p->V) + cs - 1) / cs;
    S = (S + 63) / 64 * 64;
    const int real_cs = static_cast<int>((p->V + S - 1) / S);
    const size_t smem = sizeof(Scratch) + std::max(kSortBufBytes, round_up(static_cast<size_t>(S) * pl->esize, 128));
    if (smem <= static_cast<size_t>(di.max_smem)) {
      pl->CS = real_cs;
      pl->S = static_cast<int>(S);
      pl->smem = smem;
      return SPEC_OK;
    }
    if (cs >= kMaxCluster) return SPEC_ERR_UNSUPPORTED;
    ++cs;
  }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

spec_status launch(const spec_params* p, const Plan& pl, KArgs& a, DevInfo* di) {
  if (pl.nrows == 0) return SPEC_OK;
  const int which = (p->dtype == SPEC_F32) ? 0 : 1;
  const void* fn = which == 0 ? reinterpret_cast<const void*>(&spec_rows_kernel<float>)
                              : reinterpret_cast<const void*>(&spec_rows_kernel<uint16_t>);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (di->smem_set[which] < pl.smem) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(pl.smem)) !=
          cudaSuccess)
        return SPEC_ERR_CUDA;
      di->smem_set[which] = pl.smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.nrows * pl.CS), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = static_cast<cudaStream_t>(p->stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(pl.CS);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err;
  if (which == 0)
    err = cudaLaunchKernelEx(&cfg, spec_rows_kernel<float>, a);
  else
    err = cudaLaunchKernelEx(&cfg, spec_rows_kernel<uint16_t>, a);
  if (err != cudaSuccess) {
    (void)cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SPEC_OK;
}

void fill_common(const spec_params* p, const Plan& pl, KArgs& a) {
  char* ws = static_cast<char*>(p->workspace);
  a.tickets = reinterpret_cast<unsigned long long*>(ws + pl.off_tickets);
  a.tag = next_tag();
  a.rows = reinterpret_cast<spec_row_stat*>(ws + pl.off_rows);
  a.list_idx = reinterpret_cast<int32_t*>(ws + pl.off_lidx);
  a.list_w = reinterpret_cast<float*>(ws + pl.off_lw);
  a.B = p->B;
  a.K = p->K;
  a.V = p->V;
  a.R = pl.R;
  a.S = pl.S;
  a.greedy = p->greedy ? 1 : 0;
  a.top_k = (p->greedy || p->top_k >= p->V) ? 0 : p->top_k;
  a.top_p = p->greedy ? 1.0f : p->top_p;
  a.temp = p->greedy ? 1.0f : p->temperature;
  a.c = p->greedy ? 1.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(p->temperature));
  a.status = p->status;
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
  DevInfo* di = nullptr;
  if (!dev_info(&di)) return SPEC_ERR_CUDA;
  s = plan_launch(p, *di, &pl);
  if (s != SPEC_OK) return s;
  const int64_t es = pl.esize;
  bool al = aligned16(target_logits) && (p->target_seq_stride * es) % 16 == 0 && (p->target_row_stride * es) % 16 == 0;
  if (!p->greedy)
    al = al && aligned16(draft_logits) && (p->draft_seq_stride * es) % 16 == 0 && (p->draft_row_stride * es) % 16 == 0;
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
  DevInfo* di = nullptr;
  if (!dev_info(&di)) return SPEC_ERR_CUDA;
  s = plan_launch(p, *di, &pl);
  if (s != SPEC_OK) return s;
  const int64_t es = pl.esize;
  const bool al = aligned16(draft_logits) && (p->draft_seq_stride * es) % 16 == 0 && (p->draft_row_stride * es) % 16 == 0;
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
    case SPEC_ERR_TIMEOUT: return "bounded wait on an asynchronous copy ran out";
    case SPEC_ERR_UNSUPPORTED: return "vocabulary too large for one row per thread-block cluster";
    case SPEC_ERR_SCRATCH_LIMIT: return "request needs more scratch than spec_verify_noalloc's fixed array";
  }
  return "unknown status";
}

uint64_t spec_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

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
// up once per device, with that device current, and reused.
spec_status noalloc_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
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
  const spec_status s = noalloc_address(&scratch);
  if (s != SPEC_OK) return s;
  p.workspace = scratch;
  p.workspace_bytes = kNoAllocBytes;
  return spec_verify(target_logits, draft_logits, draft_tokens, uniforms, &p, out_tokens, out_num_accepted);
}
