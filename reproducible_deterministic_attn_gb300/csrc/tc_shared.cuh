// Pieces shared by the tcgen05 kernels (backward main kernel, forward, split-K GEMM):
// launch shape and TMEM size, the TMA tensor maps, the 128-byte swizzle of a bf16 tile, the
// persistent grid's task walk and the optional wait-cycle trace helpers.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace dash {
namespace tc {

constexpr int kThreads = 512;
constexpr int kTmemCols = 512;

struct TmaMaps {
  CUtensorMap q, k, v, dO;   // 3D bf16 [B*S][H][D], boxes {64, 1, rows}
};

// byte offset of (row, 8-column chunk) in a bf16 tile of 128-byte rows, 64-column blocks
// of `rows` rows each, 128-byte swizzle
__device__ __forceinline__ uint32_t sw_chunk(int row, int chunk, int rows) {
  return (uint32_t)((chunk >> 3) * rows * 128 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Iterates this CTA's (piece, task) sequence; every role walks the same sequence. A piece
// is a run of one head's chain that covers whole KV tiles, so a new piece always starts a
// new tile. The task table is read two entries ahead so its load latency hides behind
// the work.
struct Walk {
  const BwdParams& p;
  int k, k_end, t, t_end, bh, i, j;
  int tag;                    // this piece's (split tile << 2) | part
  int32_t prev_tk, cur_tk, nxt_tk, nxt2_tk;
  bool first_of_tile, last_of_tile;
#if DASH_BOUNDS_CHECKS
  volatile int* abort_flag;   // the CTA's: raised on a failed check so no role waits on
                              // work the others will not do
#endif
  __device__ Walk(const BwdParams& pp, volatile int* cta_abort)
      : p(pp), k(__ldg(pp.cta_off + blockIdx.x) - 1), k_end(__ldg(pp.cta_off + blockIdx.x + 1)),
        t(0), t_end(0) {
#if DASH_BOUNDS_CHECKS
    abort_flag = cta_abort;
    if (k < -1 || k_end < k + 1 || k_end > p.num_pieces) {
      report_bounds(p.ws_header, CHK_CTA_RANGE, (int)blockIdx.x, k_end, p.num_pieces);
      *abort_flag = 1;
      k_end = k + 1;   // no pieces: next() returns false at once
    }
#else
    (void)cta_abort;
#endif
  }
  __device__ __forceinline__ int32_t task_at(int k) const {
    return k < t_end ? __ldg(p.tasks + k) : -1;
  }
#if DASH_BOUNDS_CHECKS
  // A task read from the table (index < t_end) must name two tiles below the bound.
  __device__ bool task_ok(int idx, int32_t tk) const {
    return idx >= t_end || (tk >= 0 && (tk >> 16) < p.check_n && (tk & 0xffff) < p.check_n);
  }
  __device__ bool fail(int site, int value, int bound) {
    report_bounds(p.ws_header, site, bh, value, bound);
    *abort_flag = 1;
    k_end = k;
    t = t_end = 0;
    return false;
  }
#endif
  __device__ bool next() {
    ++t;
    if (t >= t_end) {
      do {
        if (++k >= k_end) return false;
        const int4 pc = __ldg(reinterpret_cast<const int4*>(p.pieces) + k);
        bh = pc.x;
        t = pc.y;
        t_end = pc.z;
        tag = pc.w;
#if DASH_BOUNDS_CHECKS
        const int part = tag & 3, split = tag >> 2;
        if (bh < 0 || bh >= p.B * p.H) return fail(CHK_PIECE, bh, p.B * p.H);
        if (t < 0 || t > t_end || t_end > p.num_tasks) return fail(CHK_PIECE, t_end, p.num_tasks);
        if (part > 2 || (part != 0 && (split < 0 || split >= kSplitTiles)))
          return fail(CHK_PIECE, tag, kSplitTiles);
#endif
      } while (t >= t_end);
      prev_tk = -1;
      cur_tk = task_at(t);
      nxt_tk = task_at(t + 1);
#if DASH_BOUNDS_CHECKS
      if (!task_ok(t, cur_tk)) return fail(CHK_TASK, cur_tk, p.check_n);
      if (!task_ok(t + 1, nxt_tk)) return fail(CHK_TASK, nxt_tk, p.check_n);
#endif
    } else {
      prev_tk = cur_tk;
      cur_tk = nxt_tk;
      nxt_tk = nxt2_tk;
    }
    nxt2_tk = task_at(t + 2);
#if DASH_BOUNDS_CHECKS
    if (!task_ok(t + 2, nxt2_tk)) return fail(CHK_TASK, nxt2_tk, p.check_n);
#endif
    i = cur_tk >> 16;
    j = cur_tk & 0xffff;
    first_of_tile = prev_tk < 0 || (prev_tk >> 16) != i;
    last_of_tile = nxt_tk < 0 || (nxt_tk >> 16) != i;
    return true;
  }
};

// Optional wait-cycle trace: one writer per site, counters in shared memory, copied to
// p.trace[cta * TR_SITES + site] at exit.
struct Trace {
  unsigned long long* c;   // shared counters, null when tracing is off
  __device__ __forceinline__ long long t0() const { return c ? clock64() : 0; }
  __device__ __forceinline__ void add(int site, long long start) const {
    if (c) c[site] += (unsigned long long)(clock64() - start);
  }
};

// Gap-free variant of the trace for one thread: every cycle between two marks is charged
// to the site of the later mark, so the sites add up to the thread's whole loop time. The
// counters live in registers (site indices are compile-time constants) and are added to the
// shared counters once, by flush().
template <int N>
struct SegTrace {
  unsigned long long* c;   // shared counters, null when tracing is off
  uint32_t acc[N];
  long long last;
  __device__ __forceinline__ SegTrace(unsigned long long* counters) : c(counters), last(0) {
#pragma unroll
    for (int k = 0; k < N; ++k) acc[k] = 0;
    if (c) last = clock64();
  }
  // charge the cycles since the previous mark to slot k
  __device__ __forceinline__ void mark(int k) {
    if (c) {
      const long long now = clock64();
      acc[k] += (uint32_t)(now - last);
      last = now;
    }
  }
  __device__ __forceinline__ void flush(const int (&sites)[N]) const {
    if (c) {
#pragma unroll
      for (int k = 0; k < N; ++k) atomicAdd(c + sites[k], (unsigned long long)acc[k]);
    }
  }
};

// Gap-free trace kept in the shared counters directly (no registers beyond the last
// timestamp): mark(site) adds the cycles since the previous mark to the site.
struct SegTraceShared {
  unsigned long long* c;   // shared counters, null when tracing is off
  long long last;
  __device__ __forceinline__ SegTraceShared(unsigned long long* counters) : c(counters), last(0) {
    if (c) last = clock64();
  }
  __device__ __forceinline__ void mark(int site) {
    if (c) {
      const long long now = clock64();
      atomicAdd(c + site, (unsigned long long)(now - last));
      last = now;
    }
  }
};

}  // namespace tc
}  // namespace dash
