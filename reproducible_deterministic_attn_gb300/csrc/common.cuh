// Shared device helpers: parameter blocks, bf16 conversion, the bounded semaphore wait.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace dash {

constexpr int kTile = 128;             // KV tile rows = Q tile rows (square task grid)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device-side bounds checks (the checked build, -DDASH_BOUNDS_CHECKS=1): every index the
// backward reads from its schedule tables (a CTA's piece range, a piece's fields, a task's
// tile indices, a dQ ordinal) is checked before it is used. A failed check records
// DASH_ERR_BOUNDS in the workspace header and stops the CTA's work; it never traps. The
// product build compiles none of it.
#ifndef DASH_BOUNDS_CHECKS
#define DASH_BOUNDS_CHECKS 0
#endif

// Workspace header (int32 words). The header occupies the first 256 bytes.
enum : int {
  WS_STATUS = 0,      // 0 = ok, DASH_ERR_SYNC_TIMEOUT on a timed-out wait, DASH_ERR_BOUNDS
  WS_BH = 1,          // (batch * H + head) of the first failing wait or check
  WS_QTILE = 2,       // dQ block of the first failing wait; the site of a failed check
  WS_EXPECT = 3,      // ordinal it waited for; the value that failed a check
  WS_SEEN = 4,        // semaphore value it last saw; the bound the value failed
};
constexpr size_t kWsHeaderBytes = 256;
constexpr int kStatusSyncTimeout = 5;
constexpr int kStatusBounds = 7;
// Sites of a failed bounds check (WS_QTILE)
enum : int { CHK_CTA_RANGE = 1, CHK_PIECE = 2, CHK_TASK = 3, CHK_ORDINAL = 4 };
// The fixed dQ order of a block runs as k = deterministic interleaved chains (1 <= k <=
// kDqChains): contribution o adds, in order, into accumulator copy o % k after
// contribution o - k, so k = 1 is one serial chain; the convert adds the copies in index
// order. Semaphore of (bh, block j, chain c): sems[(bh * n + j) * kSemStride + c] -- each
// block's semaphores sit in a 128-byte line of their own, so the polls and releasing stores
// of different blocks do not meet on one L2 line; copy c of the accumulator starts at
// dq_acc + c * B*H*S*D. Measured on GB300 (full 2x8192x16x128, shift): beyond two chains
// the extra copies cost more than the shorter waits save (the first kernel: k = 1, 2, 3, 4
// gave 588, 687, 666, 675 TFLOP/s; the current one 811, 964, 942, 939), so two is the
// maximum.
constexpr int kDqChains = 2;
constexpr int kSemStride = 32;
// A KV tile split over two CTAs hands its first half's fp32 dK/dV partial to the second
// half through the workspace, one ready flag per 32-row quarter (a read-out warp's rows).
constexpr int kSplitTiles = 256;     // most split tiles in one launch
constexpr int kSplitFlags = 4;       // flags per split tile
constexpr int kStatusSmemLayout = 4;   // reported as DASH_ERR_CUDA: unusable shared-memory base

struct FwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  int B, S, H, D;
  float scale;
  int causal;
  float scale_log2;          // scale * log2(e)
  int* status;               // optional: set to kStatusSyncTimeout when a wait runs out
  long long timeout_ns;      // bound on one pipeline wait
  int withhold_kv;           // testing hook: load no K/V tiles, so the waits for them run out
};

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* o;
  const __nv_bfloat16* dO;
  const float* lse;          // [B, H, S]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* ws_header;            // status words
  float* Dsum;               // [B, H, S] rowsum(dO * O)
  float* nlse2;              // [B, H, S] -LSE * log2(e) (the exponent offset of P in base 2)
  // Head dimension 128 only (else null): per (b*H + h, 128-row tile) a 4096-byte block of
  // 128 rows x 16 bf16 in the tensor core's no-swizzle K-major layout, holding in columns
  // 0..2 the three-term bf16 split of -LSE/scale (qx) and of -Dsum (dox); zero elsewhere.
  __nv_bfloat16* qx;
  __nv_bfloat16* dox;
  float* dq_acc;             // [B, H, S, D] fp32
  float* split_acc;          // [split tile][2][128][D] fp32: first half's dK, dV partials
  int* split_flags;          // [split tile][kSplitFlags]: 1 once that quarter is stored
  int* sems;                 // [B, H, n, kSemStride]: per 128-row dQ block, one per chain
  int num_sems;               // B * H * n * kSemStride
  int chains;                 // interleaved dQ chains, 1..kDqChains (deterministic mode)
  const int32_t* cta_off;    // dealing: CTA c runs pieces [cta_off[c], cta_off[c + 1])
  const int32_t* pieces;     // dealing: 4 words per piece: head, first task, end task,
                             // (split tile << 2) | part (0 whole, 1 / 2 first / second half)
  const int32_t* tasks;      // schedule: (kv << 16) | q
  const int32_t* ord;        // schedule: ordinals, ord[bh * ord_stride + i * n + j]
  long long ord_stride;      // n * n when every head has its own order, else 0
  const int32_t* cnt;        // schedule: contributors per dQ block
  int B, S, H, D;
  int n;                     // tiles per head
  float scale;
  float scale_log2;          // scale * log2(e)
  int causal;
  int deterministic;
  long long timeout_ns;      // bound on one semaphore wait
  int ordinal_skew;          // testing hook: added to every awaited ordinal
  unsigned long long* trace; // optional per-CTA wait-cycle counters (null: off)
  // read by the bounds checks only: the tables' lengths and the tile bound (n, or less
  // under the testing hook that narrows the checks)
  int num_pieces, num_tasks, check_n;
};

// Wait sites of the optional trace (cycles spent waiting, per CTA).
enum : int {
  TR_PROD_STAGE_EMPTY = 0, TR_PROD_KV_EMPTY, TR_MMA_KV_FULL, TR_MMA_STAGE_FULL, TR_MMA_S_EMPTY,
  TR_MMA_DP_EMPTY, TR_MMA_P_FULL, TR_MMA_ACC_EMPTY, TR_MMA_DS_FULL, TR_MMA_DQ_EMPTY,
  TR_SG_S_FULL, TR_SG_P_EMPTY, TR_SG_DP_FULL, TR_SG_DS_EMPTY, TR_DQ_FULL, TR_DQ_SEM,
  TR_DQ_REDUCE, TR_DQ_ACC_FULL, TR_DQ_STAGE, TR_TOTAL, TR_ISSUE_S, TR_ISSUE_DP, TR_ISSUE_DV,
  TR_ISSUE_DKDQ, TR_X0, TR_X1, TR_X2, TR_X3, TR_X4, TR_X5, TR_X6, TR_X7, TR_SITES = 32
};

__device__ __forceinline__ long long global_timer_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_add_gpu(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

#if DASH_BOUNDS_CHECKS
// Records the first failed bounds check of a launch (any thread; the first one wins).
__device__ __noinline__ void report_bounds(int* ws, int site, int bh, int value, int bound) {
  if (atomicCAS(ws + WS_STATUS, 0, kStatusBounds) == 0) {
    ws[WS_BH] = bh;
    ws[WS_QTILE] = site;
    ws[WS_EXPECT] = value;
    ws[WS_SEEN] = bound;
    __threadfence();
  }
}
#endif

// Spin (one thread) until *sem == target. Gives up when another CTA has already
// reported a failure, or after timeout_ns, recording the first failure in the
// workspace header. Returns true when it is this CTA's turn.
__device__ __noinline__ bool wait_turn(const int* sem, int target, int* ws, long long timeout_ns,
                                       int bh, int qtile) {
  int seen = ld_acquire_gpu(sem);
  if (seen == target) return true;
  const long long t0 = global_timer_ns();
  // The hand-off latency adds to every step of the serial order, so the semaphore is
  // polled back to back (one L2 round trip per poll); the failure flag and the timer are
  // looked at every 32nd poll. The iteration cap is a second bound, independent of the
  // timer (a poll takes well over 16 ns).
  const long long max_iter = timeout_ns / 16 + (1ll << 20);
  for (long long it = 1; it <= max_iter; ++it) {
    seen = ld_acquire_gpu(sem);
    if (seen == target) return true;
    if ((it & 31) == 0) {
      if (ld_relaxed_gpu(ws + WS_STATUS) != 0) return false;
      if (global_timer_ns() - t0 > timeout_ns) break;
    }
  }
  if (atomicCAS(ws + WS_STATUS, 0, kStatusSyncTimeout) == 0) {
    ws[WS_BH] = bh;
    ws[WS_QTILE] = qtile;
    ws[WS_EXPECT] = target;
    ws[WS_SEEN] = seen;
    __threadfence();
  }
  return false;
}

// Spin (one thread) until *sem >= target (a counter that only grows). Gives up when another CTA has already
// reported a failure, or after timeout_ns, recording the first failure in the
// workspace header. Returns true when it is this CTA's turn.
__device__ __noinline__ bool wait_at_least(const int* sem, int target, int* ws, long long timeout_ns,
                                       int bh, int qtile) {
  int seen = ld_acquire_gpu(sem);
  if (seen >= target) return true;
  const long long t0 = global_timer_ns();
  // The hand-off latency adds to every step of the serial order, so the semaphore is
  // polled back to back (one L2 round trip per poll); the failure flag and the timer are
  // looked at every 32nd poll. The iteration cap is a second bound, independent of the
  // timer (a poll takes well over 16 ns).
  const long long max_iter = timeout_ns / 16 + (1ll << 20);
  for (long long it = 1; it <= max_iter; ++it) {
    seen = ld_acquire_gpu(sem);
    if (seen >= target) return true;
    if ((it & 31) == 0) {
      if (ld_relaxed_gpu(ws + WS_STATUS) != 0) return false;
      if (global_timer_ns() - t0 > timeout_ns) break;
    }
  }
  if (atomicCAS(ws + WS_STATUS, 0, kStatusSyncTimeout) == 0) {
    ws[WS_BH] = bh;
    ws[WS_QTILE] = qtile;
    ws[WS_EXPECT] = target;
    ws[WS_SEEN] = seen;
    __threadfence();
  }
  return false;
}

}  // namespace dash
