// Backward main kernel on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), head
// dimension 64 (head dimension 128 runs the kernel of kernels_tc128.cuh, which reuses the
// walk, trace and TMA-map definitions here).
//
// One persistent CTA per SM. A unit is one schedule chain (slot) of one (batch, head);
// CTA c runs units c, c + grid, ... Each schedule task (KV_i, Q_j) covers a 128 x 128
// tile of the score matrix; KV_i's K and V tiles stay in shared memory for all its
// tasks and its dK/dV accumulate in TMEM (DASH keeps a KV tile's dK/dV on one SM).
//
// Per task (BR = 128 query rows, one sub-tile; the walk supports SUB > 1 sub-tiles):
//   S^T  = K Q^T          (M = 128 kv, N = BR, K = D)      -> TMEM
//   dP^T = V dO^T         (M = 128 kv, N = BR, K = D)      -> TMEM
//   P^T  = exp2(S^T * scale*log2e - LSE*log2e)            softmax-gradient warps -> smem bf16
//   dS^T = P^T * (dP^T - Dsum)                            softmax-gradient warps -> smem bf16
//   dV  += P^T dO         (M = 128 kv, N = D, K = BR)
//   dK  += dS^T Q         (M = 128 kv, N = D, K = BR)
//   dQ   = dS K           (M = 128 q, N = 64, K = 128 kv)   TMEM lanes = q rows
//   then the dQ partial is staged in smem and added into the fp32 dQ accumulator with a
//   TMA bulk reduce-add: deterministic mode waits on the block's L2 semaphore for its
//   ordinal first and releases ordinal + 1 after the add has completed (the pages' fixed
//   serial reduction order); non-deterministic mode adds as soon as it can.
//
// Warp roles (512 threads): warp 0 = TMA producer, warp 1 = S^T/dP^T MMA issuer, warp 3 =
// dV/dK/dQ MMA issuer, warp 2 = dQ reducer (semaphore waits, TMA reduce-adds, releases),
// warps 4..11 = softmax-gradient (two warpgroups, each half of the BR columns), warps
// 12..15 = dQ read-out into the staging buffer and the dK/dV epilogue. TMEM: 512 columns.
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace dash {
namespace tc {

template <int D>
struct Cfg;

template <>
struct Cfg<64> {
  static constexpr int BR = 128;  // query rows per sub-tile
  static constexpr int SUB = 1;   // sub-tiles per 128-row schedule task
  static constexpr int STAGES = 2;  // Q/dO pipeline depth
  static constexpr int T_S = 0, T_DP = 128, T_DV = 256, T_DK = 320, T_DQ = 384;
};


constexpr int kThreads = 512;
constexpr int kMaxStages = 3;
constexpr int kTmemCols = 512;

// Shared-memory carve-up (byte offsets from a 1024-aligned base). A stage holds one
// sub-tile's Q and dO (TMA destinations, 1024-aligned); the stages' LSE and Dsum rows sit
// together after the dQ staging buffer.
template <int D>
struct Smem {
  static constexpr int BR = Cfg<D>::BR;
  static constexpr int STAGES = Cfg<D>::STAGES;
  static constexpr int KV_BYTES = kTile * D * 2;             // one of K or V
  static constexpr int QT_BYTES = BR * D * 2;                // one of Q or dO (per stage)
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV_BYTES;
  static constexpr int STAGE_OFF = V_OFF + KV_BYTES;
  static constexpr int STAGE_BYTES = 2 * QT_BYTES;
  static constexpr int Q_IN_STAGE = 0;
  static constexpr int DO_IN_STAGE = QT_BYTES;
  static constexpr int P_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
  static constexpr int PT_BYTES = kTile * BR * 2;            // P^T or dS^T tile
  static constexpr int DS_OFF = P_OFF + PT_BYTES;
  static constexpr int STG_OFF = DS_OFF + PT_BYTES;          // dQ staging (fp32)
  static constexpr int STG_BYTES = BR * D * 4;
  static constexpr int LD_OFF = STG_OFF + STG_BYTES;         // per stage: LSE[BR], Dsum[BR]
  static constexpr int LD_STAGE_BYTES = 2 * BR * 4;
  static constexpr int BAR_OFF = LD_OFF + STAGES * LD_STAGE_BYTES;
  static constexpr int TRACE_OFF = BAR_OFF + 256;
  static constexpr int TOTAL = TRACE_OFF + 8 * TR_SITES;     // barriers, flags, trace
  static constexpr int ALLOC = TOTAL + 1024;                 // slack for 1024 alignment
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Barrier indices.
enum {
  B_KV_FULL = 0, B_KV_EMPTY, B_S_FULL, B_S_EMPTY, B_DP_FULL, B_DP_EMPTY, B_P_EMPTY,
  B_DS_FULL, B_DS_EMPTY, B_DQ_FULL, B_ACC_FULL, B_ACC_EMPTY, B_DRAIN,
  B_STG_FULL, B_STG_EMPTY, B_DRAIN2,
  B_STAGE_FULL,                     // + stage
  B_STAGE_EMPTY = B_STAGE_FULL + kMaxStages,
  B_COUNT = B_STAGE_EMPTY + kMaxStages
};

struct TmaMaps {
  CUtensorMap q, k, v, dO;   // 3D bf16 [B*S][H][D], boxes {64, 1, rows}
  CUtensorMap acc;           // 2D fp32 [B*H*S][D], box {32, BR}
};

// byte offset of (row, 8-column chunk) in a bf16 tile of 128-byte rows, 64-column blocks
// of `rows` rows each, 128-byte swizzle
__device__ __forceinline__ uint32_t sw_chunk(int row, int chunk, int rows) {
  return (uint32_t)((chunk >> 3) * rows * 128 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Iterates this CTA's (unit, task) sequence; every role walks the same sequence. The
// task table is read two entries ahead so its load latency hides behind the work.
struct Walk {
  const BwdParams& p;
  int u, t, t_end, bh, i, j;
  int32_t prev_tk, cur_tk, nxt_tk, nxt2_tk;
  bool first_of_tile, last_of_tile;
  __device__ Walk(const BwdParams& pp)
      : p(pp), u((int)blockIdx.x - (int)gridDim.x), t(0), t_end(0) {}
  __device__ __forceinline__ int32_t task_at(int k) const {
    return k < t_end ? __ldg(p.tasks + k) : -1;
  }
  __device__ bool next() {
    ++t;
    if (t >= t_end) {
      do {
        u += gridDim.x;
        if (u >= p.num_units) return false;
        const int slot = u % p.num_slots;
        bh = u / p.num_slots;
        t = __ldg(p.slot_off + slot);
        t_end = __ldg(p.slot_off + slot + 1);
      } while (t >= t_end);
      prev_tk = -1;
      cur_tk = task_at(t);
      nxt_tk = task_at(t + 1);
    } else {
      prev_tk = cur_tk;
      cur_tk = nxt_tk;
      nxt_tk = nxt2_tk;
    }
    nxt2_tk = task_at(t + 2);
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

// One step of the flat sub-tile sequence (SUB sub-tiles per schedule task).
struct Sub {
  int i, j, hs, it, tile;
  bool first, last;   // first / last sub-tile of its KV tile
};

template <int SUB>
struct SubWalk {
  Walk w;
  int hs = SUB - 1, it = -1, tile = -1;
  __device__ SubWalk(const BwdParams& p) : w(p) {}
  __device__ bool next(Sub& s) {
    if (hs + 1 < SUB) {
      ++hs;
    } else {
      if (!w.next()) return false;
      hs = 0;
      if (w.first_of_tile) ++tile;
    }
    ++it;
    s.i = w.i;
    s.j = w.j;
    s.hs = hs;
    s.it = it;
    s.tile = tile;
    s.first = w.first_of_tile && hs == 0;
    s.last = w.last_of_tile && hs == SUB - 1;
    return true;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ TmaMaps maps) {
  using C = Cfg<D>;
  using L = Smem<D>;
  constexpr int BR = C::BR, SUB = C::SUB, kStages = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR_OFF);
  uint32_t* tmem_slot = (uint32_t*)(sm + L::BAR_OFF + 8 * B_COUNT);
  volatile int* abort_flag = (volatile int*)(sm + L::BAR_OFF + 8 * B_COUNT + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bars + B_KV_FULL, 1);
    ptx::mbar_init(bars + B_KV_EMPTY, 1);
    ptx::mbar_init(bars + B_S_FULL, 1);
    ptx::mbar_init(bars + B_S_EMPTY, 8);
    ptx::mbar_init(bars + B_DP_FULL, 1);
    ptx::mbar_init(bars + B_DP_EMPTY, 8);
    ptx::mbar_init(bars + B_P_EMPTY, 1);
    ptx::mbar_init(bars + B_DS_FULL, 8 + 4);   // 8 softmax-gradient warps + 4 dQ warps
    ptx::mbar_init(bars + B_DS_EMPTY, 1);
    ptx::mbar_init(bars + B_DQ_FULL, 1);
    ptx::mbar_init(bars + B_ACC_FULL, 1);
    ptx::mbar_init(bars + B_ACC_EMPTY, 4);
    ptx::mbar_init(bars + B_DRAIN, 1);
    ptx::mbar_init(bars + B_STG_FULL, 4);
    ptx::mbar_init(bars + B_STG_EMPTY, 1);
    ptx::mbar_init(bars + B_DRAIN2, 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bars + B_STAGE_FULL + s, 1);
      ptx::mbar_init(bars + B_STAGE_EMPTY + s, 1 + 8);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  unsigned long long* trace_s = (unsigned long long*)(sm + L::TRACE_OFF);
  if (threadIdx.x < TR_SITES) trace_s[threadIdx.x] = 0;
  const long long t_start = clock64();
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const size_t rs = (size_t)p.H * D;   // BSHD row stride (elements)
  const Trace tr{p.trace ? trace_s : nullptr};
  const Trace tr_none{nullptr};

  if (warp == 0) {
    // ===================================== TMA producer =====================================
    if (lane == 0) {
      SubWalk<SUB> sw(p);
      Sub x;
      int it = 0, tl = 0;
      while (sw.next(x)) {
        const int bh = sw.w.bh, b = bh / p.H, h = bh % p.H;
        const int s = it % kStages;
        const int q0 = x.j * kTile + x.hs * BR;
        // Q, dO, LSE and Dsum of this sub-tile into stage s
        long long t0 = tr.t0();
        if (it >= kStages &&
            !ptx::mbar_wait(bars + B_STAGE_EMPTY + s, ((it / kStages) - 1) & 1, abort_flag, tmo))
          break;
        tr.add(TR_PROD_STAGE_EMPTY, t0);
        uint8_t* st = sm + L::STAGE_OFF + s * L::STAGE_BYTES;
        ptx::mbar_expect_tx(bars + B_STAGE_FULL + s, 2 * L::QT_BYTES + L::LD_STAGE_BYTES);
        for (int cb = 0; cb < D / 64; ++cb) {
          ptx::tma_load_3d(st + L::Q_IN_STAGE + cb * BR * 128, &maps.q, cb * 64, h, b * p.S + q0,
                           bars + B_STAGE_FULL + s);
          ptx::tma_load_3d(st + L::DO_IN_STAGE + cb * BR * 128, &maps.dO, cb * 64, h, b * p.S + q0,
                           bars + B_STAGE_FULL + s);
        }
        uint8_t* ld = sm + L::LD_OFF + s * L::LD_STAGE_BYTES;
        ptx::bulk_load(ld, p.lse + (size_t)bh * p.S + q0, BR * 4, bars + B_STAGE_FULL + s);
        ptx::bulk_load(ld + BR * 4, p.Dsum + (size_t)bh * p.S + q0, BR * 4,
                       bars + B_STAGE_FULL + s);
        ++it;
        // a new KV tile: K and V once the previous tile's MMAs are done with the buffer
        if (x.first) {
          t0 = tr.t0();
          if (tl > 0 && !ptx::mbar_wait(bars + B_KV_EMPTY, (tl - 1) & 1, abort_flag, tmo)) break;
          tr.add(TR_PROD_KV_EMPTY, t0);
          ptx::mbar_expect_tx(bars + B_KV_FULL, 2 * L::KV_BYTES);
          for (int cb = 0; cb < D / 64; ++cb) {
            ptx::tma_load_3d(sm + L::K_OFF + cb * kTile * 128, &maps.k, cb * 64, h,
                             b * p.S + x.i * kTile, bars + B_KV_FULL);
            ptx::tma_load_3d(sm + L::V_OFF + cb * kTile * 128, &maps.v, cb * 64, h,
                             b * p.S + x.i * kTile, bars + B_KV_FULL);
          }
          ++tl;
        }
      }
      // drain: every issued load has landed before the CTA may exit
      for (int k = (it > kStages ? it - kStages : 0); k < it; ++k)
        ptx::mbar_drain(bars + B_STAGE_FULL + k % kStages, (k / kStages) & 1, 100000000ll);
      if (tl > 0) ptx::mbar_drain(bars + B_KV_FULL, (tl - 1) & 1, 100000000ll);
    }
  } else if (warp == 1 || warp == 3) {
    // ===================================== MMA issuers ======================================
    // Two issuing threads keep the tensor pipe fed while either one waits on a barrier:
    // warp 1 issues S^T and dP^T, warp 3 issues dV, dK and the dQ partial. Their TMEM
    // regions are disjoint; the softmax-gradient hand-offs order them.
    if (lane == 0) {
      // Descriptor low words of every operand buffer; each K step adds a compile-time
      // offset (in 16-byte units) to them.
      const uint32_t sK = ptx::smem_u32(sm + L::K_OFF), sV = ptx::smem_u32(sm + L::V_OFF);
      const uint32_t sP = ptx::smem_u32(sm + L::P_OFF), sdS = ptx::smem_u32(sm + L::DS_OFF);
      const uint32_t dK_k = ptx::sdesc_lo(sK, 16);                  // K, K-major
      const uint32_t dK_mn = ptx::sdesc_lo(sK, kTile * 128);        // K, MN-major
      const uint32_t dV_k = ptx::sdesc_lo(sV, 16);
      const uint32_t dP_k = ptx::sdesc_lo(sP, 16);
      const uint32_t dS_k = ptx::sdesc_lo(sdS, 16);
      const uint32_t dS_mn = ptx::sdesc_lo(sdS, kTile * 128);
      const uint32_t st0 = ptx::smem_u32(sm + L::STAGE_OFF);
      constexpr uint32_t ID_S = ptx::idesc_bf16(128, BR, 0, 0);     // S^T, dP^T
      constexpr uint32_t ID_ACC = ptx::idesc_bf16(128, D, 0, 1);    // dV, dK
      constexpr uint32_t ID_DQ = ptx::idesc_bf16(128, 64, 1, 1);    // dQ (D=64) / dQ^T (D=128)
      // K-major step ks of a [rows][D] tile in 64-column blocks: 32 bytes per step inside a
      // 128-byte row, a new block every 4 steps; MN-major step ks: 16 rows of 128 bytes.
      auto kstep = [](int ks, int rows) -> uint32_t {
        return ((ks >> 2) * rows * 128 + (ks & 3) * 32) >> 4;
      };
      constexpr uint32_t MN_STEP = 2048 >> 4;
      auto stage_lo = [&](const Sub& x, int off, uint32_t lbo) {
        return ptx::sdesc_lo(st0 + (x.it % kStages) * L::STAGE_BYTES + off, lbo);
      };
      SubWalk<SUB> sw(p);
      Sub x;
      bool ok = true;
      if (warp == 1) {
        while (ok && sw.next(x)) {
          long long t0 = tr.t0();
          if (x.first && !(ok = ptx::mbar_wait(bars + B_KV_FULL, x.tile & 1, abort_flag, tmo))) break;
          tr.add(TR_MMA_KV_FULL, t0);
          t0 = tr.t0();
          ok = ptx::mbar_wait(bars + B_STAGE_FULL + x.it % kStages, (x.it / kStages) & 1,
                              abort_flag, tmo);
          tr.add(TR_MMA_STAGE_FULL, t0);
          t0 = tr.t0();
          if (ok && x.it > 0) ok = ptx::mbar_wait(bars + B_S_EMPTY, (x.it - 1) & 1, abort_flag, tmo);
          tr.add(TR_MMA_S_EMPTY, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t dQ_k = stage_lo(x, L::Q_IN_STAGE, 16);
          const uint32_t ddO_k = stage_lo(x, L::DO_IN_STAGE, 16);
          // S^T = K Q^T: K-major A (128 kv rows), K-major B (BR rows)
          t0 = tr.t0();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            ptx::mma_lo(tmem + C::T_S, dK_k + kstep(ks, kTile), dQ_k + kstep(ks, BR), ID_S, ks > 0);
          ptx::mma_commit(bars + B_S_FULL);
          tr.add(TR_ISSUE_S, t0);
          t0 = tr.t0();
          if (x.it > 0) ok = ptx::mbar_wait(bars + B_DP_EMPTY, (x.it - 1) & 1, abort_flag, tmo);
          tr.add(TR_MMA_DP_EMPTY, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          // dP^T = V dO^T
          t0 = tr.t0();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            ptx::mma_lo(tmem + C::T_DP, dV_k + kstep(ks, kTile), ddO_k + kstep(ks, BR), ID_S, ks > 0);
          ptx::mma_commit(bars + B_DP_FULL);
          tr.add(TR_ISSUE_DP, t0);
        }
      } else {
        while (ok && sw.next(x)) {
          const uint32_t dQ_mn = stage_lo(x, L::Q_IN_STAGE, BR * 128);
          const uint32_t ddO_mn = stage_lo(x, L::DO_IN_STAGE, BR * 128);
          // One check covers the whole group (the tensor pipe queues about one MMA, so every
          // check on this thread idles it): a completed dS(t) phase means every
          // softmax-gradient warp has also published P(t) (P is written first), and the dQ
          // warps' arrivals on the same barrier mean dQ(t-1) has left TMEM.
          long long t0 = tr.t0();
          ok = ptx::mbar_wait(bars + B_DS_FULL, x.it & 1, abort_flag, tmo);
          tr.add(TR_MMA_DS_FULL, t0);
          t0 = tr.t0();
          // The first sub-tile of a KV tile overwrites the dV/dK accumulators, which the
          // previous tile's epilogue must have read out.
          if (ok && x.first && x.tile > 0)
            ok = ptx::mbar_wait(bars + B_ACC_EMPTY, (x.tile - 1) & 1, abort_flag, tmo);
          tr.add(TR_MMA_ACC_EMPTY, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t acc0 = x.first ? 0u : 1u;
          // dV += P^T dO: A = P^T (K-major, 128 kv rows x BR), B = dO (MN-major over D)
          t0 = tr.t0();
#pragma unroll
          for (int ks = 0; ks < BR / 16; ++ks)
            ptx::mma_lo(tmem + C::T_DV, dP_k + kstep(ks, kTile), ddO_mn + ks * MN_STEP, ID_ACC,
                        ks > 0 ? 1u : acc0);
          ptx::mma_commit(bars + B_P_EMPTY);
          tr.add(TR_ISSUE_DV, t0);
          // dK += dS^T Q, then the dQ partial over the 128 kv rows
          t0 = tr.t0();
#pragma unroll
          for (int ks = 0; ks < BR / 16; ++ks)
            ptx::mma_lo(tmem + C::T_DK, dS_k + kstep(ks, kTile), dQ_mn + ks * MN_STEP, ID_ACC,
                        ks > 0 ? 1u : acc0);
          // dQ = dS K: A = dS (MN-major view of the dS^T tile), B = K (MN-major, 64 d)
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            ptx::mma_lo(tmem + C::T_DQ, dS_mn + ks * MN_STEP, dK_mn + ks * MN_STEP, ID_DQ, ks > 0);
          ptx::mma_commit(bars + B_DS_EMPTY);
          ptx::mma_commit(bars + B_DQ_FULL);
          tr.add(TR_ISSUE_DKDQ, t0);
          // the stage's Q/dO were last read by dK/dV here; the S^T/dP^T reads of this stage
          // finished before the softmax-gradient warps released P and dS
          ptx::mma_commit(bars + B_STAGE_EMPTY + x.it % kStages);
          if (x.last) {
            ptx::mma_commit(bars + B_ACC_FULL);
            ptx::mma_commit(bars + B_KV_EMPTY);
          }
        }
      }
      // drain: no MMA may be in flight when TMEM is released
      uint64_t* drain = bars + (warp == 1 ? B_DRAIN : B_DRAIN2);
      ptx::mma_commit(drain);
      ptx::mbar_drain(drain, 0, 1000000000ll);
    }
  } else if (warp >= 4 && warp < 12) {
    // =============================== softmax-gradient warps =================================
    constexpr int NC = BR / 2;                 // columns per thread
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;         // kv row within the tile
    const int col0 = half * NC;
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const uint32_t sP = ptx::smem_u32(sm + L::P_OFF), sdS = ptx::smem_u32(sm + L::DS_OFF);
    const Trace& trs = (warp == 4 && lane == 0) ? tr : tr_none;
    Walk w(p);
    int it = 0;
    bool ok = true;
    while (ok && w.next()) {
      for (int hs = 0; hs < SUB && ok; ++hs, ++it) {
        const int s = it % kStages;
        const int q0 = w.j * kTile + hs * BR;
        const float* lse_s = (const float*)(sm + L::LD_OFF + s * L::LD_STAGE_BYTES);
        const float* dsum_s = lse_s + BR;
        const bool diag = p.causal && (w.i == w.j);
        const int kv_g = w.i * kTile + r;
        long long t0 = trs.t0();
        ok = ptx::warp_wait(bars + B_STAGE_FULL + s, (it / kStages) & 1, abort_flag, tmo);
        if (ok) ok = ptx::warp_wait(bars + B_S_FULL, it & 1, abort_flag, tmo);
        trs.add(TR_SG_S_FULL, t0);
        if (!ok) break;
        ptx::tc_fence_after();
        float pv[NC];
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += 32) {
          float sv[32];
          ptx::tmem_ld32(tmem + lane_addr + C::T_S + col0 + c0, sv);
#pragma unroll
          for (int c = 0; c < 32; ++c) pv[c0 + c] = sv[c];
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + B_S_EMPTY);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const int qc = col0 + c;
          const float e = ptx::ex2(fmaf(pv[c], p.scale_log2, -lse_s[qc] * kLog2e));
          pv[c] = (diag && kv_g > q0 + qc) ? 0.f : e;
        }
        t0 = trs.t0();
        if (it > 0) ok = ptx::warp_wait(bars + B_P_EMPTY, (it - 1) & 1, abort_flag, tmo);
        trs.add(TR_SG_P_EMPTY, t0);
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < NC / 8; ++k) {
          const uint32_t a = sP + sw_chunk(r, (col0 >> 3) + k, kTile);
          ptx::st_shared_v4(a, ptx::pack_bf16(pv[8 * k], pv[8 * k + 1]),
                            ptx::pack_bf16(pv[8 * k + 2], pv[8 * k + 3]),
                            ptx::pack_bf16(pv[8 * k + 4], pv[8 * k + 5]),
                            ptx::pack_bf16(pv[8 * k + 6], pv[8 * k + 7]));
        }
        // (P is published together with dS below: the dV/dK/dQ issuer waits for both)
        ptx::fence_proxy_async_smem();
        t0 = trs.t0();
        ok = ptx::warp_wait(bars + B_DP_FULL, it & 1, abort_flag, tmo);
        trs.add(TR_SG_DP_FULL, t0);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += 32) {
          float dp[32];
          ptx::tmem_ld32(tmem + lane_addr + C::T_DP + col0 + c0, dp);
#pragma unroll
          for (int c = 0; c < 32; ++c) pv[c0 + c] = pv[c0 + c] * (dp[c] - dsum_s[col0 + c0 + c]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + B_DP_EMPTY);
        t0 = trs.t0();
        if (it > 0) ok = ptx::warp_wait(bars + B_DS_EMPTY, (it - 1) & 1, abort_flag, tmo);
        trs.add(TR_SG_DS_EMPTY, t0);
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < NC / 8; ++k) {
          const uint32_t a = sdS + sw_chunk(r, (col0 >> 3) + k, kTile);
          ptx::st_shared_v4(a, ptx::pack_bf16(pv[8 * k], pv[8 * k + 1]),
                            ptx::pack_bf16(pv[8 * k + 2], pv[8 * k + 3]),
                            ptx::pack_bf16(pv[8 * k + 4], pv[8 * k + 5]),
                            ptx::pack_bf16(pv[8 * k + 6], pv[8 * k + 7]));
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(bars + B_DS_FULL);
          ptx::mbar_arrive(bars + B_STAGE_EMPTY + s);
        }
      }
    }
  } else if (warp == 2) {
    // ===================================== dQ reducer =======================================
    // Adds each staged dQ partial into the fp32 accumulator with a TMA bulk reduce-add.
    // Deterministic mode takes the 128-row block's turn (semaphore == ordinal) before its
    // first sub-tile and hands it on (ordinal + 1) once the block's reduces have
    // completed -- always before this thread waits for its next turn. (Taking the next
    // turn first would let every CTA of a shift ring hold a release while waiting for its
    // neighbour's: a cycle.) The staging buffer is handed back as soon as it has been read.
    if (lane == 0) {
      Walk w(p);
      int it = 0;
      bool ok = true;
      while (ok && w.next()) {
        for (int hs = 0; hs < SUB && ok; ++hs, ++it) {
          const int q0 = w.j * kTile + hs * BR;
          long long t0 = tr.t0();
          ok = ptx::mbar_wait(bars + B_STG_FULL, it & 1, abort_flag, tmo);
          tr.add(TR_DQ_FULL, t0);
          if (!ok) break;
          const int ord = __ldg(p.ord + w.bh * p.ord_stride + w.i * p.n + w.j);
          const int chain = ord % p.chains, o = ord / p.chains;   // interleaved chains
          const int sem_idx = (w.bh * p.n + w.j) * kDqChains + chain;
          if (p.deterministic && hs == 0) {
            t0 = tr.t0();
            ok = wait_turn(p.sems + sem_idx, o + p.ordinal_skew, p.ws_header, p.timeout_ns,
                           w.bh, w.j);
            tr.add(TR_DQ_SEM, t0);
            if (!ok) {
              *abort_flag = 1;
              break;
            }
            ptx::fence_proxy_async_global();
          }
          t0 = tr.t0();
#pragma unroll
          for (int bx = 0; bx < D / 32; ++bx)
            ptx::tma_reduce_add_2d(&maps.acc, sm + L::STG_OFF + bx * (BR * 128), bx * 32,
                                   chain * p.B * p.H * p.S + w.bh * p.S + q0);
          ptx::bulk_commit();
          ptx::bulk_wait_read_all();
          ptx::mbar_arrive(bars + B_STG_EMPTY);
          if (p.deterministic && hs == SUB - 1) {
            ptx::bulk_wait_all();
            ptx::fence_proxy_async_global();   // the completed bulk adds, then the release
            st_release_gpu(p.sems + sem_idx, o + 1 + p.ordinal_skew);
          }
          tr.add(TR_DQ_REDUCE, t0);
        }
      }
      ptx::bulk_wait_all();
    }
  } else if (warp >= 12) {
    // ================== dQ read-out into the staging buffer + dK/dV epilogue =================
    const int quarter = warp & 3;
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const uint32_t stg = ptx::smem_u32(sm + L::STG_OFF);
    const Trace& trq = (warp == 12 && lane == 0) ? tr : tr_none;
    // nothing to read out before the first sub-tile: pre-arm its dS/dQ hand-off
    if (lane == 0) ptx::mbar_arrive(bars + B_DS_FULL);
    Walk w(p);
    int it = 0, tl = 0;
    bool ok = true;
    while (ok && w.next()) {
      const int b = w.bh / p.H, h = w.bh % p.H;
      for (int hs = 0; hs < SUB && ok; ++hs, ++it) {
        ok = ptx::warp_wait(bars + B_DQ_FULL, it & 1, abort_flag, tmo);
        if (!ok) break;
        ptx::tc_fence_after();
        float v[64];
        {
          float t0v[32], t1v[32];
          ptx::tmem_ld32(tmem + lane_addr + C::T_DQ, t0v);
          ptx::tmem_ld32(tmem + lane_addr + C::T_DQ + 32, t1v);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            v[c] = t0v[c];
            v[32 + c] = t1v[c];
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + B_DS_FULL);   // dQ(it) has left TMEM
        long long t0 = trq.t0();
        if (it > 0) ok = ptx::warp_wait(bars + B_STG_EMPTY, (it - 1) & 1, abort_flag, tmo);
        trq.add(TR_DQ_STAGE, t0);
        if (!ok) break;
        {
          // lanes = q rows; 64 d values; boxes of 32 fp32 columns x BR rows
          const int row = quarter * 32 + lane;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int bx = c >> 3, ch = c & 7;
            const uint32_t a = stg + bx * (BR * 128) + row * 128 + ((ch ^ (row & 7)) << 4);
            ptx::st_shared_v4(a, __float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                              __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + B_STG_FULL);
        // ---- dK/dV epilogue after the tile's last sub-task ----
        if (w.last_of_tile && hs == SUB - 1) {
          t0 = trq.t0();
          ok = ptx::warp_wait(bars + B_ACC_FULL, tl & 1, abort_flag, tmo);
          trq.add(TR_DQ_ACC_FULL, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          const int row = quarter * 32 + lane;        // kv row
          const size_t g = ((size_t)b * p.S + (size_t)w.i * kTile + row) * rs + (size_t)h * D;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float a[32];
            ptx::tmem_ld32(tmem + lane_addr + C::T_DV + c0, a);
            uint4* dst = (uint4*)(p.dv + g + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_uint4(ptx::pack_bf16(a[8 * k], a[8 * k + 1]),
                                  ptx::pack_bf16(a[8 * k + 2], a[8 * k + 3]),
                                  ptx::pack_bf16(a[8 * k + 4], a[8 * k + 5]),
                                  ptx::pack_bf16(a[8 * k + 6], a[8 * k + 7]));
            ptx::tmem_ld32(tmem + lane_addr + C::T_DK + c0, a);
            dst = (uint4*)(p.dk + g + c0);
            const float sc = p.scale;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_uint4(ptx::pack_bf16(sc * a[8 * k], sc * a[8 * k + 1]),
                                  ptx::pack_bf16(sc * a[8 * k + 2], sc * a[8 * k + 3]),
                                  ptx::pack_bf16(sc * a[8 * k + 4], sc * a[8 * k + 5]),
                                  ptx::pack_bf16(sc * a[8 * k + 6], sc * a[8 * k + 7]));
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bars + B_ACC_EMPTY);
          ++tl;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  // A CTA that gave up on any wait reports it, so an aborted run never reads as success.
  if (threadIdx.x == 0 && *abort_flag) {
    if (atomicCAS(p.ws_header + WS_STATUS, 0, kStatusSyncTimeout) == 0) {
      p.ws_header[WS_BH] = -1;          // -1: an in-CTA pipeline wait, not a dQ semaphore
      p.ws_header[WS_QTILE] = blockIdx.x;
      __threadfence();
    }
  }
  if (p.trace) {
    if (threadIdx.x == 0) trace_s[TR_TOTAL] = (unsigned long long)(clock64() - t_start);
    __syncthreads();
    if (threadIdx.x < TR_SITES) p.trace[(size_t)blockIdx.x * TR_SITES + threadIdx.x] = trace_s[threadIdx.x];
  }
}

}  // namespace tc
}  // namespace dash
