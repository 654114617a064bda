// Backward main kernel on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent CTA per SM. A unit is one schedule chain (slot) of one (batch, head);
// CTA c runs units c, c + grid, ... Each schedule task (KV_i, Q_j) covers a 128 x 128
// tile of the score matrix; KV_i's K and V tiles stay in shared memory for all its
// tasks and its dK/dV accumulate in TMEM (DASH's "each KV tile's dK/dV stay on one SM").
//
// Per Q sub-tile (BR query rows; BR = 128 for D = 64, 64 for D = 128):
//   S^T  = K Q^T          (M = 128 kv, N = BR, K = D)      -> TMEM
//   dP^T = V dO^T         (M = 128 kv, N = BR, K = D)      -> TMEM
//   P^T  = exp2(S^T * scale*log2e - LSE*log2e)            softmax-gradient warps -> smem bf16
//   dS^T = P^T * (dP^T - Dsum)                            softmax-gradient warps -> smem bf16
//   dV  += P^T dO         (M = 128 kv, N = D, K = BR)
//   dK  += dS^T Q         (M = 128 kv, N = D, K = BR)
//   D = 64 : dQ   = dS K    (M = 128 q, N = 64, K = 128 kv)   TMEM lanes = q rows
//   D = 128: dQ^T = K^T dS^T (M = 128 d, N = 64, K = 128 kv)  TMEM lanes = d columns
//   then the dQ partial is staged in smem and added into the fp32 dQ accumulator with a
//   TMA bulk reduce-add: deterministic mode waits on the block's L2 semaphore for its
//   ordinal first and releases ordinal + 1 after the add has completed (the pages' fixed
//   serial reduction order); non-deterministic mode adds as soon as it can.
//
// Warp roles (512 threads): warp 0 = TMA producer, warp 1 = MMA issuer, warps 4..11 =
// softmax-gradient (two warpgroups, each half of the BR columns), warps 12..15 = dQ
// reduction and dK/dV epilogue. Warps 2..3 idle. TMEM: 512 columns.
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
  static constexpr int T_S = 0, T_DP = 128, T_DV = 256, T_DK = 320, T_DQ = 384;
};

template <>
struct Cfg<128> {
  static constexpr int BR = 64;
  static constexpr int SUB = 2;
  static constexpr int T_S = 0, T_DP = 64, T_DV = 128, T_DK = 256, T_DQ = 384;
};

constexpr int kThreads = 512;
constexpr int kStages = 2;
constexpr int kTmemCols = 512;

// Shared-memory carve-up (byte offsets from a 1024-aligned base).
template <int D>
struct Smem {
  static constexpr int BR = Cfg<D>::BR;
  static constexpr int KV_BYTES = kTile * D * 2;             // one of K or V
  static constexpr int QT_BYTES = BR * D * 2;                // one of Q or dO (per stage)
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV_BYTES;
  static constexpr int STAGE_OFF = V_OFF + KV_BYTES;
  static constexpr int STAGE_BYTES = ((2 * QT_BYTES + 2 * BR * 4) + 1023) / 1024 * 1024;
  static constexpr int Q_IN_STAGE = 0;
  static constexpr int DO_IN_STAGE = QT_BYTES;
  static constexpr int LSE_IN_STAGE = 2 * QT_BYTES;
  static constexpr int DSUM_IN_STAGE = 2 * QT_BYTES + BR * 4;
  static constexpr int P_OFF = STAGE_OFF + kStages * STAGE_BYTES;
  static constexpr int PT_BYTES = kTile * BR * 2;            // P^T or dS^T tile
  static constexpr int DS_OFF = P_OFF + PT_BYTES;
  static constexpr int STG_OFF = DS_OFF + PT_BYTES;          // dQ staging (fp32)
  static constexpr int STG_BYTES = BR * D * 4;
  static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
  static constexpr int TRACE_OFF = BAR_OFF + 256;
  static constexpr int TOTAL = TRACE_OFF + 8 * TR_SITES;     // barriers, flags, trace
  static constexpr int ALLOC = TOTAL + 1024;                 // slack for 1024 alignment
};

// Barrier indices.
enum {
  B_KV_FULL = 0, B_KV_EMPTY, B_S_FULL, B_S_EMPTY, B_DP_FULL, B_DP_EMPTY, B_P_FULL, B_P_EMPTY,
  B_DS_FULL, B_DS_EMPTY, B_DQ_FULL, B_DQ_EMPTY, B_ACC_FULL, B_ACC_EMPTY, B_DRAIN,
  B_STAGE_FULL,                     // + stage
  B_STAGE_EMPTY = B_STAGE_FULL + kStages,
  B_COUNT = B_STAGE_EMPTY + kStages
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

// Iterates this CTA's (unit, task) sequence; every role walks the same sequence.
struct Walk {
  const BwdParams& p;
  int u, t, t_end, bh, i, j;
  bool first_of_tile, last_of_tile;
  __device__ Walk(const BwdParams& pp) : p(pp), u((int)blockIdx.x - (int)gridDim.x), t(0), t_end(0) {}
  __device__ bool next() {
    ++t;
    while (t >= t_end) {
      u += gridDim.x;
      if (u >= p.num_units) return false;
      const int slot = u % p.num_slots;
      bh = u / p.num_slots;
      t = p.slot_off[slot];
      t_end = p.slot_off[slot + 1];
    }
    const int32_t tk = __ldg(p.tasks + t);
    i = tk >> 16;
    j = tk & 0xffff;
    first_of_tile = (t == p.slot_off[u % p.num_slots]) || ((__ldg(p.tasks + t - 1) >> 16) != i);
    last_of_tile = (t + 1 == t_end) || ((__ldg(p.tasks + t + 1) >> 16) != i);
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
  constexpr int BR = C::BR, SUB = C::SUB;
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
    ptx::mbar_init(bars + B_P_FULL, 8);
    ptx::mbar_init(bars + B_P_EMPTY, 1);
    ptx::mbar_init(bars + B_DS_FULL, 8);
    ptx::mbar_init(bars + B_DS_EMPTY, 1);
    ptx::mbar_init(bars + B_DQ_FULL, 1);
    ptx::mbar_init(bars + B_DQ_EMPTY, 4);
    ptx::mbar_init(bars + B_ACC_FULL, 1);
    ptx::mbar_init(bars + B_ACC_EMPTY, 4);
    ptx::mbar_init(bars + B_DRAIN, 1);
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
        ptx::mbar_expect_tx(bars + B_STAGE_FULL + s, 2 * L::QT_BYTES + 2 * BR * 4);
        for (int cb = 0; cb < D / 64; ++cb) {
          ptx::tma_load_3d(st + L::Q_IN_STAGE + cb * BR * 128, &maps.q, cb * 64, h, b * p.S + q0,
                           bars + B_STAGE_FULL + s);
          ptx::tma_load_3d(st + L::DO_IN_STAGE + cb * BR * 128, &maps.dO, cb * 64, h, b * p.S + q0,
                           bars + B_STAGE_FULL + s);
        }
        ptx::bulk_load(st + L::LSE_IN_STAGE, p.lse + (size_t)bh * p.S + q0, BR * 4,
                       bars + B_STAGE_FULL + s);
        ptx::bulk_load(st + L::DSUM_IN_STAGE, p.Dsum + (size_t)bh * p.S + q0, BR * 4,
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
  } else if (warp == 1) {
    // ===================================== MMA issuer =======================================
    // Software-pipelined issue order per sub-tile t:
    //   dV(t), S(t+1), dK(t), dQ(t), dP(t+1)
    // so the softmax-gradient warps compute P(t+1) while dK(t)/dQ(t) run. At a KV-tile
    // boundary S(t+1) waits for the new K/V tile instead.
    if (lane == 0) {
      const uint32_t sK = ptx::smem_u32(sm + L::K_OFF), sV = ptx::smem_u32(sm + L::V_OFF);
      const uint32_t sP = ptx::smem_u32(sm + L::P_OFF), sdS = ptx::smem_u32(sm + L::DS_OFF);
      constexpr uint32_t ID_S = ptx::idesc_bf16(128, BR, 0, 0);     // S^T, dP^T
      constexpr uint32_t ID_ACC = ptx::idesc_bf16(128, D, 0, 1);    // dV, dK
      constexpr uint32_t ID_DQ = ptx::idesc_bf16(128, 64, 1, 1);    // dQ (D=64) / dQ^T (D=128)
      auto stage_addr = [&](const Sub& x) {
        return ptx::smem_u32(sm + L::STAGE_OFF + (x.it % kStages) * L::STAGE_BYTES);
      };
      auto issue_S = [&](const Sub& x) -> bool {
        long long t0 = tr.t0();
        if (x.first && !ptx::mbar_wait(bars + B_KV_FULL, x.tile & 1, abort_flag, tmo)) return false;
        tr.add(TR_MMA_KV_FULL, t0);
        t0 = tr.t0();
        if (!ptx::mbar_wait(bars + B_STAGE_FULL + x.it % kStages, (x.it / kStages) & 1, abort_flag,
                            tmo))
          return false;
        tr.add(TR_MMA_STAGE_FULL, t0);
        t0 = tr.t0();
        if (x.it > 0 && !ptx::mbar_wait(bars + B_S_EMPTY, (x.it - 1) & 1, abort_flag, tmo))
          return false;
        tr.add(TR_MMA_S_EMPTY, t0);
        ptx::tc_fence_after();
        const uint32_t sQ = stage_addr(x) + L::Q_IN_STAGE;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ao = (ks / 4) * (kTile * 128) + (ks % 4) * 32;
          const uint32_t bo = (ks / 4) * (BR * 128) + (ks % 4) * 32;
          ptx::mma_bf16(tmem + C::T_S, ptx::sdesc(sK + ao, 16, 1024), ptx::sdesc(sQ + bo, 16, 1024),
                        ID_S, ks > 0);
        }
        ptx::mma_commit(bars + B_S_FULL);
        return true;
      };
      auto issue_dP = [&](const Sub& x) -> bool {
        const long long t0 = tr.t0();
        if (x.it > 0 && !ptx::mbar_wait(bars + B_DP_EMPTY, (x.it - 1) & 1, abort_flag, tmo))
          return false;
        tr.add(TR_MMA_DP_EMPTY, t0);
        ptx::tc_fence_after();
        const uint32_t sdO = stage_addr(x) + L::DO_IN_STAGE;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ao = (ks / 4) * (kTile * 128) + (ks % 4) * 32;
          const uint32_t bo = (ks / 4) * (BR * 128) + (ks % 4) * 32;
          ptx::mma_bf16(tmem + C::T_DP, ptx::sdesc(sV + ao, 16, 1024),
                        ptx::sdesc(sdO + bo, 16, 1024), ID_S, ks > 0);
        }
        ptx::mma_commit(bars + B_DP_FULL);
        return true;
      };
      SubWalk<SUB> sw(p);
      Sub cur, nxt;
      bool have = sw.next(cur);
      bool ok = true;
      if (have) ok = issue_S(cur) && issue_dP(cur);
      while (ok && have) {
        const bool have_n = sw.next(nxt);
        const bool same_tile = have_n && !nxt.first;
        const uint32_t st = stage_addr(cur);
        const uint32_t sQ = st + L::Q_IN_STAGE, sdO = st + L::DO_IN_STAGE;
        // dV += P^T dO: A = P^T (K-major, 128 kv rows x BR), B = dO (MN-major over D).
        // The first sub-tile of a KV tile overwrites the accumulators, which the previous
        // tile's epilogue must have read out.
        long long t0 = tr.t0();
        ok = ptx::mbar_wait(bars + B_P_FULL, cur.it & 1, abort_flag, tmo);
        tr.add(TR_MMA_P_FULL, t0);
        t0 = tr.t0();
        if (ok && cur.first && cur.tile > 0)
          ok = ptx::mbar_wait(bars + B_ACC_EMPTY, (cur.tile - 1) & 1, abort_flag, tmo);
        tr.add(TR_MMA_ACC_EMPTY, t0);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BR / 16; ++ks) {
          const uint32_t ao = (ks / 4) * (kTile * 128) + (ks % 4) * 32;
          ptx::mma_bf16(tmem + C::T_DV, ptx::sdesc(sP + ao, 16, 1024),
                        ptx::sdesc(sdO + ks * 2048, BR * 128, 1024), ID_ACC,
                        !(cur.first && ks == 0));
        }
        ptx::mma_commit(bars + B_P_EMPTY);
        if (same_tile && !(ok = issue_S(nxt))) break;
        // dK += dS^T Q, then the dQ partial over the 128 kv rows
        t0 = tr.t0();
        ok = ptx::mbar_wait(bars + B_DS_FULL, cur.it & 1, abort_flag, tmo);
        tr.add(TR_MMA_DS_FULL, t0);
        t0 = tr.t0();
        if (ok && cur.it > 0) ok = ptx::mbar_wait(bars + B_DQ_EMPTY, (cur.it - 1) & 1, abort_flag, tmo);
        tr.add(TR_MMA_DQ_EMPTY, t0);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BR / 16; ++ks) {
          const uint32_t ao = (ks / 4) * (kTile * 128) + (ks % 4) * 32;
          ptx::mma_bf16(tmem + C::T_DK, ptx::sdesc(sdS + ao, 16, 1024),
                        ptx::sdesc(sQ + ks * 2048, BR * 128, 1024), ID_ACC,
                        !(cur.first && ks == 0));
        }
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          if (D == 64) {
            // dQ = dS K: A = dS (MN-major view of the dS^T tile), B = K (MN-major, 64 d)
            ptx::mma_bf16(tmem + C::T_DQ, ptx::sdesc(sdS + ks * 2048, kTile * 128, 1024),
                          ptx::sdesc(sK + ks * 2048, kTile * 128, 1024), ID_DQ, ks > 0);
          } else {
            // dQ^T = K^T dS^T: A = K^T (MN-major over 128 d), B = dS^T (MN-major, 64 q)
            ptx::mma_bf16(tmem + C::T_DQ, ptx::sdesc(sK + ks * 2048, kTile * 128, 1024),
                          ptx::sdesc(sdS + ks * 2048, kTile * 128, 1024), ID_DQ, ks > 0);
          }
        }
        ptx::mma_commit(bars + B_DS_EMPTY);
        ptx::mma_commit(bars + B_DQ_FULL);
        ptx::mma_commit(bars + B_STAGE_EMPTY + cur.it % kStages);
        if (cur.last) {
          ptx::mma_commit(bars + B_ACC_FULL);
          ptx::mma_commit(bars + B_KV_EMPTY);
        }
        if (have_n) {
          if (!same_tile && !(ok = issue_S(nxt))) break;
          if (!(ok = issue_dP(nxt))) break;
        }
        cur = nxt;
        have = have_n;
      }
      // drain: no MMA may be in flight when TMEM is released
      ptx::mma_commit(bars + B_DRAIN);
      ptx::mbar_drain(bars + B_DRAIN, 0, 1000000000ll);
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
        const float* lse_s = (const float*)(sm + L::STAGE_OFF + s * L::STAGE_BYTES + L::LSE_IN_STAGE);
        const float* dsum_s = (const float*)(sm + L::STAGE_OFF + s * L::STAGE_BYTES + L::DSUM_IN_STAGE);
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
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + B_P_FULL);
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
  } else if (warp >= 12) {
    // ============================ dQ reduction + dK/dV epilogue ============================
    // Every named barrier below is reached by all four warps unconditionally; a failed
    // wait is agreed on through wg_ok before anyone leaves the loop.
    const int quarter = warp & 3;
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const uint32_t stg = ptx::smem_u32(sm + L::STG_OFF);
    const bool leader = (warp == 12 && lane == 0);
    const Trace& trq = leader ? tr : tr_none;
    __shared__ int go_flag;
    __shared__ int wg_ok[4];
    auto agree = [&](bool mine) -> bool {
      if (lane == 0) wg_ok[quarter] = mine ? 1 : 0;
      ptx::named_bar(1, 128);
      const bool all = wg_ok[0] && wg_ok[1] && wg_ok[2] && wg_ok[3];
      ptx::named_bar(1, 128);
      return all;
    };
    Walk w(p);
    int it = 0, tl = 0;
    bool ok = true;
    while (ok && w.next()) {
      const int b = w.bh / p.H, h = w.bh % p.H;
      for (int hs = 0; hs < SUB && ok; ++hs, ++it) {
        const int q0 = w.j * kTile + hs * BR;
        long long t0 = trq.t0();
        ok = agree(ptx::warp_wait(bars + B_DQ_FULL, it & 1, abort_flag, tmo));
        trq.add(TR_DQ_FULL, t0);
        if (!ok) break;
        t0 = trq.t0();
        ptx::tc_fence_after();
        float v[64];
        {
          float t0[32], t1[32];
          ptx::tmem_ld32(tmem + lane_addr + C::T_DQ, t0);
          ptx::tmem_ld32(tmem + lane_addr + C::T_DQ + 32, t1);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            v[c] = t0[c];
            v[32 + c] = t1[c];
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + B_DQ_EMPTY);
        // the staging buffer is free: the previous reduce finished reading it before the
        // leader reached the last barrier of the previous iteration
        if (D == 64) {
          // lanes = q rows; 64 d values; boxes of 32 fp32 columns x BR rows
          const int row = quarter * 32 + lane;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int bx = c >> 3, ch = c & 7;
            const uint32_t a = stg + bx * (BR * 128) + row * 128 + ((ch ^ (row & 7)) << 4);
            ptx::st_shared_v4(a, __float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                              __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
          }
        } else {
          // lanes = d (= 32 * quarter + lane); 64 q values; box = quarter
#pragma unroll
          for (int q = 0; q < 64; ++q) {
            const uint32_t a = stg + quarter * (BR * 128) + q * 128 +
                               ((((lane >> 2) ^ (q & 7))) << 4) + (lane & 3) * 4;
            ptx::st_shared_f32(a, v[q]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::named_bar(1, 128);
        trq.add(TR_DQ_STAGE, t0);
        if (leader) {
          int go = 1;
          const int sem_idx = (w.bh * p.n + w.j) * SUB + hs;
          const int o = p.ord[w.i * p.n + w.j];
          t0 = trq.t0();
          if (p.deterministic) {
            go = wait_turn(p.sems + sem_idx, o + p.ordinal_skew, p.ws_header, p.timeout_ns,
                           w.bh, w.j)
                     ? 1
                     : 0;
            ptx::fence_proxy_async_global();
          }
          trq.add(TR_DQ_SEM, t0);
          t0 = trq.t0();
          if (go) {
#pragma unroll
            for (int bx = 0; bx < D / 32; ++bx)
              ptx::tma_reduce_add_2d(&maps.acc, sm + L::STG_OFF + bx * (BR * 128), bx * 32,
                                     w.bh * p.S + q0);
            ptx::bulk_commit();
            if (p.deterministic) {
              ptx::bulk_wait_all();
              ptx::fence_proxy_async_global();
              __threadfence();
              st_release_gpu(p.sems + sem_idx, o + 1 + p.ordinal_skew);
            } else {
              ptx::bulk_wait_read_all();
            }
          } else {
            *abort_flag = 1;
          }
          trq.add(TR_DQ_REDUCE, t0);
          go_flag = go;
        }
        ptx::named_bar(1, 128);
        if (!go_flag) {
          ok = false;
          break;
        }
        // ---- dK/dV epilogue after the tile's last sub-task ----
        if (w.last_of_tile && hs == SUB - 1) {
          t0 = trq.t0();
          ok = agree(ptx::warp_wait(bars + B_ACC_FULL, tl & 1, abort_flag, tmo));
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
    if (leader) ptx::bulk_wait_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (p.trace) {
    if (threadIdx.x == 0) trace_s[TR_TOTAL] = (unsigned long long)(clock64() - t_start);
    __syncthreads();
    if (threadIdx.x < TR_SITES) p.trace[(size_t)blockIdx.x * TR_SITES + threadIdx.x] = trace_s[threadIdx.x];
  }
}

}  // namespace tc
}  // namespace dash
