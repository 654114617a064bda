// Backward main kernel for head dimension 128: whole 128 x 128 tasks, software-pipelined.
//
// Same persistent grid, units, schedule walk and ordered dQ reduction as the general
// kernel (kernels_tc.cuh); what differs is how one task (KV_i, Q_j) maps onto the SM:
//
//   S    = Q K^T        M = 128 q, N = 128 kv, K = 128 d     TMEM cols [0, 128)
//   P    = exp2(S * scale*log2e - LSE*log2e)                 smem bf16 [q][kv]
//   dP   = dO V^T       M = 128 q, N = 128 kv, K = 128 d     TMEM cols [0, 128) again
//   dS   = P * (dP - Dsum)                                   smem bf16 [q][kv], P's buffer
//   dV  += P^T dO       M = 128 kv, N = 128 d, K = 128 q     TMEM cols [256, 384)
//   dK  += dS^T Q       M = 128 kv, N = 128 d, K = 128 q     TMEM cols [384, 512)
//   dQ^T = K^T dS^T     M = 128 d, N = 128 q, K = 128 kv     TMEM cols [128, 256)
//
// S and dP have the query rows in the TMEM lanes, so each softmax-gradient thread owns one
// query row: its -LSE*log2e and Dsum are two scalars, and forming P and dS needs no
// shared-memory reads at all. P^T and dS^T are read by the tensor core as MN-major views
// of the [q][kv] tiles.
//
// Every MMA is 128 x 128 x 16 per instruction; measured on GB300 each such instruction
// takes ~65 cycles whatever the operand majors, i.e. the tensor core's full rate, so a
// task's five products need ~2600 cycles of tensor time. The kernel is laid out so that
// the tensor pipe never waits for the softmax-gradient warps: one thread issues the
// products in the fixed order
//
//   S(t), dK(t-1), dQ^T(t-1), dP(t), dV(t)
//
// so that between any product and the softmax-gradient result it needs there is at
// least one other product already queued:
//   - dP(t) reuses S's columns; it waits only for the softmax-gradient warps to have
//     loaded S(t) (dK(t-1) and dQ^T(t-1) run meanwhile);
//   - dV(t) waits for P(t), which the exponentials produce while dK(t-1), dQ^T(t-1)
//     and dP(t) run;
//   - S(t+1) reuses the columns again once dP(t) has been loaded (dV(t) runs meanwhile);
//   - dK(t) and dQ^T(t) wait for dS(t), formed while dV(t) and S(t+1) run.
// P and dS share one shared-memory tile: dS(t) is stored once dV(t) has read P(t), and
// P(t+1) once dQ^T(t) has read dS(t). Q and dO are double-buffered by task
// parity: Q(t+2) loads once dK(t) has run, dO(t+2) once dV(t) has. At the end of a KV
// tile the pending dK/dQ^T are issued before the next tile's S^T (they still read the old
// K), and K, V reload after them.
//
// The dQ^T columns are read into registers by the read-out warpgroup and handed back at
// once; the partial is then added into the fp32 dQ accumulator with coalesced red.global
// (TMEM lane = d, so one warp instruction covers 32 consecutive d of one row: a full
// 128-byte line). In deterministic mode the adds of a 128-row block wait for the block's
// turn and the turn is handed on after they have been performed.
//
// Shared memory (1024-aligned base, checked): K, V, Q x 2, dO x 2, P^T/dS^T, -LSE*log2e
// and Dsum per Q buffer, barriers, trace: 231,936 bytes.
//
// Warp roles (512 threads): 0 = TMA producer, 1 = MMA issuer, 2, 3 = idle,
// 4..11 = softmax-gradient (quarter = TMEM lanes = query rows, half = 64 kv columns),
// 12..15 = dQ read-out and reduction, and the dK/dV epilogue.
#pragma once

#include "kernels_tc.cuh"

namespace dash {
namespace tc {

struct L128 {
  static constexpr int D = 128;
  static constexpr int TILE_BYTES = kTile * D * 2;            // one 128 x 128 bf16 tile
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE_BYTES;
  static constexpr int Q_OFF = V_OFF + TILE_BYTES;            // two Q buffers
  static constexpr int DO_OFF = Q_OFF + 2 * TILE_BYTES;       // two dO buffers
  static constexpr int PDS_OFF = DO_OFF + 2 * TILE_BYTES;     // P, then dS [q][kv]
  static constexpr int LD_OFF = PDS_OFF + TILE_BYTES;         // per Q buffer: -LSE*log2e, Dsum
  static constexpr int LD_BYTES = 2 * kTile * 4;
  static constexpr int BAR_OFF = LD_OFF + 2 * LD_BYTES;
  static constexpr int TRACE_OFF = BAR_OFF + 320;
  static constexpr int ALLOC = TRACE_OFF + 8 * TR_SITES;
  static_assert(ALLOC <= 232448, "shared memory budget");
  // TMEM columns
  static constexpr int T_SP = 0, T_DQ = 128, T_DV = 256, T_DK = 384;
  // registers per thread after the re-split (launch: 128 x 512 threads)
  static constexpr int REGS_LAUNCH = 128, REGS_SINGLE = 88, REGS_READOUT = 168;
  static_assert(REGS_SINGLE + 2 * REGS_LAUNCH + REGS_READOUT == 4 * REGS_LAUNCH,
                "the four warpgroups must share exactly the launch's registers");
};

enum {
  E_KV_FULL = 0, E_KV_EMPTY, E_Q_FULL, E_Q_EMPTY = E_Q_FULL + 2, E_DO_FULL = E_Q_EMPTY + 2,
  E_DO_EMPTY = E_DO_FULL + 2, E_S_FULL = E_DO_EMPTY + 2, E_S_LOADED, E_P_FULL, E_DP_FULL,
  E_DP_LOADED, E_P_READ, E_DS_FULL, E_DS_READ, E_DQ_FULL, E_DQ_EMPTY, E_ACC_FULL,
  E_ACC_EMPTY, E_DRAIN, E_TURN, E_REDS, E_COUNT
};
static_assert(8 * E_COUNT + 8 <= 320, "barrier area");

// Wait- and work-cycle sites of this kernel's optional trace, each counted in one of the
// shared trace slots (dash_debug_set_trace; one writer per slot).
enum : int {
  K_PROD_Q_EMPTY = TR_PROD_STAGE_EMPTY,   // producer: a Q buffer is free
  K_PROD_KV_EMPTY = TR_PROD_KV_EMPTY,     // producer: K and V are free
  K_PROD_DO_EMPTY = TR_MMA_DQ_EMPTY,      // producer: a dO buffer is free
  K_X_KV_FULL = TR_MMA_KV_FULL,           // issuer: K and V landed
  K_X_Q_FULL = TR_MMA_STAGE_FULL,         // issuer: Q landed
  K_X_DP_LOADED = TR_MMA_S_EMPTY,         // issuer: previous dP^T loaded out of TMEM
  K_X_DO_S_LOADED = TR_MMA_DP_EMPTY,      // issuer: dO landed, S^T loaded out of TMEM
  K_X_P_FULL = TR_MMA_P_FULL,             // issuer: P^T stored
  K_X_ACC_EMPTY = TR_MMA_ACC_EMPTY,       // issuer: dK/dV accumulators read out
  K_X_DS_FULL = TR_MMA_DS_FULL,           // issuer: dS^T stored
  K_X_DQ_EMPTY = TR_SG_DS_EMPTY,          // issuer: previous dQ^T read out
  K_SG_S_FULL = TR_SG_S_FULL,             // softmax-gradient: S^T ready
  K_SG_P_COMPUTE = TR_DQ_FULL,            // softmax-gradient: exp2 of the scores
  K_SG_DP_FULL = TR_SG_DP_FULL,           // softmax-gradient: dP^T ready
  K_SG_BUF = TR_DQ_STAGE,                 // softmax-gradient: the P^T/dS^T tile is free
  K_SG_DS_COMPUTE = TR_SG_P_EMPTY,        // softmax-gradient: dP^T load and dS^T
  K_SG_S_LOAD = TR_X1,                    // softmax-gradient: S^T out of TMEM
  K_SG_P_STORE = TR_X2,                   // softmax-gradient: P^T into shared memory
  K_SG_DS_STORE = TR_X3,                  // softmax-gradient: dS^T into shared memory
  K_X_WALK = TR_X0,                       // issuer: stepping the task walk
  K_RO_DQ_LOAD = TR_X4,                   // read-out: dQ^T out of TMEM
  K_RO_EPILOGUE = TR_X5,                  // read-out: dK/dV out of TMEM to global memory
  K_RO_DQ_FULL = TR_ISSUE_DP,             // read-out: dQ^T ready
  K_RO_SEM = TR_DQ_SEM,                   // read-out: the block's turn (deterministic)
  K_RO_REDUCE = TR_DQ_REDUCE,             // read-out: adds and hand-off
  K_RO_ACC_FULL = TR_DQ_ACC_FULL,         // read-out: dK/dV accumulators final
  K_ISSUE_SDP = TR_ISSUE_S,               // issuer: issuing S^T and dP^T
  K_ISSUE_DV = TR_ISSUE_DV,               // issuer: issuing dV
  K_ISSUE_DQDK = TR_ISSUE_DKDQ            // issuer: issuing dK and dQ^T
};

// K-major step ks of a [128 rows][128] bf16 tile in 64-column blocks, in 16-byte units;
// an MN-major step is 16 rows of 128 bytes.
__device__ __forceinline__ uint32_t kstep128(int ks) {
  return ((ks >> 2) * kTile * 128 + (ks & 3) * 32) >> 4;
}
constexpr uint32_t kMnStep = 2048 >> 4;

// Slots of the MMA issuer's gap-free trace and the shared trace sites they are added to.
enum : int {
  X_WALK = 0, X_KV_FULL, X_Q_FULL, X_DP_LOADED, X_ISSUE_SDP, X_DS_FULL, X_ISSUE_DKDQ,
  X_DQ_EMPTY, X_DO_S_LOADED, X_P_FULL, X_ACC_EMPTY, X_ISSUE_DV, X_SLOTS
};
__device__ constexpr int kIssuerSites[X_SLOTS] = {
    K_X_WALK, K_X_KV_FULL, K_X_Q_FULL, K_X_DP_LOADED, K_ISSUE_SDP, K_X_DS_FULL, K_ISSUE_DQDK,
    K_X_DQ_EMPTY, K_X_DO_S_LOADED, K_X_P_FULL, K_X_ACC_EMPTY, K_ISSUE_DV};
using IssuerTrace = SegTrace<X_SLOTS>;

// Sites of the softmax-gradient warps' gap-free trace (one thread: warp 4, lane 0).
enum : int {
  G_S_FULL = K_SG_S_FULL, G_S_LOAD = K_SG_S_LOAD, G_EXP = K_SG_P_COMPUTE, G_BUF = K_SG_BUF,
  G_P_STORE = K_SG_P_STORE, G_DP_FULL = K_SG_DP_FULL, G_DS = K_SG_DS_COMPUTE,
  G_DS_STORE = K_SG_DS_STORE
};

// Issues S(t) = Q(t) K^T into the S/dP columns once Q(t) has landed and the
// softmax-gradient warps have loaded dP(t-1) out of those columns.
__device__ __forceinline__ bool issue_s128(uint64_t* bars, volatile int* abort_flag, long long tmo,
                                           IssuerTrace& tr, uint32_t tmem, uint32_t dQ_k,
                                           uint32_t dK_k, int t) {
  constexpr uint32_t ID_S = ptx::idesc_bf16(128, 128, 0, 0);
  bool good = ptx::mbar_wait(bars + E_Q_FULL + (t & 1), (t >> 1) & 1, abort_flag, tmo);
  tr.mark(X_Q_FULL);
  if (good && t > 0) good = ptx::mbar_wait(bars + E_DP_LOADED, (t - 1) & 1, abort_flag, tmo);
  tr.mark(X_DP_LOADED);
  if (!good) return false;
  ptx::tc_fence_after();
#pragma unroll
  for (int ks = 0; ks < 128 / 16; ++ks)
    ptx::mma_lo(tmem + L128::T_SP, dQ_k + kstep128(ks), dK_k + kstep128(ks), ID_S, ks > 0);
  ptx::mma_commit(bars + E_S_FULL);
  tr.mark(X_ISSUE_SDP);
  return true;
}

// Issues dK(t) += dS^T Q(t) once dS(t) is stored, then dQ^T(t) = K^T dS^T once the
// read-out has taken dQ^T(t-1) out of its columns.
__device__ __forceinline__ bool issue_dk_dq128(uint64_t* bars, volatile int* abort_flag,
                                               long long tmo, IssuerTrace& tr, uint32_t tmem,
                                               uint32_t dQ_mn, uint32_t dPDS_mn, uint32_t dK_mn,
                                               uint32_t dDS_k, int t, bool first) {
  constexpr uint32_t ID_ACC = ptx::idesc_bf16(128, 128, 1, 1);  // dK
  constexpr uint32_t ID_DQT = ptx::idesc_bf16(128, 128, 1, 0);  // dQ^T = K^T dS^T
  bool good = ptx::mbar_wait(bars + E_DS_FULL, t & 1, abort_flag, tmo);
  tr.mark(X_DS_FULL);
  if (!good) return false;
  ptx::tc_fence_after();
  // dK += dS^T Q: A = dS^T (MN-major over kv), B = Q (MN-major over d)
#pragma unroll
  for (int ks = 0; ks < kTile / 16; ++ks)
    ptx::mma_lo(tmem + L128::T_DK, dPDS_mn + ks * kMnStep, dQ_mn + ks * kMnStep, ID_ACC,
                (ks > 0 || !first) ? 1u : 0u);
  ptx::mma_commit(bars + E_Q_EMPTY + (t & 1));       // Q(t)'s last reader
  tr.mark(X_ISSUE_DKDQ);
  if (t > 0) good = ptx::mbar_wait(bars + E_DQ_EMPTY, (t - 1) & 1, abort_flag, tmo);
  tr.mark(X_DQ_EMPTY);
  if (!good) return false;
  ptx::tc_fence_after();
  // dQ^T = K^T dS^T: A = K^T (MN-major over d), B = dS^T (K-major over kv)
#pragma unroll
  for (int ks = 0; ks < kTile / 16; ++ks)
    ptx::mma_lo(tmem + L128::T_DQ, dK_mn + ks * kMnStep, dDS_k + kstep128(ks), ID_DQT, ks > 0);
  ptx::mma_commit(bars + E_DS_READ);                 // dK(t) and dQ^T(t) have read dS(t)
  ptx::mma_commit(bars + E_DQ_FULL);
  tr.mark(X_ISSUE_DKDQ);
  return true;
}

// Writes 64 values of query row r (kv columns col0..col0+63) as bf16 into the [q][kv] tile
// at sPDS (128-byte swizzle), then makes them visible to the tensor core.
__device__ __forceinline__ void store_row128(uint32_t sPDS, int r, int col0, const float (&v)[64]) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    ptx::st_shared_v4(sPDS + sw_chunk(r, (col0 >> 3) + k, kTile),
                      ptx::pack_bf16(v[8 * k], v[8 * k + 1]), ptx::pack_bf16(v[8 * k + 2], v[8 * k + 3]),
                      ptx::pack_bf16(v[8 * k + 4], v[8 * k + 5]), ptx::pack_bf16(v[8 * k + 6], v[8 * k + 7]));
  ptx::fence_proxy_async_smem();
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc128_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ TmaMaps maps) {
  using L = L128;
  constexpr int D = 128;
  extern __shared__ __align__(1024) uint8_t smem128[];
  uint8_t* sm = smem128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The layout fills the opt-in maximum, so there is no room to realign the base.
  if (ptx::smem_u32(sm) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.ws_header + WS_STATUS, 0, kStatusSmemLayout);
    return;
  }
  uint64_t* bars = (uint64_t*)(sm + L::BAR_OFF);
  uint32_t* tmem_slot = (uint32_t*)(sm + L::BAR_OFF + 8 * E_COUNT);
  volatile int* abort_flag = (volatile int*)(sm + L::BAR_OFF + 8 * E_COUNT + 4);
  const long long tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bars + E_KV_FULL, 1);
    ptx::mbar_init(bars + E_KV_EMPTY, 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bars + E_Q_FULL + b, 1);
      ptx::mbar_init(bars + E_Q_EMPTY + b, 1);
      ptx::mbar_init(bars + E_DO_FULL + b, 1);
      ptx::mbar_init(bars + E_DO_EMPTY + b, 1);
    }
    ptx::mbar_init(bars + E_S_FULL, 1);
    ptx::mbar_init(bars + E_S_LOADED, 8);
    ptx::mbar_init(bars + E_P_FULL, 8);
    ptx::mbar_init(bars + E_DP_FULL, 1);
    ptx::mbar_init(bars + E_DP_LOADED, 8);
    ptx::mbar_init(bars + E_P_READ, 1);
    ptx::mbar_init(bars + E_DS_FULL, 8);
    ptx::mbar_init(bars + E_DS_READ, 1);
    ptx::mbar_init(bars + E_DQ_FULL, 1);
    ptx::mbar_init(bars + E_DQ_EMPTY, 4);
    ptx::mbar_init(bars + E_ACC_FULL, 1);
    ptx::mbar_init(bars + E_ACC_EMPTY, 4);
    ptx::mbar_init(bars + E_DRAIN, 1);
    ptx::mbar_init(bars + E_TURN, 1);
    ptx::mbar_init(bars + E_REDS, 3);
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

  // Warpgroup 0 runs one thread per warp and gives registers to the read-out warpgroup,
  // which holds a 128-column row. Each re-split is one instruction executed by all four
  // warps of its warpgroup, ahead of (and dominating) that warpgroup's role code.
  if (warp < 4) {
    ptx::regs_dec<L::REGS_SINGLE>();
    if (warp == 0 && lane == 0) {
      // ===================================== TMA producer =====================================
      const Trace tr{p.trace ? trace_s : nullptr};
      Walk w(p);
      int it = 0, tl = 0;
      bool ok = true;
      while (ok && w.next()) {
        const int b = w.bh / p.H, h = w.bh % p.H;
        const int q0 = w.j * kTile, qb = it & 1;
        // Q_j with its -LSE*log2e and Dsum rows into Q buffer qb (free once dK of task it-2
        // has run)
        long long t0 = tr.t0();
        if (it >= 2 && !(ok = ptx::mbar_wait(bars + E_Q_EMPTY + qb, ((it >> 1) - 1) & 1, abort_flag, tmo)))
          break;
        tr.add(K_PROD_Q_EMPTY, t0);
        uint8_t* qs = sm + L::Q_OFF + qb * L::TILE_BYTES;
        uint8_t* ld = sm + L::LD_OFF + qb * L::LD_BYTES;
        ptx::mbar_expect_tx(bars + E_Q_FULL + qb, L::TILE_BYTES + L::LD_BYTES);
        for (int cb = 0; cb < 2; ++cb)
          ptx::tma_load_3d(qs + cb * kTile * 128, &maps.q, cb * 64, h, b * p.S + q0, bars + E_Q_FULL + qb);
        ptx::bulk_load(ld, p.nlse2 + (size_t)w.bh * p.S + q0, kTile * 4, bars + E_Q_FULL + qb);
        ptx::bulk_load(ld + kTile * 4, p.Dsum + (size_t)w.bh * p.S + q0, kTile * 4, bars + E_Q_FULL + qb);
        // K and V of a new KV tile, once the previous tile's last MMAs have read them
        if (w.first_of_tile) {
          t0 = tr.t0();
          if (tl > 0 && !(ok = ptx::mbar_wait(bars + E_KV_EMPTY, (tl - 1) & 1, abort_flag, tmo))) break;
          tr.add(K_PROD_KV_EMPTY, t0);
          ptx::mbar_expect_tx(bars + E_KV_FULL, 2 * L::TILE_BYTES);
          for (int cb = 0; cb < 2; ++cb) {
            ptx::tma_load_3d(sm + L::K_OFF + cb * kTile * 128, &maps.k, cb * 64, h,
                             b * p.S + w.i * kTile, bars + E_KV_FULL);
            ptx::tma_load_3d(sm + L::V_OFF + cb * kTile * 128, &maps.v, cb * 64, h,
                             b * p.S + w.i * kTile, bars + E_KV_FULL);
          }
          ++tl;
        }
        // dO_j into dO buffer qb (free once dV of task it-2 has run)
        t0 = tr.t0();
        if (it >= 2 && !(ok = ptx::mbar_wait(bars + E_DO_EMPTY + qb, ((it >> 1) - 1) & 1, abort_flag, tmo)))
          break;
        tr.add(K_PROD_DO_EMPTY, t0);
        ptx::mbar_expect_tx(bars + E_DO_FULL + qb, L::TILE_BYTES);
        for (int cb = 0; cb < 2; ++cb)
          ptx::tma_load_3d(sm + L::DO_OFF + qb * L::TILE_BYTES + cb * kTile * 128, &maps.dO, cb * 64,
                           h, b * p.S + q0, bars + E_DO_FULL + qb);
        ++it;
      }
      // drain: every issued load has landed before the CTA may exit
      for (int k = (it > 2 ? it - 2 : 0); k < it; ++k) {
        ptx::mbar_drain(bars + E_Q_FULL + (k & 1), (k >> 1) & 1, 100000000ll);
        ptx::mbar_drain(bars + E_DO_FULL + (k & 1), (k >> 1) & 1, 100000000ll);
      }
      if (tl > 0) ptx::mbar_drain(bars + E_KV_FULL, (tl - 1) & 1, 100000000ll);
    } else if (warp == 1 && lane == 0) {
      // ===================================== MMA issuer =======================================
      IssuerTrace tr(p.trace ? trace_s : nullptr);
      const uint32_t sK = ptx::smem_u32(sm + L::K_OFF), sV = ptx::smem_u32(sm + L::V_OFF);
      const uint32_t sQ = ptx::smem_u32(sm + L::Q_OFF), sdO = ptx::smem_u32(sm + L::DO_OFF);
      const uint32_t sPDS = ptx::smem_u32(sm + L::PDS_OFF);
      const uint32_t dK_k = ptx::sdesc_lo(sK, 16), dV_k = ptx::sdesc_lo(sV, 16);
      const uint32_t dK_mn = ptx::sdesc_lo(sK, kTile * 128);
      // P / dS [q][kv]: P^T and dS^T as MN-major A operands of dV and dK; dS^T as the
      // K-major B operand of dQ^T
      const uint32_t dPDS_mn = ptx::sdesc_lo(sPDS, kTile * 128), dDS_k = ptx::sdesc_lo(sPDS, 16);
      const uint32_t dQ_k0 = ptx::sdesc_lo(sQ, 16), dQ_mn0 = ptx::sdesc_lo(sQ, kTile * 128);
      const uint32_t ddO_k0 = ptx::sdesc_lo(sdO, 16), ddO_mn0 = ptx::sdesc_lo(sdO, kTile * 128);
      constexpr uint32_t ID_S = ptx::idesc_bf16(128, 128, 0, 0);    // dP
      constexpr uint32_t ID_ACC = ptx::idesc_bf16(128, 128, 1, 1);  // dV
      constexpr uint32_t BUF_STEP = L::TILE_BYTES >> 4;             // next Q / dO buffer
      Walk w(p);
      int it = 0, tile = -1;
      bool ok = true, pend = false, pend_first = false;   // task it-1's dK/dQ^T not yet issued
      bool have = w.next();
      tr.mark(X_WALK);
      while (ok) {
        // At the end of a KV tile the pending dK/dQ^T still read the old K: they go before
        // the next tile's S. Within a tile S(it) goes first.
        const bool boundary = !have || w.first_of_tile;
        if (have && !boundary)
          if (!(ok = issue_s128(bars, abort_flag, tmo, tr, tmem, dQ_k0 + (it & 1) * BUF_STEP, dK_k, it)))
            break;
        if (pend) {
          if (!(ok = issue_dk_dq128(bars, abort_flag, tmo, tr, tmem,
                                    dQ_mn0 + ((it - 1) & 1) * BUF_STEP, dPDS_mn, dK_mn, dDS_k,
                                    it - 1, pend_first)))
            break;
          if (boundary) {
            ptx::mma_commit(bars + E_ACC_FULL);
            ptx::mma_commit(bars + E_KV_EMPTY);
          }
          pend = false;
        }
        if (!have) break;
        if (boundary) {
          ++tile;
          ok = ptx::mbar_wait(bars + E_KV_FULL, tile & 1, abort_flag, tmo);
          tr.mark(X_KV_FULL);
          if (!ok) break;
          if (!(ok = issue_s128(bars, abort_flag, tmo, tr, tmem, dQ_k0 + (it & 1) * BUF_STEP, dK_k, it)))
            break;
        }
        // ---- dP(it) = dO V^T into the S/dP columns, once S(it) has been loaded
        ok = ptx::mbar_wait(bars + E_DO_FULL + (it & 1), (it >> 1) & 1, abort_flag, tmo);
        if (ok) ok = ptx::mbar_wait(bars + E_S_LOADED, it & 1, abort_flag, tmo);
        tr.mark(X_DO_S_LOADED);
        if (!ok) break;
        ptx::tc_fence_after();
        {
          const uint32_t ddO_k = ddO_k0 + (it & 1) * BUF_STEP;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            ptx::mma_lo(tmem + L::T_SP, ddO_k + kstep128(ks), dV_k + kstep128(ks), ID_S, ks > 0);
        }
        ptx::mma_commit(bars + E_DP_FULL);
        tr.mark(X_ISSUE_SDP);
        // ---- dV(it) += P^T dO, once P(it) is stored (and, for a new tile, the previous
        // tile's accumulators have been read out)
        ok = ptx::mbar_wait(bars + E_P_FULL, it & 1, abort_flag, tmo);
        tr.mark(X_P_FULL);
        if (ok && w.first_of_tile && tile > 0)
          ok = ptx::mbar_wait(bars + E_ACC_EMPTY, (tile - 1) & 1, abort_flag, tmo);
        tr.mark(X_ACC_EMPTY);
        if (!ok) break;
        ptx::tc_fence_after();
        {
          const uint32_t ddO_mn = ddO_mn0 + (it & 1) * BUF_STEP;
          const uint32_t acc0 = w.first_of_tile ? 0u : 1u;
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            ptx::mma_lo(tmem + L::T_DV, dPDS_mn + ks * kMnStep, ddO_mn + ks * kMnStep, ID_ACC,
                        ks > 0 ? 1u : acc0);
        }
        ptx::mma_commit(bars + E_DO_EMPTY + (it & 1));   // dO(it)'s last reader
        ptx::mma_commit(bars + E_P_READ);
        tr.mark(X_ISSUE_DV);
        pend = true;
        pend_first = w.first_of_tile;
        ++it;
        have = w.next();
        tr.mark(X_WALK);
      }
      tr.flush(kIssuerSites);
      // drain: no MMA may be in flight when TMEM is released
      ptx::mma_commit(bars + E_DRAIN);
      ptx::mbar_drain(bars + E_DRAIN, 0, 1000000000ll);
    }
  } else if (warp < 12) {
    // =============================== softmax-gradient warps =================================
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;         // query row within the tile
    const int col0 = half * 64;                // this thread's 64 kv columns
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const uint32_t sPDS = ptx::smem_u32(sm + L::PDS_OFF);
    SegTraceShared trs((p.trace && warp == 4 && lane == 0) ? trace_s : nullptr);
    Walk w(p);
    int it = 0;
    bool ok = true;
    while (ok && w.next()) {
      const int qb = it & 1;
      const float* ld_s = (const float*)(sm + L::LD_OFF + qb * L::LD_BYTES);
      ok = ptx::warp_wait(bars + E_Q_FULL + qb, (it >> 1) & 1, abort_flag, tmo);
      // this row's -LSE*log2e and Dsum
      const float nlse = ld_s[r], dsum = ld_s[kTile + r];
      if (ok) ok = ptx::warp_wait(bars + E_S_FULL, it & 1, abort_flag, tmo);
      trs.mark(G_S_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      float pv[64];
      ptx::tmem_ld64(tmem + lane_addr + L::T_SP + col0, pv);
      // S is in registers: dP(it) may overwrite its columns
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_S_LOADED);
      trs.mark(G_S_LOAD);
#pragma unroll
      for (int c = 0; c < 64; ++c) pv[c] = ptx::ex2(fmaf(pv[c], p.scale_log2, nlse));
      if (p.causal && w.i == w.j) {
        // diagonal tile: keys after the query are masked out
        const int lim = r - col0;              // the last visible column of this thread
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) pv[c] = 0.f;
      }
      trs.mark(G_EXP);
      // P(it) replaces dS(it-1) in the shared tile: dK(it-1) and dQ^T(it-1) must have read it
      if (it > 0) ok = ptx::warp_wait(bars + E_DS_READ, (it - 1) & 1, abort_flag, tmo);
      trs.mark(G_BUF);
      if (!ok) break;
      store_row128(sPDS, r, col0, pv);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_P_FULL);
      trs.mark(G_P_STORE);
      ok = ptx::warp_wait(bars + E_DP_FULL, it & 1, abort_flag, tmo);
      trs.mark(G_DP_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float dp[32];
        ptx::tmem_ld32(tmem + lane_addr + L::T_SP + col0 + c0, dp);
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c0 + c] *= dp[c] - dsum;
      }
      // dP is in registers: S(it+1) may overwrite its columns
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_DP_LOADED);
      trs.mark(G_DS);
      // dS(it) replaces P(it): dV(it) must have read it
      ok = ptx::warp_wait(bars + E_P_READ, it & 1, abort_flag, tmo);
      trs.mark(G_BUF);
      if (!ok) break;
      store_row128(sPDS, r, col0, pv);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_DS_FULL);
      trs.mark(G_DS_STORE);
      ++it;
    }
  } else {
    // ============== dQ read-out and reduction into the accumulator + dK/dV epilogue ===========
    ptx::regs_inc<L::REGS_READOUT>();
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;       // d column of dQ^T; kv row of dK/dV
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const Trace trq{(p.trace && warp == 12 && lane == 0) ? trace_s : nullptr};
    Walk w(p);
    int it = 0, tl = 0;
    bool ok = true;
    while (ok && w.next()) {
      const int b = w.bh / p.H, h = w.bh % p.H;
      long long t0 = trq.t0();
      ok = ptx::warp_wait(bars + E_DQ_FULL, it & 1, abort_flag, tmo);
      trq.add(K_RO_DQ_FULL, t0);
      if (!ok) break;
      ptx::tc_fence_after();
      t0 = trq.t0();
      float v[128];                            // dQ[q0 + c][row], c = 0..127
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float t[32];
        ptx::tmem_ld32(tmem + lane_addr + L::T_DQ + c0, t);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c0 + c] = t[c];
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_DQ_EMPTY);   // dQ^T(it) has left TMEM
      trq.add(K_RO_DQ_LOAD, t0);
      // The block's fixed order runs as p.chains interleaved chains: contribution o waits
      // for o - chains, in chain o % chains, adding into accumulator copy o % chains.
      const int ord = __ldg(p.ord + w.bh * p.ord_stride + w.i * p.n + w.j);
      const int chain = ord % p.chains, o = ord / p.chains;
      const int sem_idx = (w.bh * p.n + w.j) * kDqChains + chain;
      if (p.deterministic) {
        // The 128-row block's turn: lane 0 of warp 12 polls the semaphore and signals
        // E_TURN; the other read-out warps wait on it (bounded, like every wait here).
        t0 = trq.t0();
        int got = 1;
        if (warp == 12) {
          if (lane == 0) {
            got = wait_turn(p.sems + sem_idx, o + p.ordinal_skew, p.ws_header, p.timeout_ns,
                            w.bh, w.j) ? 1 : 0;
            if (got) ptx::mbar_arrive(bars + E_TURN);
            else *abort_flag = 1;
          }
          got = __shfl_sync(0xffffffffu, got, 0);
        } else {
          got = ptx::warp_wait(bars + E_TURN, it & 1, abort_flag, tmo) ? 1 : 0;
        }
        trq.add(K_RO_SEM, t0);
        if (!got) break;
      }
      t0 = trq.t0();
      float* dst = p.dq_acc + (size_t)chain * p.B * p.H * p.S * D +
                   ((size_t)w.bh * p.S + (size_t)w.j * kTile) * D + row;
#pragma unroll
      for (int c = 0; c < 128; ++c) ptx::red_add_f32(dst + (size_t)c * D, v[c]);
      if (p.deterministic) {
        // Hand the turn on once every read-out thread's adds are ordered before it: warps
        // 13..15 arrive on E_REDS (release), warp 12's lane 0 waits on it (acquire), then
        // the releasing store.
        __syncwarp();
        int done = 1;
        if (warp != 12) {
          if (lane == 0) ptx::mbar_arrive(bars + E_REDS);
        } else {
          if (lane == 0) {
            done = ptx::mbar_wait(bars + E_REDS, it & 1, abort_flag, tmo) ? 1 : 0;
            if (done)   // release store: orders every add above (this warp's via __syncwarp,
                        // the others' via E_REDS) before the new ordinal at gpu scope
              st_release_gpu(p.sems + sem_idx, o + 1 + p.ordinal_skew);
          }
          done = __shfl_sync(0xffffffffu, done, 0);
        }
        if (!done) break;
      }
      trq.add(K_RO_REDUCE, t0);
      // ---- dK/dV epilogue after the tile's last task ----
      if (w.last_of_tile) {
        t0 = trq.t0();
        ok = ptx::warp_wait(bars + E_ACC_FULL, tl & 1, abort_flag, tmo);
        trq.add(K_RO_ACC_FULL, t0);
        if (!ok) break;
        ptx::tc_fence_after();
        t0 = trq.t0();
        const size_t g = ((size_t)b * p.S + (size_t)w.i * kTile + row) * rs + (size_t)h * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float a[32];
          ptx::tmem_ld32(tmem + lane_addr + L::T_DV + c0, a);
          uint4* dst4 = (uint4*)(p.dv + g + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst4[k] = make_uint4(ptx::pack_bf16(a[8 * k], a[8 * k + 1]),
                                 ptx::pack_bf16(a[8 * k + 2], a[8 * k + 3]),
                                 ptx::pack_bf16(a[8 * k + 4], a[8 * k + 5]),
                                 ptx::pack_bf16(a[8 * k + 6], a[8 * k + 7]));
          ptx::tmem_ld32(tmem + lane_addr + L::T_DK + c0, a);
          dst4 = (uint4*)(p.dk + g + c0);
          const float sc = p.scale;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst4[k] = make_uint4(ptx::pack_bf16(sc * a[8 * k], sc * a[8 * k + 1]),
                                 ptx::pack_bf16(sc * a[8 * k + 2], sc * a[8 * k + 3]),
                                 ptx::pack_bf16(sc * a[8 * k + 4], sc * a[8 * k + 5]),
                                 ptx::pack_bf16(sc * a[8 * k + 6], sc * a[8 * k + 7]));
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + E_ACC_EMPTY);
        trq.add(K_RO_EPILOGUE, t0);
        ++tl;
      }
      ++it;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
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
