// Backward main kernel for head dimension 128: whole 128 x 128 tasks.
//
// Same persistent grid, units, schedule walk and ordered dQ reduction as the general
// kernel (kernels_tc.cuh); what differs is how one task (KV_i, Q_j) maps onto the SM:
//
//   S^T  = K Q^T        M = 128 kv, N = 128 q, K = 128 d     TMEM cols [0, 128)
//   dP^T = V dO^T       M = 128 kv, N = 128 q, K = 128 d     TMEM cols [128, 256)
//   P^T  = exp2(S^T * scale*log2e - LSE*log2e)               smem bf16 [kv][q]
//   dS^T = P^T * (dP^T - Dsum)                               smem bf16 [kv][q]
//   dV  += P^T dO                                            TMEM cols [256, 384)
//   dQ^T = K^T dS^T     M = 128 d, N = 128 q, K = 128 kv     into the dP^T columns
//   dK  += dS^T Q                                            TMEM cols [384, 512)
//
// Every MMA is 128 x 128 x 128, so the tensor pipe reads at most 8 KB of shared memory
// per 64-cycle K step. The S^T columns are handed back as soon as the softmax-gradient
// warps have loaded them, so S^T of the next task runs while P^T of this one is being
// computed. dQ^T
// reuses the dP^T columns once the softmax-gradient warps have read them, so the next
// dP^T waits for the dQ read-out: the read-out warps load all 128 columns into registers
// (their warpgroup takes registers from the single-thread roles' warpgroup), hand the
// columns back at once, and only then add the partial into the fp32 dQ accumulator with
// coalesced red.global (TMEM lane = d, so one warp instruction covers 32 consecutive d
// of one row: a full 128-byte line). In deterministic mode the adds of a 128-row block
// wait for the block's turn and the turn is handed on after they have been performed.
//
// Q is double-buffered by task parity; dO has one buffer, reloaded as soon as dP^T and dV
// have read it (the next dP^T waits for the dQ read-out anyway); P^T and dS^T have a
// buffer each, so forming dS^T never waits for dV.
//
// Shared memory (1024-aligned base, checked): K, V, Q x 2, dO, P^T, dS^T, -LSE*log2e and
// Dsum per Q buffer, barriers, trace: 231,936 bytes.
//
// Warp roles (512 threads): 0 = TMA producer, 1 = S^T/dP^T issuer, 3 = dV/dQ^T/dK issuer,
// 2 = idle, 4..11 = softmax-gradient (quarter = TMEM lanes, half = 64 q columns),
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
  static constexpr int DO_OFF = Q_OFF + 2 * TILE_BYTES;       // one dO buffer
  static constexpr int P_OFF = DO_OFF + TILE_BYTES;           // P^T [kv][q]
  static constexpr int DS_OFF = P_OFF + TILE_BYTES;           // dS^T [kv][q]
  static constexpr int LD_OFF = DS_OFF + TILE_BYTES;          // per Q buffer: -LSE*log2e, Dsum
  static constexpr int LD_BYTES = 2 * kTile * 4;
  static constexpr int BAR_OFF = LD_OFF + 2 * LD_BYTES;
  static constexpr int TRACE_OFF = BAR_OFF + 320;
  static constexpr int ALLOC = TRACE_OFF + 8 * TR_SITES;
  static_assert(ALLOC <= 232448, "shared memory budget");
  // TMEM columns
  static constexpr int T_S = 0, T_DP = 128, T_DV = 256, T_DK = 384;
  // registers per thread after the re-split (launch: 128 x 512 threads)
  static constexpr int REGS_LAUNCH = 128, REGS_SINGLE = 72, REGS_READOUT = 184;
  static_assert(REGS_SINGLE + 2 * REGS_LAUNCH + REGS_READOUT == 4 * REGS_LAUNCH,
                "the four warpgroups must share exactly the launch's registers");
};

enum {
  E_KV_FULL = 0, E_KV_EMPTY, E_Q_FULL, E_Q_EMPTY = E_Q_FULL + 2, E_DO_FULL = E_Q_EMPTY + 2,
  E_DO_EMPTY, E_S_FULL, E_S_EMPTY, E_P_FULL, E_P_EMPTY, E_DP_FULL,
  E_DS_FULL, E_DS_EMPTY, E_DQ_FULL, E_DQ_EMPTY, E_ACC_FULL, E_ACC_EMPTY, E_DRAIN, E_DRAIN2,
  E_TURN, E_REDS, E_COUNT
};
static_assert(8 * E_COUNT + 8 <= 320, "barrier area");

// Wait- and work-cycle sites of this kernel's optional trace, each counted in one of the
// shared trace slots (dash_debug_set_trace; one writer per slot).
enum : int {
  K_PROD_Q_EMPTY = TR_PROD_STAGE_EMPTY,   // producer: a Q buffer is free
  K_PROD_KV_EMPTY = TR_PROD_KV_EMPTY,     // producer: K and V are free
  K_PROD_DO_EMPTY = TR_MMA_DQ_EMPTY,      // producer: the dO buffer is free
  K_X_KV_FULL = TR_MMA_KV_FULL,           // S/dP issuer: K and V landed
  K_X_Q_FULL = TR_MMA_STAGE_FULL,         // S/dP issuer: Q landed
  K_X_S_EMPTY = TR_MMA_S_EMPTY,           // S/dP issuer: previous S^T loaded out of TMEM
  K_X_DO_DQ_EMPTY = TR_MMA_DP_EMPTY,      // S/dP issuer: dO landed, previous dQ^T read out
  K_Y_P_DO_FULL = TR_MMA_P_FULL,          // dV/dQ/dK issuer: P^T stored and dO landed
  K_Y_ACC_EMPTY = TR_MMA_ACC_EMPTY,       // dV/dQ/dK issuer: dK/dV accumulators read out
  K_Y_DP_DS_FULL = TR_MMA_DS_FULL,        // dV/dQ/dK issuer: dP^T done, dS^T stored
  K_SG_S_FULL = TR_SG_S_FULL,             // softmax-gradient: S^T ready
  K_SG_P_COMPUTE = TR_DQ_FULL,            // softmax-gradient: S^T load, exp2, P^T store
  K_SG_DP_FULL = TR_SG_DP_FULL,           // softmax-gradient: dP^T ready
  K_SG_BUF_EMPTY = TR_SG_DS_EMPTY,        // softmax-gradient: P^T or dS^T buffer free
  K_SG_DS_COMPUTE = TR_DQ_STAGE,          // softmax-gradient: dP^T load, dS^T, store
  K_RO_DQ_FULL = TR_SG_P_EMPTY,           // read-out: dQ^T ready
  K_RO_SEM = TR_DQ_SEM,                   // read-out: the block's turn (deterministic)
  K_RO_REDUCE = TR_DQ_REDUCE,             // read-out: adds and hand-off
  K_RO_ACC_FULL = TR_DQ_ACC_FULL,         // read-out: dK/dV accumulators final
  K_ISSUE_S = TR_ISSUE_S, K_ISSUE_DP = TR_ISSUE_DP, K_ISSUE_DV = TR_ISSUE_DV,
  K_ISSUE_DQDK = TR_ISSUE_DKDQ            // MMA issue time of each group
};

// 2^x on the FMA pipe, for x <= ~0 (P = 2^x with x = S*scale*log2e - LSE*log2e).
// Range reduction x = n + f with n = round(x) (adding and subtracting 1.5 * 2^23 leaves
// round-to-nearest(x) in the low mantissa bits of the sum), f in [-1/2, 1/2]; 2^f from a
// cubic fitted for minimax relative error on that interval (fit_exp2_poly.py; max relative
// error 7.5e-5, a 26th of a bf16 half-ulp); 2^n by adding n to the exponent field. x is
// clamped at -126 so the result stays a normal float. The special-function unit that
// evaluates ex2 handles 16 lanes per clock per SM, the FMA pipe 128, so evaluating a share
// of the exponentials here shortens the softmax-gradient step.
__device__ __forceinline__ float exp2_fma(float x) {
  constexpr float kRound = 12582912.0f;                  // 1.5 * 2^23
  constexpr float c0 = 0.9999281168f, c1 = 0.6932609677f, c2 = 0.2426105440f,
                  c3 = 0.0551713221f;
  x = fmaxf(x, -126.0f);
  const float t = x + kRound;
  const float f = x - (t - kRound);
  const float p = fmaf(fmaf(fmaf(c3, f, c2), f, c1), f, c0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// Columns c with (c & 3) < kFmaExpQuarters take exp2_fma, the rest the ex2 instruction.
// Measured on the full 2 x 8192 x 16 x 128 backward: 2 (half the columns) lengthened the
// P^T step from ~3100 to ~4000 cycles per task -- that step is latency-bound here, not
// limited by the special-function unit -- so this kernel keeps every exponential on ex2.
constexpr int kFmaExpQuarters = 0;

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
    }
    ptx::mbar_init(bars + E_DO_FULL, 1);
    ptx::mbar_init(bars + E_DO_EMPTY, 1);
    ptx::mbar_init(bars + E_S_FULL, 1);
    ptx::mbar_init(bars + E_S_EMPTY, 8);
    ptx::mbar_init(bars + E_P_FULL, 8);
    ptx::mbar_init(bars + E_P_EMPTY, 1);
    ptx::mbar_init(bars + E_DP_FULL, 1);
    ptx::mbar_init(bars + E_DS_FULL, 8);
    ptx::mbar_init(bars + E_DS_EMPTY, 1);
    ptx::mbar_init(bars + E_DQ_FULL, 1);
    ptx::mbar_init(bars + E_DQ_EMPTY, 4);
    ptx::mbar_init(bars + E_ACC_FULL, 1);
    ptx::mbar_init(bars + E_ACC_EMPTY, 4);
    ptx::mbar_init(bars + E_DRAIN, 1);
    ptx::mbar_init(bars + E_DRAIN2, 1);
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
  const Trace tr{p.trace ? trace_s : nullptr};
  const Trace tr_none{nullptr};

  // Warpgroup 0 runs one thread per warp and gives registers to the read-out warpgroup,
  // which holds a 128-column row. Each re-split is one instruction executed by all four
  // warps of its warpgroup, ahead of (and dominating) that warpgroup's role code.
  if (warp < 4) {
    ptx::regs_dec<L::REGS_SINGLE>();
  if (warp == 0) {
    // ===================================== TMA producer =====================================
    if (lane == 0) {
      Walk w(p);
      int it = 0, tl = 0;
      bool ok = true;
      while (ok && w.next()) {
        const int b = w.bh / p.H, h = w.bh % p.H;
        const int q0 = w.j * kTile, qb = it & 1;
        // Q_j with its -LSE*log2e and Dsum rows into Q buffer qb (free once dK of task it-2
        // is done)
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
        // K and V of a new KV tile, once the previous tile's last MMA has read them
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
        // dO_j into the dO buffer (free once dP^T and dV of task it-1 have read it)
        t0 = tr.t0();
        if (it >= 1 && !(ok = ptx::mbar_wait(bars + E_DO_EMPTY, (it - 1) & 1, abort_flag, tmo))) break;
        tr.add(K_PROD_DO_EMPTY, t0);
        ptx::mbar_expect_tx(bars + E_DO_FULL, L::TILE_BYTES);
        for (int cb = 0; cb < 2; ++cb)
          ptx::tma_load_3d(sm + L::DO_OFF + cb * kTile * 128, &maps.dO, cb * 64, h, b * p.S + q0,
                           bars + E_DO_FULL);
        ++it;
      }
      // drain: every issued load has landed before the CTA may exit
      for (int k = (it > 2 ? it - 2 : 0); k < it; ++k)
        ptx::mbar_drain(bars + E_Q_FULL + (k & 1), (k >> 1) & 1, 100000000ll);
      if (it > 0) ptx::mbar_drain(bars + E_DO_FULL, (it - 1) & 1, 100000000ll);
      if (tl > 0) ptx::mbar_drain(bars + E_KV_FULL, (tl - 1) & 1, 100000000ll);
    }
  } else if (warp == 1 || warp == 3) {
    // ===================================== MMA issuers ======================================
    if (lane == 0) {
      const uint32_t sK = ptx::smem_u32(sm + L::K_OFF), sV = ptx::smem_u32(sm + L::V_OFF);
      const uint32_t sQ = ptx::smem_u32(sm + L::Q_OFF), sdO = ptx::smem_u32(sm + L::DO_OFF);
      const uint32_t sP = ptx::smem_u32(sm + L::P_OFF), sdS = ptx::smem_u32(sm + L::DS_OFF);
      const uint32_t dK_k = ptx::sdesc_lo(sK, 16), dV_k = ptx::sdesc_lo(sV, 16);
      const uint32_t dK_mn = ptx::sdesc_lo(sK, kTile * 128);
      // P^T: K-major (over q) for dV; dS^T: K-major for dK, MN-major for dQ^T
      const uint32_t dP_k = ptx::sdesc_lo(sP, 16);
      const uint32_t dS_k = ptx::sdesc_lo(sdS, 16), dS_mn = ptx::sdesc_lo(sdS, kTile * 128);
      constexpr uint32_t ID_S = ptx::idesc_bf16(128, 128, 0, 0);    // S^T, dP^T
      constexpr uint32_t ID_ACC = ptx::idesc_bf16(128, 128, 0, 1);  // dV, dK
      constexpr uint32_t ID_DQT = ptx::idesc_bf16(128, 128, 1, 1);  // dQ^T = K^T dS^T
      constexpr uint32_t BUF_STEP = L::TILE_BYTES >> 4;             // next Q buffer
      // K-major step ks of a [128 rows][128] tile in 64-column blocks; MN-major step: 16
      // rows of 128 bytes.
      auto kstep = [](int ks) -> uint32_t { return ((ks >> 2) * kTile * 128 + (ks & 3) * 32) >> 4; };
      constexpr uint32_t MN_STEP = 2048 >> 4;
      Walk w(p);
      int it = 0, tile = -1;
      bool ok = true;
      if (warp == 1) {
        const uint32_t dQ_k0 = ptx::sdesc_lo(sQ, 16), ddO_k = ptx::sdesc_lo(sdO, 16);
        while (ok && w.next()) {
          long long t0 = tr.t0();
          if (w.first_of_tile) {
            ++tile;
            if (!(ok = ptx::mbar_wait(bars + E_KV_FULL, tile & 1, abort_flag, tmo))) break;
          }
          tr.add(K_X_KV_FULL, t0);
          t0 = tr.t0();
          ok = ptx::mbar_wait(bars + E_Q_FULL + (it & 1), (it >> 1) & 1, abort_flag, tmo);
          tr.add(K_X_Q_FULL, t0);
          t0 = tr.t0();
          // S^T overwrites the previous task's S^T: the softmax-gradient warps must have
          // loaded it
          if (ok && it > 0) ok = ptx::mbar_wait(bars + E_S_EMPTY, (it - 1) & 1, abort_flag, tmo);
          tr.add(K_X_S_EMPTY, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t dQ_k = dQ_k0 + (it & 1) * BUF_STEP;
          t0 = tr.t0();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            ptx::mma_lo(tmem + L::T_S, dK_k + kstep(ks), dQ_k + kstep(ks), ID_S, ks > 0);
          ptx::mma_commit(bars + E_S_FULL);
          tr.add(K_ISSUE_S, t0);
          t0 = tr.t0();
          ok = ptx::mbar_wait(bars + E_DO_FULL, it & 1, abort_flag, tmo);
          // dP^T overwrites the previous task's dQ^T: the read-out must have taken it
          if (ok && it > 0) ok = ptx::mbar_wait(bars + E_DQ_EMPTY, (it - 1) & 1, abort_flag, tmo);
          tr.add(K_X_DO_DQ_EMPTY, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          t0 = tr.t0();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            ptx::mma_lo(tmem + L::T_DP, dV_k + kstep(ks), ddO_k + kstep(ks), ID_S, ks > 0);
          ptx::mma_commit(bars + E_DP_FULL);
          tr.add(K_ISSUE_DP, t0);
          ++it;
        }
      } else {
        const uint32_t dQ_mn0 = ptx::sdesc_lo(sQ, kTile * 128);
        const uint32_t ddO_mn = ptx::sdesc_lo(sdO, kTile * 128);
        while (ok && w.next()) {
          if (w.first_of_tile) ++tile;
          // P^T is in shared memory, and dO of this task has landed (P_FULL does not imply
          // it: the softmax-gradient warps publish P^T before dP^T, the other reader of dO,
          // has run)
          long long t0 = tr.t0();
          ok = ptx::mbar_wait(bars + E_P_FULL, it & 1, abort_flag, tmo);
          if (ok) ok = ptx::mbar_wait(bars + E_DO_FULL, it & 1, abort_flag, tmo);
          tr.add(K_Y_P_DO_FULL, t0);
          t0 = tr.t0();
          if (ok && w.first_of_tile && tile > 0)
            ok = ptx::mbar_wait(bars + E_ACC_EMPTY, (tile - 1) & 1, abort_flag, tmo);
          tr.add(K_Y_ACC_EMPTY, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t acc0 = w.first_of_tile ? 0u : 1u;
          // dV += P^T dO: A = P^T (K-major over q), B = dO (MN-major over d)
          t0 = tr.t0();
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            ptx::mma_lo(tmem + L::T_DV, dP_k + kstep(ks), ddO_mn + ks * MN_STEP, ID_ACC,
                        ks > 0 ? 1u : acc0);
          // P^T has been read: the next P^T may overwrite it
          ptx::mma_commit(bars + E_P_EMPTY);
          tr.add(K_ISSUE_DV, t0);
          // dO's other reader, dP^T, has completed too: then the next dO may be loaded
          t0 = tr.t0();
          ok = ptx::mbar_wait(bars + E_DP_FULL, it & 1, abort_flag, tmo);
          tr.add(K_Y_DP_DS_FULL, t0);
          if (!ok) break;
          ptx::mma_commit(bars + E_DO_EMPTY);
          t0 = tr.t0();
          ok = ptx::mbar_wait(bars + E_DS_FULL, it & 1, abort_flag, tmo);
          tr.add(K_Y_DP_DS_FULL, t0);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t dQ_mn = dQ_mn0 + (it & 1) * BUF_STEP;
          t0 = tr.t0();
          // dQ^T = K^T dS^T first (its read-out gates the next dP^T): A = K^T (MN-major
          // over d), B = dS^T (MN-major over q), into the dP^T columns
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            ptx::mma_lo(tmem + L::T_DP, dK_mn + ks * MN_STEP, dS_mn + ks * MN_STEP, ID_DQT, ks > 0);
          ptx::mma_commit(bars + E_DQ_FULL);
          // dK += dS^T Q: A = dS^T (K-major over q), B = Q (MN-major over d)
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            ptx::mma_lo(tmem + L::T_DK, dS_k + kstep(ks), dQ_mn + ks * MN_STEP, ID_ACC,
                        ks > 0 ? 1u : acc0);
          ptx::mma_commit(bars + E_DS_EMPTY);
          ptx::mma_commit(bars + E_Q_EMPTY + (it & 1));
          if (w.last_of_tile) {
            ptx::mma_commit(bars + E_ACC_FULL);
            ptx::mma_commit(bars + E_KV_EMPTY);
          }
          tr.add(K_ISSUE_DQDK, t0);
          ++it;
        }
      }
      // drain: no MMA may be in flight when TMEM is released
      uint64_t* drain = bars + (warp == 1 ? E_DRAIN : E_DRAIN2);
      ptx::mma_commit(drain);
      ptx::mbar_drain(drain, 0, 1000000000ll);
    }
  }
  } else if (warp >= 4 && warp < 12) {
    // =============================== softmax-gradient warps =================================
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;         // kv row within the tile
    const int col0 = half * 64;                // this thread's 64 q columns
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const uint32_t sP = ptx::smem_u32(sm + L::P_OFF), sdS = ptx::smem_u32(sm + L::DS_OFF);
    const Trace& trs = (warp == 4 && lane == 0) ? tr : tr_none;
    // writes 64 values of row r (q columns col0..col0+63) as bf16 into a [kv][q] tile
    auto store_row = [&](uint32_t base, const float (&v)[64]) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        ptx::st_shared_v4(base + sw_chunk(r, (col0 >> 3) + k, kTile),
                          ptx::pack_bf16(v[8 * k], v[8 * k + 1]), ptx::pack_bf16(v[8 * k + 2], v[8 * k + 3]),
                          ptx::pack_bf16(v[8 * k + 4], v[8 * k + 5]), ptx::pack_bf16(v[8 * k + 6], v[8 * k + 7]));
      ptx::fence_proxy_async_smem();
    };
    Walk w(p);
    int it = 0;
    bool ok = true;
    while (ok && w.next()) {
      const int qb = it & 1;
      const float* nlse_s = (const float*)(sm + L::LD_OFF + qb * L::LD_BYTES);   // -LSE*log2e
      const float* dsum_s = nlse_s + kTile;
      long long t0 = trs.t0();
      ok = ptx::warp_wait(bars + E_Q_FULL + qb, (it >> 1) & 1, abort_flag, tmo);
      if (ok) ok = ptx::warp_wait(bars + E_S_FULL, it & 1, abort_flag, tmo);
      trs.add(K_SG_S_FULL, t0);
      if (!ok) break;
      ptx::tc_fence_after();
      long long tp = trs.t0();
      float pv[64];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float sv[32];
        ptx::tmem_ld32(tmem + lane_addr + L::T_S + col0 + c0, sv);
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c0 + c] = sv[c];
      }
      // S^T is in registers: the next task's S^T may be issued
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_S_EMPTY);
      const float4* nl4 = reinterpret_cast<const float4*>(nlse_s + col0);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 nl = nl4[c4];
        const float x[4] = {fmaf(pv[4 * c4 + 0], p.scale_log2, nl.x),
                            fmaf(pv[4 * c4 + 1], p.scale_log2, nl.y),
                            fmaf(pv[4 * c4 + 2], p.scale_log2, nl.z),
                            fmaf(pv[4 * c4 + 3], p.scale_log2, nl.w)};
#pragma unroll
        for (int k = 0; k < 4; ++k) pv[4 * c4 + k] = k < kFmaExpQuarters ? exp2_fma(x[k]) : ptx::ex2(x[k]);
      }
      if (p.causal && w.i == w.j) {
        // diagonal tile: keys after the query are masked out
        const int d = r - col0;                // kv_row - q_col offset of column 0
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (d > c) pv[c] = 0.f;
      }
      // P^T replaces the previous task's: dV must have read it
      trs.add(K_SG_P_COMPUTE, tp); 
      t0 = trs.t0();
      if (it > 0) ok = ptx::warp_wait(bars + E_P_EMPTY, (it - 1) & 1, abort_flag, tmo);
      trs.add(K_SG_BUF_EMPTY, t0);
      if (!ok) break;
      tp = trs.t0();
      store_row(sP, pv);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_P_FULL);
      trs.add(K_SG_P_COMPUTE, tp); 
      t0 = trs.t0();
      ok = ptx::warp_wait(bars + E_DP_FULL, it & 1, abort_flag, tmo);
      trs.add(K_SG_DP_FULL, t0);
      if (!ok) break;
      ptx::tc_fence_after();
      tp = trs.t0();
      const float4* ds4 = reinterpret_cast<const float4*>(dsum_s + col0);
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float dp[32];
        ptx::tmem_ld32(tmem + lane_addr + L::T_DP + c0 + col0, dp);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 ds = ds4[(c0 >> 2) + c4];
          float* pc = pv + c0 + 4 * c4;
          pc[0] *= dp[4 * c4 + 0] - ds.x;
          pc[1] *= dp[4 * c4 + 1] - ds.y;
          pc[2] *= dp[4 * c4 + 2] - ds.z;
          pc[3] *= dp[4 * c4 + 3] - ds.w;
        }
      }
      // dS^T replaces the previous task's: dQ^T and dK must have read it
      trs.add(K_SG_DS_COMPUTE, tp);
      t0 = trs.t0();
      if (it > 0) ok = ptx::warp_wait(bars + E_DS_EMPTY, (it - 1) & 1, abort_flag, tmo);
      trs.add(K_SG_BUF_EMPTY, t0);
      if (!ok) break;
      tp = trs.t0();
      store_row(sdS, pv);
      // the dP^T loads above have completed: dQ^T may now overwrite those columns
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_DS_FULL);
      trs.add(K_SG_DS_COMPUTE, tp);
      ++it;
    }
  } else {
    // ============== dQ read-out and reduction into the accumulator + dK/dV epilogue ===========
    ptx::regs_inc<L::REGS_READOUT>();
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;       // d column of dQ^T; kv row of dK/dV
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const Trace& trq = (warp == 12 && lane == 0) ? tr : tr_none;
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
      float v[128];                            // dQ[q0 + c][row], c = 0..127
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float t[32];
        ptx::tmem_ld32(tmem + lane_addr + L::T_DP + c0, t);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c0 + c] = t[c];
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_DQ_EMPTY);   // dQ^T(it) has left TMEM
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
