// Backward main kernel (head dimension 64 or 128): whole 128 x 128 tasks with the KV rows
// in the TMEM lanes.
//
// One persistent CTA per SM. A unit is one schedule chain (slot) of one (batch, head); CTA
// c runs units c, c + grid, ... Each schedule task (KV_i, Q_j) covers a 128 x 128 tile of
// the score matrix; KV_i's K and V stay in shared memory for all its tasks and its dK/dV
// accumulate in TMEM (DASH keeps a KV tile's dK/dV on one SM). One task maps onto the SM
// as (shown for D = 128):
//
//   S''^T  = K Q^T - LSE/scale  M = 128 kv, N = 128 q, K = 128 d + 16   TMEM cols [0, 128)
//   P^T    = exp2(S''^T * scale*log2e)                 bf16, TMEM, over S''^T's columns
//   dP''^T = V dO^T - Dsum      M = 128 kv, N = 128 q, K = 128 d + 16   TMEM cols [128, 256)
//   dS^T   = P^T * dP''^T                              bf16, TMEM over S''^T, and smem [kv][q]
//   dV    += P^T dO             M = 128 kv, N = 128 d, K = 128 q, A from TMEM  [256, 384)
//   dK    += dS^T Q             M = 128 kv, N = 128 d, K = 128 q, A from TMEM  [384, 512)
//   dQ^T   = K^T dS^T           M = 128 d,  N = 128 q, K = 128 kv       TMEM cols [128, 256)
//
// At D = 64 the score products take 4 + 1 K steps and dV and dK are 64 wide (TMEM [256, 320)
// and [320, 384)). dQ^T stays an M = 128 product: K^T is padded with a zero block to 128
// rows, so the partial lands with d in TMEM lanes 0..63 and is added in whole 128-byte
// lines like at D = 128 (by read-out warps 12 and 13).
//
// The per-query offsets -LSE/scale and -Dsum enter the two score products as one extra
// K step of 16: the A side holds ones in K columns 0..2 (a constant block), the B side the
// offset split into three bf16 terms hi + mid + lo (exact to ~2^-24 of the offset; the
// preprocess kernel writes these blocks). The softmax-gradient threads therefore need no
// per-column data at all: P = exp2(S'' * scale*log2e), dS = P * dP''.
//
// P^T and dS^T stay in TMEM as the A operand of dV and dK (the MMA reads A from TMEM, so
// those products leave the shared-memory data path to the other traffic); dS^T is also
// stored to shared memory as the B operand of dQ^T. Each softmax-gradient thread owns one
// kv row and 64 query columns (half h: columns [64h, 64h + 64)); it writes its P^T into
// packed bf16 columns [64h, 64h + 32) and its dS^T into [64h + 32, 64h + 64), columns of
// S''^T it has already loaded.
//
// One thread issues, per task t: S(t), dP(t), dV(t), dK(t), dQ^T(t). S(t+1) waits for
// dK(t) to have completed (it overwrites P^T and dS^T), which the dQ^T(t) products cover;
// dP(t+1) waits for the read-out to have taken dQ^T(t) out of the columns the two share;
// dQ^T(t) waits for dS^T(t), stored after dP(t) was loaded. Q is double-buffered by task
// parity (its last reader dK(t) runs after S(t+1) has been waited for), dO single-buffered
// (its last reader is dV(t); dP(t+1) is three products later).
//
// The dQ^T columns are read into registers by the read-out warpgroup and handed back at
// once; the partial is then added into the fp32 dQ accumulator with coalesced red.global
// (TMEM lane = d, so one warp instruction covers 32 consecutive d of one row: a full
// 128-byte line). In deterministic mode the adds of a 128-row block wait for the block's
// turn and the turn is handed on after they have been performed.
//
// Shared memory (1024-aligned base, checked): K, V, Q x 2, dO, dS^T, the offset blocks of
// Q x 2 and dO, the ones block, barriers, trace (213.6 KB at D = 128, 131 KB at D = 64).
//
// Warp roles (512 threads): 0 = TMA producer, 1 = MMA issuer, 2 = dQ hand-off
// (deterministic mode), 3 = idle,
// 4..11 = softmax-gradient (quarter = TMEM lanes = kv rows, half = 64 query columns),
// 12..15 = dQ read-out and reduction, and the dK/dV epilogue.
#pragma once

#include "tc_shared.cuh"

namespace dash {
namespace tc {

template <int D_>
struct LTc {
  static constexpr int D = D_;
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  static constexpr int TILE_BYTES = kTile * D * 2;            // one 128-row bf16 tile of Q/K/V/dO
  static constexpr int DS_BYTES = kTile * kTile * 2;          // dS^T [kv][q]
  static constexpr int EXT_BYTES = kTile * 16 * 2;            // 128 rows x 16 bf16, no swizzle
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE_BYTES;
  static constexpr int NQ = D == 64 ? 3 : 2;                  // Q buffers (task t: t % NQ)
  static constexpr int Q_OFF = V_OFF + TILE_BYTES;
  static constexpr int DO_OFF = Q_OFF + NQ * TILE_BYTES;      // one dO buffer
  static constexpr int DS_OFF = DO_OFF + TILE_BYTES;          // dS^T [kv][q]
  static constexpr int QX_OFF = DS_OFF + DS_BYTES;            // the Q buffers' offset blocks
  static constexpr int DOX_OFF = QX_OFF + NQ * EXT_BYTES;     // dO offset block
  static constexpr int ONES_OFF = DOX_OFF + EXT_BYTES;        // ones in K columns 0..2
  // D = 64: a zero block after which K^T is padded to 128 rows, so that dQ^T = K^T dS^T
  // can be an M = 128 product (its rows 64..127 are zero and unused)
  static constexpr int ZERO_OFF = ONES_OFF + EXT_BYTES;
  static constexpr int ZERO_BYTES = D == 64 ? TILE_BYTES : 0;
  static_assert(ZERO_OFF % 1024 == 0, "swizzled block alignment");
  static constexpr int BAR_OFF = ZERO_OFF + ZERO_BYTES;
  static constexpr int TRACE_OFF = BAR_OFF + 320;
  static constexpr int ALLOC = TRACE_OFF + 8 * TR_SITES;
  static_assert(ALLOC <= 232448, "shared memory budget");
  // TMEM columns: S''^T (then P^T, dS^T), dP''^T (then dQ), dV, dK
  static constexpr int T_SP = 0, T_DPQ = 128, T_DV = 256, T_DK = 256 + D;
  // registers per thread after the re-split (launch: 128 x 512 threads)
  static constexpr int REGS_LAUNCH = 128, REGS_SINGLE = 88, REGS_READOUT = 168;
  static_assert(REGS_SINGLE + 2 * REGS_LAUNCH + REGS_READOUT == 4 * REGS_LAUNCH,
                "the four warpgroups must share exactly the launch's registers");
};
using L128 = LTc<128>;

enum {
  E_KV_FULL = 0, E_KV_EMPTY, E_Q_FULL, E_Q_EMPTY = E_Q_FULL + 3, E_DO_FULL = E_Q_EMPTY + 3,
  E_DO_EMPTY, E_S_FULL, E_SP_FREE, E_P_FULL, E_DP_FULL, E_DS_FULL, E_DQ_FULL,
  E_DQ_EMPTY, E_ACC_FULL, E_ACC_EMPTY, E_DRAIN, E_TURN, E_REDS, E_RELD, E_COUNT
};
static_assert(8 * E_COUNT + 8 <= 320, "barrier area");

// Wait- and work-cycle sites of this kernel's optional trace, each counted in one of the
// shared trace slots (dash_debug_set_trace; one writer per slot).
enum : int {
  K_PROD_Q_EMPTY = TR_PROD_STAGE_EMPTY,   // producer: a Q buffer is free
  K_PROD_KV_EMPTY = TR_PROD_KV_EMPTY,     // producer: K and V are free
  K_PROD_DO_EMPTY = TR_MMA_DQ_EMPTY,      // producer: the dO buffer is free
  K_X_KV_FULL = TR_MMA_KV_FULL,           // issuer: K and V landed
  K_X_Q_FULL = TR_MMA_STAGE_FULL,         // issuer: Q landed
  K_X_SP_FREE = TR_MMA_S_EMPTY,           // issuer: dK(t-1) done, S's columns free
  K_X_DO_FULL = TR_MMA_DP_EMPTY,          // issuer: dO landed
  K_X_P_FULL = TR_MMA_P_FULL,             // issuer: P^T in TMEM
  K_X_ACC_EMPTY = TR_MMA_ACC_EMPTY,       // issuer: dK/dV accumulators read out
  K_X_DS_FULL = TR_MMA_DS_FULL,           // issuer: dS^T in TMEM and shared memory
  K_X_DQ_EMPTY = TR_SG_DS_EMPTY,          // issuer: previous dQ^T read out
  K_SG_S_FULL = TR_SG_S_FULL,             // softmax-gradient: S''^T ready
  K_SG_P_COMPUTE = TR_DQ_FULL,            // softmax-gradient: exp2 and P^T into TMEM
  K_SG_DP_FULL = TR_SG_DP_FULL,           // softmax-gradient: dP''^T ready
  K_SG_BUF = TR_DQ_STAGE,                 // softmax-gradient: the dS^T tile is free
  K_SG_DS_COMPUTE = TR_SG_P_EMPTY,        // softmax-gradient: dP''^T loads, dS^T stores
  K_SG_S_LOAD = TR_X1,                    // softmax-gradient: S''^T out of TMEM
  K_SG_P_STORE = TR_X2,                   // softmax-gradient: P^T stores complete
  K_SG_DS_STORE = TR_X3,                  // softmax-gradient: dS^T stores complete
  K_X_WALK = TR_X0,                       // issuer: stepping the task walk
  K_RO_DQ_LOAD = TR_X4,                   // read-out: dQ^T out of TMEM
  K_RO_EPILOGUE = TR_X5,                  // read-out: dK/dV out of TMEM to global memory
  K_RO_DQ_FULL = TR_X6,                   // read-out: dQ^T ready
  K_RO_SEM = TR_DQ_SEM,                   // read-out: the block's turn (deterministic)
  K_RO_REDUCE = TR_DQ_REDUCE,             // read-out: adds and hand-off
  K_RO_ACC_FULL = TR_DQ_ACC_FULL,         // read-out: dK/dV accumulators final
  K_ISSUE_S = TR_ISSUE_S,                 // issuer: issuing S''^T
  K_ISSUE_DP = TR_ISSUE_DP,               // issuer: issuing dP''^T
  K_ISSUE_DV = TR_ISSUE_DV,               // issuer: issuing dV
  K_ISSUE_DKDQ = TR_ISSUE_DKDQ            // issuer: issuing dK and dQ^T
};

// K-major step ks of a [128 rows][128] bf16 tile in 64-column blocks, in 16-byte units;
// an MN-major step is 16 rows of 128 bytes.
// The issue loops step running descriptors: from step ks to ks + 1 a K-major operand moves
// 32 bytes, or to the next 64-column block after step 3; an MN-major operand moves 16 rows.
constexpr uint32_t kKStep = 32 >> 4, kKBlockStep = (kTile * 128 - 3 * 32) >> 4;
constexpr uint32_t kMnStep = 2048 >> 4;
template <int KS>
__device__ __forceinline__ uint32_t next_k(uint32_t d) {
  return KS == 3 ? ptx::step_add<kKBlockStep>(d) : ptx::step_add<kKStep>(d);
}
// P^T (base column 0) and dS^T (base column 32) in TMEM: step ks reads 8 packed columns at
// 64 * (ks / 4) + 8 * (ks % 4) from the base
template <int KS>
__device__ __forceinline__ uint32_t next_ts(uint32_t t) {
  return KS == 3 ? ptx::step_add<64 - 24>(t) : ptx::step_add<8>(t);
}

// The NK K steps (of 16) of one product: A and B both shared-memory descriptors (K-major or
// MN-major each), or A in TMEM (always 8 steps: K = 128 query rows).
template <bool A_MN, bool B_MN, int NK = 8>
__device__ __forceinline__ void issue_ss(uint32_t d, uint32_t a, uint32_t b, uint32_t id,
                                         uint32_t acc0) {
#pragma unroll
  for (int ks = 0; ks < NK; ++ks) {
    ptx::mma_lo(d, a, b, id, ks > 0 ? 1u : acc0);
    if (ks < NK - 1) {
      a = A_MN ? ptx::step_add<kMnStep>(a) : (ks == 3 ? next_k<3>(a) : next_k<0>(a));
      b = B_MN ? ptx::step_add<kMnStep>(b) : (ks == 3 ? next_k<3>(b) : next_k<0>(b));
    }
  }
}
// dQ^T's K steps K0 .. K1 - 1 (A and B MN-major), leaving a and b at step K1: dQ^T issued
// in two parts around another product, in the same step order as issue_ss<true, true>
template <int K0, int K1>
__device__ __forceinline__ void issue_ss_mn_part(uint32_t d, uint32_t& a, uint32_t& b, uint32_t id) {
#pragma unroll
  for (int ks = K0; ks < K1; ++ks) {
    ptx::mma_lo(d, a, b, id, ks > 0 ? 1u : 0u);
    a = ptx::step_add<kMnStep>(a);
    b = ptx::step_add<kMnStep>(b);
  }
}
__device__ __forceinline__ void issue_ts(uint32_t d, uint32_t a_tmem, uint32_t b_mn, uint32_t id,
                                         uint32_t acc0) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    ptx::mma_ts(d, a_tmem, b_mn, id, ks > 0 ? 1u : acc0);
    if (ks < 7) {
      a_tmem = ks == 3 ? next_ts<3>(a_tmem) : next_ts<0>(a_tmem);
      b_mn = ptx::step_add<kMnStep>(b_mn);
    }
  }
}

// S''^T = [K | ones] [Q | Qx]^T: the D / 16 K steps of the scores and the offset step, then
// the commit that signals it.
template <int D>
__device__ __forceinline__ void issue_s_mmas(uint32_t tmem, uint32_t dK_k, uint32_t dQ_k,
                                             uint32_t dOnes, uint32_t dQx, uint64_t* bar) {
  constexpr uint32_t ID_S = ptx::idesc_bf16(128, 128, 0, 0);
  issue_ss<false, false, D / 16>(tmem + LTc<D>::T_SP, dK_k, dQ_k, ID_S, 0u);
  ptx::mma_lo_noswz(tmem + LTc<D>::T_SP, dOnes, dQx, ID_S, 1u);
  ptx::mma_commit(bar);
}

// Slots of the MMA issuer's gap-free trace and the shared trace sites they are added to.
enum : int {
  X_WALK = 0, X_KV_FULL, X_Q_FULL, X_SP_FREE, X_ISSUE_S, X_DO_FULL, X_DQ_EMPTY, X_ISSUE_DP,
  X_P_FULL, X_ACC_EMPTY, X_ISSUE_DV, X_DS_FULL, X_ISSUE_DKDQ, X_SLOTS
};
__device__ constexpr int kIssuerSites[X_SLOTS] = {
    K_X_WALK, K_X_KV_FULL, K_X_Q_FULL, K_X_SP_FREE, K_ISSUE_S, K_X_DO_FULL, K_X_DQ_EMPTY,
    K_ISSUE_DP, K_X_P_FULL, K_X_ACC_EMPTY, K_ISSUE_DV, K_X_DS_FULL, K_ISSUE_DKDQ};
using IssuerTrace = SegTrace<X_SLOTS>;

// Sites of the softmax-gradient warps' gap-free trace (one thread: warp 4, lane 0).
enum : int {
  G_S_FULL = K_SG_S_FULL, G_S_LOAD = K_SG_S_LOAD, G_EXP = K_SG_P_COMPUTE, G_BUF = K_SG_BUF,
  G_P_STORE = K_SG_P_STORE, G_DP_FULL = K_SG_DP_FULL, G_DS = K_SG_DS_COMPUTE,
  G_DS_STORE = K_SG_DS_STORE
};

// P = exp2(S'' * scale*log2e) for 32 of a thread's 64 columns, in place.
__device__ __forceinline__ void exp_half(float (&pv)[64], int c0, float scale_log2) {
#pragma unroll
  for (int c = 0; c < 32; ++c) pv[c0 + c] = ptx::ex2(pv[c0 + c] * scale_log2);
}

// Writes 8 values of kv row r (16-byte chunk `chunk` of the row's 128 query columns) as
// bf16 into a [kv][q] tile at sTile (128-byte swizzle).
__device__ __forceinline__ void store_chunk8(uint32_t sTile, int r, int chunk, const uint32_t* u) {
  ptx::st_shared_v4(sTile + sw_chunk(r, chunk, kTile), u[0], u[1], u[2], u[3]);
}

// kTrace: compiled with the optional wait-cycle trace (launched only while a trace buffer
// is set); without it the trace code and its registers are absent. kSplit: compiled with
// the epilogue of KV tiles split over two CTAs (launched only for a dealing that splits
// one); without it the epilogue is the whole-tile one alone. kEarly (D = 128; launched for
// shift's order in two chains): S(t+1) is issued between the two halves of dQ^T(t).
template <int D, bool kTrace, bool kSplit, bool kEarly>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ TmaMaps maps) {
  using L = LTc<D>;
  extern __shared__ __align__(1024) uint8_t smem128[];
  uint8_t* sm = smem128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The layout fills most of the opt-in maximum, so there is no room to realign the base.
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
    for (int b = 0; b < L::NQ; ++b) {
      ptx::mbar_init(bars + E_Q_FULL + b, 1);
      ptx::mbar_init(bars + E_Q_EMPTY + b, 1);
    }
    ptx::mbar_init(bars + E_DO_FULL, 1);
    ptx::mbar_init(bars + E_DO_EMPTY, 1);
    ptx::mbar_init(bars + E_S_FULL, 1);
    ptx::mbar_init(bars + E_SP_FREE, 1);
    ptx::mbar_init(bars + E_P_FULL, 8);
    ptx::mbar_init(bars + E_DP_FULL, 1);
    ptx::mbar_init(bars + E_DS_FULL, 8);
    ptx::mbar_init(bars + E_DQ_FULL, 1);
    ptx::mbar_init(bars + E_DQ_EMPTY, 4);
    ptx::mbar_init(bars + E_ACC_FULL, 1);
    ptx::mbar_init(bars + E_ACC_EMPTY, 4);
    ptx::mbar_init(bars + E_DRAIN, 1);
    ptx::mbar_init(bars + E_TURN, 1);
    ptx::mbar_init(bars + E_REDS, 4);
    ptx::mbar_init(bars + E_RELD, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  // The ones block: row r, K column k < 3 is 1.0, everything else 0 (threads 0..255 write
  // one 16-byte core-matrix row each: row t / 2, K half t % 2).
  if (threadIdx.x < 2 * kTile) {
    const int row = threadIdx.x >> 1, kh = threadIdx.x & 1;
    const uint32_t one = 0x3F80u;   // bf16 1.0
    const uint4 v = kh == 0 ? make_uint4(one | (one << 16), one, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    *(uint4*)(sm + L::ONES_OFF + (row >> 3) * 256 + kh * 128 + (row & 7) * 16) = v;
  }
  for (int e = threadIdx.x; e < L::ZERO_BYTES / 16; e += blockDim.x)
    *(uint4*)(sm + L::ZERO_OFF + 16 * e) = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
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
      const Trace tr{(kTrace && p.trace) ? trace_s : nullptr};
      const uint8_t* qx = (const uint8_t*)p.qx;
      const uint8_t* dox = (const uint8_t*)p.dox;
      Walk w(p, abort_flag);
      int it = 0, tl = 0;
      bool ok = true;
      while (ok && w.next()) {
        const int b = w.bh / p.H, h = w.bh % p.H;
        const int q0 = w.j * kTile, qb = it % L::NQ;
        const size_t blk = ((size_t)w.bh * p.n + w.j) * L::EXT_BYTES;   // this Q tile's offsets
        // Q_j and its offset block into Q buffer qb (free once dK of task it-NQ has run)
        long long t0 = tr.t0();
        if (it >= L::NQ &&
            !(ok = ptx::mbar_wait(bars + E_Q_EMPTY + qb, (it / L::NQ - 1) & 1, abort_flag, tmo)))
          break;
        tr.add(K_PROD_Q_EMPTY, t0);
        ptx::mbar_expect_tx(bars + E_Q_FULL + qb, L::TILE_BYTES + L::EXT_BYTES);
        for (int cb = 0; cb < D / 64; ++cb)
          ptx::tma_load_3d(sm + L::Q_OFF + qb * L::TILE_BYTES + cb * kTile * 128, &maps.q, cb * 64,
                           h, b * p.S + q0, bars + E_Q_FULL + qb);
        ptx::bulk_load(sm + L::QX_OFF + qb * L::EXT_BYTES, qx + blk, L::EXT_BYTES, bars + E_Q_FULL + qb);
        // K and V of a new KV tile, once the previous tile's last MMAs have read them
        if (w.first_of_tile) {
          t0 = tr.t0();
          if (tl > 0 && !(ok = ptx::mbar_wait(bars + E_KV_EMPTY, (tl - 1) & 1, abort_flag, tmo))) break;
          tr.add(K_PROD_KV_EMPTY, t0);
          ptx::mbar_expect_tx(bars + E_KV_FULL, 2 * L::TILE_BYTES);
          for (int cb = 0; cb < D / 64; ++cb) {
            ptx::tma_load_3d(sm + L::K_OFF + cb * kTile * 128, &maps.k, cb * 64, h,
                             b * p.S + w.i * kTile, bars + E_KV_FULL);
            ptx::tma_load_3d(sm + L::V_OFF + cb * kTile * 128, &maps.v, cb * 64, h,
                             b * p.S + w.i * kTile, bars + E_KV_FULL);
          }
          ++tl;
        }
        // dO_j and its offset block (free once dV of task it-1 has run)
        t0 = tr.t0();
        if (it >= 1 && !(ok = ptx::mbar_wait(bars + E_DO_EMPTY, (it - 1) & 1, abort_flag, tmo)))
          break;
        tr.add(K_PROD_DO_EMPTY, t0);
        ptx::mbar_expect_tx(bars + E_DO_FULL, L::TILE_BYTES + L::EXT_BYTES);
        for (int cb = 0; cb < D / 64; ++cb)
          ptx::tma_load_3d(sm + L::DO_OFF + cb * kTile * 128, &maps.dO, cb * 64, h, b * p.S + q0,
                           bars + E_DO_FULL);
        ptx::bulk_load(sm + L::DOX_OFF, dox + blk, L::EXT_BYTES, bars + E_DO_FULL);
        ++it;
      }
      // drain: every issued load has landed before the CTA may exit
      for (int k = (it > L::NQ ? it - L::NQ : 0); k < it; ++k)
        ptx::mbar_drain(bars + E_Q_FULL + k % L::NQ, (k / L::NQ) & 1, 100000000ll);
      if (it > 0) ptx::mbar_drain(bars + E_DO_FULL, (it - 1) & 1, 100000000ll);
      if (tl > 0) ptx::mbar_drain(bars + E_KV_FULL, (tl - 1) & 1, 100000000ll);
    } else if (warp == 2 && lane == 0 && p.deterministic) {
      // ================================ dQ hand-off (deterministic) ===========================
      // Once all four read-out warps have issued task it's adds (E_REDS: their arrivals
      // release them at CTA scope, this wait acquires them), the releasing store orders
      // every one of those adds before the block's new ordinal at GPU scope; it waits for
      // them to be performed, which the read-out no longer does. E_RELD tells warp 12 the
      // hand-off is done; it grants the next turn only after that, so E_REDS never runs a
      // phase ahead of this wait.
      Walk w(p, abort_flag);
      int it = 0;
      bool ok = true;
      while (ok && w.next()) {
        if (!(ok = ptx::mbar_wait(bars + E_REDS, it & 1, abort_flag, tmo))) break;
        const int ord = __ldg(p.ord + w.bh * p.ord_stride + w.i * p.n + w.j);
#if DASH_BOUNDS_CHECKS
        if (ord < 0 || ord >= p.check_n) {
          report_bounds(p.ws_header, CHK_ORDINAL, w.bh, ord, p.check_n);
          *abort_flag = 1;
          break;
        }
#endif
        const int chain = ord % p.chains, o = ord / p.chains;
        st_release_gpu(p.sems + (w.bh * p.n + w.j) * kSemStride + chain, o + 1 + p.ordinal_skew);
        ptx::mbar_arrive(bars + E_RELD);
        ++it;
      }
    } else if (warp == 1 && lane == 0) {
      // ===================================== MMA issuer =======================================
      IssuerTrace tr((kTrace && p.trace) ? trace_s : nullptr);
      const uint32_t sK = ptx::smem_u32(sm + L::K_OFF), sV = ptx::smem_u32(sm + L::V_OFF);
      const uint32_t sQ = ptx::smem_u32(sm + L::Q_OFF), sdO = ptx::smem_u32(sm + L::DO_OFF);
      const uint32_t sDS = ptx::smem_u32(sm + L::DS_OFF);
      const uint32_t dK_k = ptx::sdesc_lo(sK, 16), dV_k = ptx::sdesc_lo(sV, 16);
      const uint32_t dK_mn = ptx::sdesc_lo(sK, kTile * 128);
      // K^T as the MN-major A operand of dQ^T (M = d): at D = 64 its second 64-row block is
      // the zero block
      const uint32_t dKt_mn = D == 128 ? dK_mn : ptx::sdesc_lo(sK, L::ZERO_OFF - L::K_OFF);
      const uint32_t dQ_k0 = ptx::sdesc_lo(sQ, 16), dQ_mn0 = ptx::sdesc_lo(sQ, kTile * 128);
      const uint32_t ddO_k = ptx::sdesc_lo(sdO, 16), ddO_mn = ptx::sdesc_lo(sdO, kTile * 128);
      // dS^T [kv][q] as the MN-major B operand of dQ^T (K = kv rows, N = q contiguous)
      const uint32_t dDS_mn = ptx::sdesc_lo(sDS, kTile * 128);
      // the offset step: ones (A) against the Q / dO offset blocks (B), no swizzle
      // (no swizzle: 8-row x 16-byte core matrices, K halves 128 bytes apart, 8-row groups
      // 256 bytes apart)
      const uint32_t dOnes = ptx::sdesc_lo(ptx::smem_u32(sm + L::ONES_OFF), 128);
      const uint32_t dQx0 = ptx::sdesc_lo(ptx::smem_u32(sm + L::QX_OFF), 128);
      const uint32_t dDOx = ptx::sdesc_lo(ptx::smem_u32(sm + L::DOX_OFF), 128);
      constexpr uint32_t ID_S = ptx::idesc_bf16(128, 128, 0, 0);    // S''^T, dP''^T
      constexpr uint32_t ID_TS = ptx::idesc_bf16(128, D, 0, 1);     // dV, dK (A in TMEM)
      // dQ^T = K^T dS^T: M = 128 (d, padded with zero rows at D = 64), N = 128 q, K = 128 kv
      constexpr uint32_t ID_DQ = ptx::idesc_bf16(128, 128, 1, 1);
      constexpr uint32_t BUF_STEP = L::TILE_BYTES >> 4;             // next Q buffer
      constexpr uint32_t XBUF_STEP = L::EXT_BYTES >> 4;             // next Q offset block
      // The walk is stepped to the next task right after dV is issued, so that its table
      // loads overlap the wait for dS; this task's tile flags are kept in locals.
      Walk w(p, abort_flag);
      int it = 0, tile = -1;
      bool ok = true;
      bool have = w.next(), s_done = false;   // s_done: S(it) was issued ahead
      tr.mark(X_WALK);
      while (ok && have) {
        const bool first = w.first_of_tile, last = w.last_of_tile;
        const int qb = it % L::NQ;
        if (first) {
          ++tile;
          ok = ptx::mbar_wait(bars + E_KV_FULL, tile & 1, abort_flag, tmo);
          tr.mark(X_KV_FULL);
          if (!ok) break;
        }
        // ---- S''^T(it) = [K | ones] [Q | Qx]^T, once Q(it) has landed and dK(it-1) has
        // released the P^T / dS^T columns (unless it was issued ahead, below)
        if (!s_done) {
          ok = ptx::mbar_wait(bars + E_Q_FULL + qb, (it / L::NQ) & 1, abort_flag, tmo);
          tr.mark(X_Q_FULL);
          if (ok && it > 0) ok = ptx::mbar_wait(bars + E_SP_FREE, (it - 1) & 1, abort_flag, tmo);
          tr.mark(X_SP_FREE);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s_mmas<D>(tmem, dK_k, dQ_k0 + qb * BUF_STEP, dOnes, dQx0 + qb * XBUF_STEP, bars + E_S_FULL);
          tr.mark(X_ISSUE_S);
        }
        // ---- dP''^T(it) = [V | ones] [dO | dOx]^T, once dO(it) has landed and the read-out
        // has taken dQ^T(it-1) out of the columns the two share
        ok = ptx::mbar_wait(bars + E_DO_FULL, it & 1, abort_flag, tmo);
        tr.mark(X_DO_FULL);
        if (ok && it > 0) ok = ptx::mbar_wait(bars + E_DQ_EMPTY, (it - 1) & 1, abort_flag, tmo);
        tr.mark(X_DQ_EMPTY);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_ss<false, false, D / 16>(tmem + L::T_DPQ, dV_k, ddO_k, ID_S, 0u);
        ptx::mma_lo_noswz(tmem + L::T_DPQ, dOnes, dDOx, ID_S, 1u);
        ptx::mma_commit(bars + E_DP_FULL);
        tr.mark(X_ISSUE_DP);
        // ---- dV += P^T dO (A = P^T from TMEM), once P^T(it) is stored and, for a new tile,
        // the previous tile's accumulators have been read out
        ok = ptx::mbar_wait(bars + E_P_FULL, it & 1, abort_flag, tmo);
        tr.mark(X_P_FULL);
        if (ok && first && tile > 0)
          ok = ptx::mbar_wait(bars + E_ACC_EMPTY, (tile - 1) & 1, abort_flag, tmo);
        tr.mark(X_ACC_EMPTY);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t acc0 = first ? 0u : 1u;
        issue_ts(tmem + L::T_DV, tmem + L::T_SP, ddO_mn, ID_TS, acc0);
        ptx::mma_commit(bars + E_DO_EMPTY);              // dO(it)'s last reader
        tr.mark(X_ISSUE_DV);
        have = w.next();
        tr.mark(X_WALK);
        // ---- dK += dS^T Q (A = dS^T from TMEM), then dQ^T = K^T dS^T, once dS^T(it) is
        // stored (which also means dP''^T(it) has left the columns dQ^T overwrites)
        ok = ptx::mbar_wait(bars + E_DS_FULL, it & 1, abort_flag, tmo);
        tr.mark(X_DS_FULL);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_ts(tmem + L::T_DK, tmem + L::T_SP + 32, dQ_mn0 + qb * BUF_STEP, ID_TS, acc0);
        ptx::mma_commit(bars + E_Q_EMPTY + qb);          // Q(it)'s last reader
        ptx::mma_commit(bars + E_SP_FREE);               // P^T and dS^T have been read
        tr.mark(X_ISSUE_DKDQ);
        // ---- S''^T(it+1) ahead of dQ^T(it) when task it+1 uses the same K, once dK(it) has
        // completed (S overwrites the dS^T it reads), so the softmax-gradient warps get it
        // earlier. D = 64: always, ahead of the whole dQ^T. D = 128: only in the kEarly
        // instance, between dQ^T's two halves, which keep the pipe busy while dK(it)
        // completes. The host picks it where it measured faster (shift's order in two
        // chains: +2 %); with unordered adds their burst then meets the earlier S load.
        s_done = (D == 64 || kEarly) && have && !w.first_of_tile;
        uint32_t dq_a = dKt_mn, dq_b = dDS_mn;
        if (D == 128 && s_done) issue_ss_mn_part<0, 4>(tmem + L::T_DPQ, dq_a, dq_b, ID_DQ);
        if (s_done) {
          const int qn = (it + 1) % L::NQ;
          ok = ptx::mbar_wait(bars + E_Q_FULL + qn, ((it + 1) / L::NQ) & 1, abort_flag, tmo);
          tr.mark(X_Q_FULL);
          if (ok) ok = ptx::mbar_wait(bars + E_SP_FREE, it & 1, abort_flag, tmo);
          tr.mark(X_SP_FREE);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s_mmas<D>(tmem, dK_k, dQ_k0 + qn * BUF_STEP, dOnes, dQx0 + qn * XBUF_STEP, bars + E_S_FULL);
          tr.mark(X_ISSUE_S);
        }
        if (D == 128 && s_done) issue_ss_mn_part<4, 8>(tmem + L::T_DPQ, dq_a, dq_b, ID_DQ);
        else issue_ss<true, true>(tmem + L::T_DPQ, dKt_mn, dDS_mn, ID_DQ, 0u);
        ptx::mma_commit(bars + E_DQ_FULL);
        if (last) {
          ptx::mma_commit(bars + E_ACC_FULL);
          ptx::mma_commit(bars + E_KV_EMPTY);
        }
        tr.mark(X_ISSUE_DKDQ);
        ++it;
      }
      tr.flush(kIssuerSites);
      // drain: no MMA may be in flight when TMEM is released
      ptx::mma_commit(bars + E_DRAIN);
      ptx::mbar_drain(bars + E_DRAIN, 0, 1000000000ll);
    }
  } else if (warp < 12) {
    // =============================== softmax-gradient warps =================================
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const int r = quarter * 32 + lane;         // kv row within the tile (TMEM lane)
    const int col0 = half * 64;                // this thread's 64 query columns
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const uint32_t sDS = ptx::smem_u32(sm + L::DS_OFF);
    SegTraceShared trs((kTrace && p.trace && warp == 4 && lane == 0) ? trace_s : nullptr);
    Walk w(p, abort_flag);
    int it = 0;
    bool ok = true;
    while (ok && w.next()) {
      ok = ptx::warp_wait(bars + E_S_FULL, it & 1, abort_flag, tmo);
      trs.mark(G_S_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      // S''^T in two 32-column loads: the second is in flight while the first half's
      // exponentials run
      float pv[64];
      {
        uint32_t a[32], b[32];
        ptx::tmem_ld32_issue(tmem + lane_addr + L::T_SP + col0, a);
        ptx::tmem_ld32_wait(a);
        ptx::tmem_ld32_issue(tmem + lane_addr + L::T_SP + col0 + 32, b);
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c] = __uint_as_float(a[c]);
        trs.mark(G_S_LOAD);
        exp_half(pv, 0, p.scale_log2);
        ptx::tmem_ld32_wait(b);
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[32 + c] = __uint_as_float(b[c]);
        exp_half(pv, 32, p.scale_log2);
      }
      // P^T, 16 columns at a time into packed bf16 TMEM columns [col0, col0 + 32). Diagonal
      // tile: query c is visible to key r iff c >= r.
      const bool diag = p.causal && w.i == w.j;
      const int lim = r - col0;                // first visible column of this thread
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t u[8];
        if (diag) {
#pragma unroll
          for (int c = 16 * g; c < 16 * g + 16; ++c)
            if (c < lim) pv[c] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) u[k] = ptx::pack_bf16(pv[16 * g + 2 * k], pv[16 * g + 2 * k + 1]);
        ptx::tmem_st8(tmem + lane_addr + L::T_SP + col0 + 8 * g, u);
      }
      trs.mark(G_EXP);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + E_P_FULL);
      trs.mark(G_P_STORE);
      // dP''^T(it) is complete. Its commit tracks every MMA issued before it, so dQ^T(it-1)
      // -- the last reader of the shared dS^T tile -- has completed too, and dS^T(it) may
      // replace it.
      ok = ptx::warp_wait(bars + E_DP_FULL, it & 1, abort_flag, tmo);
      trs.mark(G_DP_FULL);
      if (!ok) break;
      ptx::tc_fence_after();
      // dS^T = P^T * dP'', 16 columns per TMEM load (P^T is held in fp32 registers, so the
      // loads stay small enough not to spill); each 16 columns go to packed TMEM columns
      // [col0 + 32, col0 + 64) and to the shared [kv][q] tile
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) {
        float dp[16];
        ptx::tmem_ld16(tmem + lane_addr + L::T_DPQ + col0 + c0, dp);
        uint32_t u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          u[k] = ptx::pack_bf16(pv[c0 + 2 * k] * dp[2 * k], pv[c0 + 2 * k + 1] * dp[2 * k + 1]);
        ptx::tmem_st8(tmem + lane_addr + L::T_SP + col0 + 32 + c0 / 2, u);
        store_chunk8(sDS, r, (col0 + c0) / 8, u);
        store_chunk8(sDS, r, (col0 + c0) / 8 + 1, u + 4);
      }
      trs.mark(G_DS);
      ptx::tmem_wait_st();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
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
    const Trace trq{(kTrace && p.trace && warp == 12 && lane == 0) ? trace_s : nullptr};
    Walk w(p, abort_flag);
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
      // dQ^T: this thread's lane is d and its 128 columns the query rows. At D = 64 only
      // warps 12 and 13 hold d rows (lanes 64..127 are the zero padding).
      const bool holds_d = D == 128 || warp < 14;
      float v[128];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float t[32];
        ptx::tmem_ld32(tmem + lane_addr + L::T_DPQ + c0, t);
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
#if DASH_BOUNDS_CHECKS
      if (ord < 0 || ord >= p.check_n) {
        report_bounds(p.ws_header, CHK_ORDINAL, w.bh, ord, p.check_n);
        *abort_flag = 1;
        break;
      }
#endif
      const int chain = ord % p.chains, o = ord / p.chains;
      const int sem_idx = (w.bh * p.n + w.j) * kSemStride + chain;
      if (p.deterministic) {
        // The 128-row block's turn: lane 0 of warp 12 polls the semaphore, then waits until
        // the releasing warp has handed on the previous task's block (so that every read-out
        // warp has passed its wait for the previous turn), and signals E_TURN; the other
        // read-out warps wait on it (bounded, like every wait here). The poll's round trip
        // overlaps the previous hand-off's wait for its adds.
        t0 = trq.t0();
        int got = 1;
        if (warp == 12) {
          if (lane == 0) {
            got = wait_turn(p.sems + sem_idx, o + p.ordinal_skew, p.ws_header, p.timeout_ns,
                            w.bh, w.j) ? 1 : 0;
            if (got && it > 0) got = ptx::mbar_wait(bars + E_RELD, (it - 1) & 1, abort_flag, tmo) ? 1 : 0;
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
      if (holds_d) {
        // lane = d: one warp instruction adds 32 consecutive d of one query row (128 bytes)
        float* dst = p.dq_acc + (size_t)chain * p.B * p.H * p.S * D +
                     ((size_t)w.bh * p.S + (size_t)w.j * kTile) * D + row;
#pragma unroll
        for (int c = 0; c < 128; ++c) ptx::red_add_f32(dst + (size_t)c * D, v[c]);
      }
      if (p.deterministic) {
        // Every read-out warp arrives on E_REDS once its adds are issued (release); warp 2
        // hands the turn on (below).
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + E_REDS);
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
        // A KV tile split over two CTAs: the first half stores its fp32 partials (dK
        // unscaled) for the second, which adds them to its own before writing dK/dV.
        const int part = kSplit ? (w.tag & 3) : 0;
        float* half_acc = p.split_acc + ((size_t)(w.tag >> 2) * 2 * kTile + row) * D;
        int* half_flag = p.split_flags + (w.tag >> 2) * kSplitFlags + quarter;
        if (part == 2) {
          int got = 1;
          if (lane == 0) got = wait_at_least(half_flag, 1, p.ws_header, p.timeout_ns, w.bh, w.i) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            if (lane == 0) *abort_flag = 1;
            break;
          }
          __syncwarp();
        }
        if (part == 1) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float a[32];
            ptx::tmem_ld32(tmem + lane_addr + L::T_DK + c0, a);
            float4* dk4 = (float4*)(half_acc + c0);
#pragma unroll
            for (int k = 0; k < 8; ++k) dk4[k] = make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]);
            ptx::tmem_ld32(tmem + lane_addr + L::T_DV + c0, a);
            float4* dv4 = (float4*)(half_acc + kTile * D + c0);
#pragma unroll
            for (int k = 0; k < 8; ++k) dv4[k] = make_float4(a[4 * k], a[4 * k + 1], a[4 * k + 2], a[4 * k + 3]);
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float a[32];
            ptx::tmem_ld32(tmem + lane_addr + L::T_DV + c0, a);
            if (part == 2) {
              const float4* hv4 = (const float4*)(half_acc + kTile * D + c0);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float4 x = hv4[k];
                a[4 * k] = x.x + a[4 * k];
                a[4 * k + 1] = x.y + a[4 * k + 1];
                a[4 * k + 2] = x.z + a[4 * k + 2];
                a[4 * k + 3] = x.w + a[4 * k + 3];
              }
            }
            uint4* dst4 = (uint4*)(p.dv + g + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst4[k] = make_uint4(ptx::pack_bf16(a[8 * k], a[8 * k + 1]),
                                   ptx::pack_bf16(a[8 * k + 2], a[8 * k + 3]),
                                   ptx::pack_bf16(a[8 * k + 4], a[8 * k + 5]),
                                   ptx::pack_bf16(a[8 * k + 6], a[8 * k + 7]));
            ptx::tmem_ld32(tmem + lane_addr + L::T_DK + c0, a);
            if (part == 2) {
              const float4* hk4 = (const float4*)(half_acc + c0);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float4 x = hk4[k];
                a[4 * k] = x.x + a[4 * k];
                a[4 * k + 1] = x.y + a[4 * k + 1];
                a[4 * k + 2] = x.z + a[4 * k + 2];
                a[4 * k + 3] = x.w + a[4 * k + 3];
              }
            }
            dst4 = (uint4*)(p.dk + g + c0);
            const float sc = p.scale;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst4[k] = make_uint4(ptx::pack_bf16(sc * a[8 * k], sc * a[8 * k + 1]),
                                   ptx::pack_bf16(sc * a[8 * k + 2], sc * a[8 * k + 3]),
                                   ptx::pack_bf16(sc * a[8 * k + 4], sc * a[8 * k + 5]),
                                   ptx::pack_bf16(sc * a[8 * k + 6], sc * a[8 * k + 7]));
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(bars + E_ACC_EMPTY);
          if (part == 1) st_release_gpu(half_flag, 1);   // this quarter's partial is stored
        }
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
  if (kTrace && p.trace) {
    if (threadIdx.x == 0) trace_s[TR_TOTAL] = (unsigned long long)(clock64() - t_start);
    __syncthreads();
    if (threadIdx.x < TR_SITES) p.trace[(size_t)blockIdx.x * TR_SITES + threadIdx.x] = trace_s[threadIdx.x];
  }
}

}  // namespace tc
}  // namespace dash
