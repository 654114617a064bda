// Forward pass on the 5th-generation tensor cores: O = softmax(scale * Q K^T) V and the
// natural-log LSE per row, the inputs from which the backward recomputes P.
//
// One CTA per pair of 128-row Q tiles (A and B, adjacent tiles of one batch * head); the
// pairs with the longest causal rows are launched first. Each tile has its own softmax
// warpgroup and its own TMEM, and both walk the same K/V tiles. Per KV tile j (128 keys),
// for tile x in {A, B}:
//   S_x = Q_x K_j^T       M = 128 q, N = 128 kv, K = D    TMEM cols [128 x, +128)
//   P_x = exp2(S_x * scale*log2e - m)                    packed bf16 (kv 2c, 2c + 1 in col
//                                                        c): over S_x's first 64 columns
//                                                        at D = 128, in 64 columns of its
//                                                        own at D = 64
//   O_x += P_x V_j        M = 128 q, N = D, K = 128 kv    TMEM cols [256 + D x, +D), A = P_x
//                                                        read from TMEM
// The two tiles ping-pong on the tensor pipe: while one warpgroup turns S into P, the MMAs
// of the other run. The MMA issuer polls both tiles' barriers and issues what is ready,
// each tile's P V before either S (the pipe runs MMAs in issue order, and a P V gates its
// tile's next S and the K/V stage's release). At D = 128, S_x(j+1) overwrites P_x(j) once
// P_x(j) V_j has completed; at D = 64 it only follows that P V in issue order.
// The exponent's reference m of a row moves only when the row max exceeds it by more than
// 8 in log2 units, so P <= 2^8 (lazy rescaling; O and l share the reference, so O / l and
// LSE are unchanged), and O is rescaled in TMEM only on those tiles. On the first and last
// KV tile of a Q tile a softmax thread reads its scores twice (row max, then P); on the
// others once, computing P against the current reference and the row max alongside. If
// some row's max crossed the threshold there, the issuer issues S_x(j) again and the
// softmax takes the two-pass path.
// At the end O / l goes to global memory as bf16 and LSE = (m + log2 l) * ln 2.
//
// Warp roles (384 threads): 0 = TMA producer (both Q tiles once, K and V in two stages),
// 1 = MMA issuer, 2..3 idle, 4..7 = softmax of tile A, 8..11 = softmax of tile B (thread =
// one Q row = one TMEM lane). Every wait is bounded; a CTA that gives up writes NaN into
// its LSE rows and, when the caller passed a status word, records DASH_ERR_SYNC_TIMEOUT
// there, so the failure cannot pass unnoticed.
#pragma once

#include "tc_shared.cuh"

namespace dash {
namespace tc {

template <int D>
struct FwdL {
  static constexpr int TILE = kTile * D * 2;                  // one 128-row bf16 tile
  static constexpr int Q_OFF = 0;                             // tile A, then tile B
  static constexpr int KV_OFF = Q_OFF + 2 * TILE;             // stage s: K at +2s*TILE, V next
  static constexpr int BAR_OFF = KV_OFF + 4 * TILE;
  static constexpr int TOTAL = BAR_OFF + 256;
  static constexpr int ALLOC = TOTAL + 1024;                  // slack for 1024 alignment
  static_assert(ALLOC <= 232448, "shared memory budget");
  static constexpr int T_S = 0, T_O = 256;                    // TMEM columns (+128 x, +D x)
  static_assert(T_O + 2 * D <= 512, "TMEM columns");
  // D = 64 leaves 128 columns free: P gets its own 64 packed columns per Q tile there, so
  // S_x(j+1) need not wait for P_x(j) V_j to complete. D = 128: P over S's first 64.
  static constexpr bool kSepP = T_O + 2 * D + 2 * 64 <= 512;
  static constexpr int T_P = kSepP ? T_O + 2 * D : T_S;       // + (kSepP ? 64 : 128) x
  static constexpr int P_STRIDE = kSepP ? 64 : 128;
};

// registers per thread: launched at 168 (384 threads), re-split so the two softmax
// warpgroups hold a row's scores and the producer / issuer warpgroup gives them its share
constexpr int kFwdThreads = 384;
constexpr float kFwdRescaleLog2 = 8.f;   // lazy rescale threshold (log2 units): P <= 2^8
constexpr int kFwdRegsLaunch = 168, kFwdRegsCtrl = 88, kFwdRegsSoftmax = 208;
static_assert(kFwdRegsCtrl + 2 * kFwdRegsSoftmax == 3 * kFwdRegsLaunch,
              "the three warpgroups must share exactly the launch's registers");

enum {
  F_Q_FULL = 0, F_KV_FULL, F_KV_EMPTY = F_KV_FULL + 2, F_S_FULL = F_KV_EMPTY + 2,
  F_P_FULL = F_S_FULL + 2, F_PV_DONE = F_P_FULL + 2, F_DECIDED = F_PV_DONE + 2,
  F_DRAIN = F_DECIDED + 2, F_COUNT
};

// Non-blocking test of an mbarrier phase. The issuer polls several barriers in turn, so it
// must not use try_wait, which may suspend the thread on a phase that is not yet complete
// while another barrier is already ready.
__device__ __forceinline__ bool fwd_mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(ptx::smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// The running max folded with 32 scores of a row (columns c0 .. c0 + 31 of S). kDiag: the
// causal diagonal tile, where keys after row r are left out; every other tile has no
// masked key, so its version carries no per-score test.
template <bool kDiag>
__device__ __forceinline__ float fwd_chunk_max(const uint32_t (&t)[32], int c0, int r, float mx) {
#pragma unroll
  for (int c = 0; c < 32; ++c)
    if (!kDiag || c0 + c <= r) mx = fmaxf(mx, __uint_as_float(t[c]));
  return mx;
}

// P for 32 scores of a row (columns c0 .. c0 + 31 of S): exp2(S * scale*log2e - m_new),
// on the diagonal tile (kDiag) zero where the causal mask removes the key, added into the
// row's partial sums (column c into lt4[c % 4]) and stored as 16 packed bf16 columns at
// t_p.
template <bool kDiag>
__device__ __forceinline__ void fwd_p_chunk(const uint32_t (&t)[32], int c0, int r,
                                            float scale_log2, float m_new, float (&lt4)[4],
                                            uint32_t t_p) {
  uint32_t u[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int c = c0 + 2 * k;
    float e0 = ptx::ex2(fmaf(__uint_as_float(t[2 * k]), scale_log2, -m_new));
    float e1 = ptx::ex2(fmaf(__uint_as_float(t[2 * k + 1]), scale_log2, -m_new));
    if (kDiag) {
      e0 = c <= r ? e0 : 0.f;
      e1 = c + 1 <= r ? e1 : 0.f;
    }
    lt4[(2 * k) & 3] += e0;
    lt4[(2 * k + 1) & 3] += e1;
    u[k] = ptx::pack_bf16(e0, e1);
  }
  ptx::tmem_st8(t_p, u);
  ptx::tmem_st8(t_p + 8, u + 8);
}

// P for 32 scores of a row of a tile that is neither the first nor the causal diagonal,
// against the current reference m (the same P and partial sums as fwd_p_chunk<false> with
// m_new = m), folding the scores into the row max mx as it goes.
__device__ __forceinline__ void fwd_p_chunk_spec(const uint32_t (&t)[32], float scale_log2,
                                                 float m, float (&lt4)[4], uint32_t t_p,
                                                 float& mx) {
  uint32_t u[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float s0 = __uint_as_float(t[2 * k]), s1 = __uint_as_float(t[2 * k + 1]);
    mx = fmaxf(mx, fmaxf(s0, s1));
    const float e0 = ptx::ex2(fmaf(s0, scale_log2, -m));
    const float e1 = ptx::ex2(fmaf(s1, scale_log2, -m));
    lt4[(2 * k) & 3] += e0;
    lt4[(2 * k + 1) & 3] += e1;
    u[k] = ptx::pack_bf16(e0, e1);
  }
  ptx::tmem_st8(t_p, u);
  ptx::tmem_st8(t_p + 8, u + 8);
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_tc_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ TmaMaps maps) {
  using L = FwdL<D>;
  extern __shared__ uint8_t smem_fwd[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_fwd + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR_OFF);
  uint32_t* tmem_slot = (uint32_t*)(sm + L::BAR_OFF + 8 * F_COUNT);
  volatile int* abort_flag = (volatile int*)(sm + L::BAR_OFF + 8 * F_COUNT + 4);
  // per Q tile: set by a softmax warp whose rows need the exact path on a speculative tile;
  // the issuer's decision for the tile (1 = S is issued again)
  volatile int* redo_flag = (volatile int*)(sm + L::BAR_OFF + 8 * F_COUNT + 8);
  volatile int* decision = (volatile int*)(sm + L::BAR_OFF + 8 * F_COUNT + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tmo = p.timeout_ns;   // per wait: far beyond any legitimate wait

  const int n = p.S / kTile;
  const int qa = n - 1 - 2 * (int)blockIdx.y;      // longest causal rows first
  const int qb = qa - 1;                            // tile B (absent when qa is tile 0)
  const bool has_b = qb >= 0;
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int nt_a = p.causal ? qa + 1 : n;          // KV tiles each Q tile sees
  const int nt_b = has_b ? (p.causal ? qb + 1 : n) : 0;
  const int nt = nt_a;                              // KV tiles loaded (nt_b <= nt_a)

  if (threadIdx.x == 0) {
    ptx::mbar_init(bars + F_Q_FULL, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bars + F_KV_FULL + s, 1);
      ptx::mbar_init(bars + F_KV_EMPTY + s, 1);
      ptx::mbar_init(bars + F_S_FULL + s, 1);      // per Q tile from here on
      ptx::mbar_init(bars + F_P_FULL + s, 4);
      ptx::mbar_init(bars + F_PV_DONE + s, 1);
      ptx::mbar_init(bars + F_DECIDED + s, 1);
      redo_flag[s] = 0;
    }
    ptx::mbar_init(bars + F_DRAIN, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    ptx::regs_dec<kFwdRegsCtrl>();
    if (warp == 0 && lane == 0) {
      // ===================================== TMA producer =====================================
      ptx::mbar_expect_tx(bars + F_Q_FULL, (has_b ? 2 : 1) * L::TILE);
      for (int x = 0; x < (has_b ? 2 : 1); ++x)
        for (int cb = 0; cb < D / 64; ++cb)
          ptx::tma_load_3d(sm + L::Q_OFF + x * L::TILE + cb * kTile * 128, &maps.q, cb * 64, h,
                           b * p.S + (x ? qb : qa) * kTile, bars + F_Q_FULL);
      int j = 0;
      for (; j < (p.withhold_kv ? 0 : nt); ++j) {
        const int s = j & 1;
        if (j >= 2 && !ptx::mbar_wait(bars + F_KV_EMPTY + s, ((j >> 1) - 1) & 1, abort_flag, tmo))
          break;
        uint8_t* ks = sm + L::KV_OFF + 2 * s * L::TILE;
        ptx::mbar_expect_tx(bars + F_KV_FULL + s, 2 * L::TILE);
        for (int cb = 0; cb < D / 64; ++cb) {
          ptx::tma_load_3d(ks + cb * kTile * 128, &maps.k, cb * 64, h, b * p.S + j * kTile,
                           bars + F_KV_FULL + s);
          ptx::tma_load_3d(ks + L::TILE + cb * kTile * 128, &maps.v, cb * 64, h,
                           b * p.S + j * kTile, bars + F_KV_FULL + s);
        }
      }
      // drain: every issued load has landed before the CTA may exit
      ptx::mbar_drain(bars + F_Q_FULL, 0, 100000000ll);
      for (int k = (j > 2 ? j - 2 : 0); k < j; ++k)
        ptx::mbar_drain(bars + F_KV_FULL + (k & 1), (k >> 1) & 1, 100000000ll);
    } else if (warp == 1 && lane == 0) {
      // ====================================== MMA issuer ======================================
      // Per tile x: ns[x] = next S to issue, np[x] = next P V to issue. S_x(t) needs K_t
      // landed and P_x(t-1) V_{t-1} done (S_x overwrites P_x), and follows P_x(t-1) V_{t-1}
      // in issue order; P_x(t) V_t needs P_x(t) stored. A KV stage is released once both
      // tiles have issued their P V for its tile. The loop polls and issues what is ready.
      // On a speculative tile (neither the first nor the last of its Q tile) the softmax
      // computes P against the current reference without the max pass; if a row's max
      // exceeded it by more than the threshold, the issuer issues S_x(t) again (K_t is still
      // resident: its stage is released only after both P V) instead of P_x(t) V_t, and the
      // softmax takes the exact path. Each round checks both tiles' P V before either S:
      // the tensor pipe runs MMAs in issue order, and a P V issued first completes first,
      // which is what its tile's next S and the K/V stage release wait for (measured 10 %
      // faster than checking S first).
      const uint32_t sQ = ptx::smem_u32(sm + L::Q_OFF), sKV = ptx::smem_u32(sm + L::KV_OFF);
      constexpr uint32_t ID_S = ptx::idesc_bf16(128, 128, 0, 0);   // S = Q K^T
      constexpr uint32_t ID_O = ptx::idesc_bf16(128, D, 0, 1);     // O += P V (V MN-major)
      constexpr uint32_t TILE16 = L::TILE >> 4;
      constexpr uint32_t MN_STEP = 2048 >> 4;
      int ns[2] = {0, 0}, np[2] = {0, 0};
      int pf_par[2] = {0, 0};             // P_FULL phases (a redone tile completes it twice)
      bool redone[2] = {false, false};    // S_x(np[x]) was issued again: its P is exact
      const int ntx[2] = {nt_a, nt_b};
      auto issue_s = [&](int x, int t) {
        const uint32_t dQ_k = ptx::sdesc_lo(sQ, 16) + x * TILE16;
        const uint32_t dK_k = ptx::sdesc_lo(sKV, 16) + 2 * (t & 1) * TILE16;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t step = ((ks >> 2) * kTile * 128 + (ks & 3) * 32) >> 4;
          ptx::mma_lo(tmem + L::T_S + 128 * x, dQ_k + step, dK_k + step, ID_S, ks > 0);
        }
        ptx::mma_commit(bars + F_S_FULL + x);
      };
      int kv_rel = 0;
      bool ok = ptx::mbar_wait(bars + F_Q_FULL, 0, abort_flag, tmo);
      long long t_last = global_timer_ns();
      while (ok && (np[0] < nt_a || np[1] < nt_b)) {
        bool progress = false;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int u = np[x];
          if (u < ns[x] && fwd_mbar_test(bars + F_P_FULL + x, pf_par[x])) {
            pf_par[x] ^= 1;
            ptx::tc_fence_after();
            if (u > 0 && u < ntx[x] - 1 && !redone[x]) {   // speculative P: post the decision
              const int redo = redo_flag[x];
              redo_flag[x] = 0;
              decision[x] = redo;
              ptx::mbar_arrive(bars + F_DECIDED + x);
              if (redo) {
                issue_s(x, u);
                redone[x] = true;
                progress = true;
                continue;
              }
            }
            redone[x] = false;
            // O_x += P_x V_u: A = P_x from TMEM (16 kv = 8 packed columns per step), B = V
            // (MN-major over d)
            const uint32_t dV_mn = ptx::sdesc_lo(sKV + (2 * (u & 1) + 1) * L::TILE, kTile * 128);
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
              ptx::mma_ts(tmem + L::T_O + D * x, tmem + L::T_P + L::P_STRIDE * x + 8 * ks,
                          dV_mn + ks * MN_STEP, ID_O, (u > 0 || ks > 0) ? 1u : 0u);
            ptx::mma_commit(bars + F_PV_DONE + x);
            np[x] = u + 1;
            progress = true;
          }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int t = ns[x];
          // With P in its own columns (kSepP), S_x(t) only has to follow P_x(t-1) V_{t-1} in
          // issue order (t == np[x]); its commit then also covers that P V, which the
          // softmax's next P stores need complete.
          if (t < ntx[x] && t == np[x] &&
              fwd_mbar_test(bars + F_KV_FULL + (t & 1), (t >> 1) & 1) &&
              (t == 0 || L::kSepP || fwd_mbar_test(bars + F_PV_DONE + x, (t - 1) & 1))) {
            ptx::tc_fence_after();
            issue_s(x, t);
            ns[x] = t + 1;
            progress = true;
          }
        }
        // KV stage of tile kv_rel: free once every tile that reads it has issued its P V
        while (kv_rel < nt && (np[0] > kv_rel || nt_a <= kv_rel) &&
               (np[1] > kv_rel || nt_b <= kv_rel)) {
          ptx::mma_commit(bars + F_KV_EMPTY + (kv_rel & 1));
          ++kv_rel;
        }
        if (progress) {
          t_last = global_timer_ns();
        } else if (*abort_flag) {   // idle: poll again at once (a sleep measured slower)
          ok = false;
        } else if (global_timer_ns() - t_last > tmo) {
          *abort_flag = 1;
          ok = false;
        }
      }
      ptx::mma_commit(bars + F_DRAIN);
      ptx::mbar_drain(bars + F_DRAIN, 0, 1000000000ll);
    }
  } else {
    ptx::regs_inc<kFwdRegsSoftmax>();
    // ======================================= softmax ========================================
    const int x = (warp - 4) >> 2;                   // Q tile: 0 = A, 1 = B
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;               // Q row within the tile = TMEM lane
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    const int qt = x ? qb : qa, ntt = x ? nt_b : nt_a;
    const uint32_t t_s = tmem + lane_addr + L::T_S + 128 * x;
    const uint32_t t_pp = tmem + lane_addr + L::T_P + L::P_STRIDE * x;   // P's packed columns
    const uint32_t t_o = tmem + lane_addr + L::T_O + D * x;
    float m = -INFINITY, l = 0.f;                   // running max (log2 units) and sum
    bool ok = true;
    int s_par = 0, v_par = 0;                       // S_FULL / DECIDED phases
    for (int j = 0; ok && j < ntt; ++j) {
      ok = ptx::warp_wait(bars + F_S_FULL + x, s_par, abort_flag, tmo);
      s_par ^= 1;
      if (!ok) break;
      ptx::tc_fence_after();
      if (j > 0 && j < ntt - 1) {
        // Speculative tile: P against the current reference m in one pass, the row max
        // alongside. That P is the exact path's unless some row's max exceeds m by more
        // than kFwdRescaleLog2; then this warpgroup asks for S again (the issuer's decision)
        // and takes the exact path on it.
        float mx = -INFINITY;
        float lt4[4] = {0.f, 0.f, 0.f, 0.f};
        {
          uint32_t ta[32], tb[32];
          ptx::tmem_ld32_issue(t_s, ta);
          ptx::tmem_ld32_wait(ta);
#pragma unroll
          for (int c0 = 0; c0 < kTile; c0 += 64) {
            ptx::tmem_ld32_issue(t_s + c0 + 32, tb);
            fwd_p_chunk_spec(ta, p.scale_log2, m, lt4, t_pp + c0 / 2, mx);
            ptx::tmem_ld32_wait(tb);
            if (c0 + 64 < kTile) ptx::tmem_ld32_issue(t_s + c0 + 64, ta);
            fwd_p_chunk_spec(tb, p.scale_log2, m, lt4, t_pp + (c0 + 32) / 2, mx);
            if (c0 + 64 < kTile) ptx::tmem_ld32_wait(ta);
          }
        }
        if (__any_sync(0xffffffffu, mx * p.scale_log2 > m + kFwdRescaleLog2) && lane == 0)
          redo_flag[x] = 1;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bars + F_P_FULL + x);
        ok = ptx::warp_wait(bars + F_DECIDED + x, v_par, abort_flag, tmo);
        v_par ^= 1;
        if (!ok) break;
        if (!decision[x]) {                          // P_x(j) V_j is issued; m stays
          const float lt = (lt4[0] + lt4[1]) + (lt4[2] + lt4[3]);
          l = l * 1.f + lt;
          continue;
        }
        ok = ptx::warp_wait(bars + F_S_FULL + x, s_par, abort_flag, tmo);   // S_x(j) again
        s_par ^= 1;
        if (!ok) break;
        ptx::tc_fence_after();
      }
      const bool diag = p.causal && j == qt;         // keys after row r are masked there
      // Both passes read S 32 columns at a time with the next 32 loading while the current
      // ones are used (one load in flight at a time; a wait covers every earlier load).
      // pass 1: the row maximum of the scaled scores
      float mx = -INFINITY;
      {
        uint32_t ta[32], tb[32];
        ptx::tmem_ld32_issue(t_s, ta);
        ptx::tmem_ld32_wait(ta);
#pragma unroll
        for (int c0 = 0; c0 < kTile; c0 += 64) {
          ptx::tmem_ld32_issue(t_s + c0 + 32, tb);
          mx = diag ? fwd_chunk_max<true>(ta, c0, r, mx) : fwd_chunk_max<false>(ta, c0, r, mx);
          ptx::tmem_ld32_wait(tb);
          if (c0 + 64 < kTile) ptx::tmem_ld32_issue(t_s + c0 + 64, ta);
          mx = diag ? fwd_chunk_max<true>(tb, c0 + 32, r, mx)
                    : fwd_chunk_max<false>(tb, c0 + 32, r, mx);
          if (c0 + 64 < kTile) ptx::tmem_ld32_wait(ta);
        }
      }
      // The exponent's reference m moves only when the row max exceeds it by more than
      // kFwdRescaleLog2, so P is at most 2^8: far from fp32 overflow, and bf16's relative
      // precision does not depend on magnitude. O and l share the reference, so O / l and
      // LSE = m + log2 l are the same; O is rescaled only on tiles where a row's reference
      // moves (the first, then rarely) instead of whenever a row's max grows.
      const float m_row = mx * p.scale_log2;
      const bool moved = m_row > m + kFwdRescaleLog2;
      const float m_new = moved ? m_row : m;
      // pass 2: P = exp2(S * scale*log2e - m_new), row sum, packed bf16 into P's columns
      // (D = 128: over S's first 64: columns c0 .. c0 + 31 go to packed columns c0 / 2 ..
      // c0 / 2 + 15, which lie in scores this thread has already read and not in the 32
      // loading meanwhile).
      // The row sum is four partial sums, added in a fixed order at the end.
      float lt4[4] = {0.f, 0.f, 0.f, 0.f};
      {
        uint32_t ta[32], tb[32];
        ptx::tmem_ld32_issue(t_s, ta);
        ptx::tmem_ld32_wait(ta);
#pragma unroll
        for (int c0 = 0; c0 < kTile; c0 += 64) {
          ptx::tmem_ld32_issue(t_s + c0 + 32, tb);
          if (diag) fwd_p_chunk<true>(ta, c0, r, p.scale_log2, m_new, lt4, t_pp + c0 / 2);
          else fwd_p_chunk<false>(ta, c0, r, p.scale_log2, m_new, lt4, t_pp + c0 / 2);
          ptx::tmem_ld32_wait(tb);
          if (c0 + 64 < kTile) ptx::tmem_ld32_issue(t_s + c0 + 64, ta);
          if (diag)
            fwd_p_chunk<true>(tb, c0 + 32, r, p.scale_log2, m_new, lt4, t_pp + (c0 + 32) / 2);
          else
            fwd_p_chunk<false>(tb, c0 + 32, r, p.scale_log2, m_new, lt4, t_pp + (c0 + 32) / 2);
          if (c0 + 64 < kTile) ptx::tmem_ld32_wait(ta);
        }
      }
      const float lt = (lt4[0] + lt4[1]) + (lt4[2] + lt4[3]);
      const float alpha = moved ? ptx::ex2(m - m_new) : 1.f;   // 0 on the first tile (m = -inf)
      l = l * alpha + lt;
      m = m_new;
      // rescale this warp's O rows when any of their references moved (P_x(j-1) V_{j-1} is
      // done: S_x(j) was issued after it)
      if (j > 0 && __any_sync(0xffffffffu, moved)) {
        uint32_t oa[32], ob[32];
        ptx::tmem_ld32_issue(t_o, oa);
        ptx::tmem_ld32_wait(oa);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
          ptx::tmem_ld32_issue(t_o + c0 + 32, ob);
#pragma unroll
          for (int c = 0; c < 32; ++c) oa[c] = __float_as_uint(__uint_as_float(oa[c]) * alpha);
          ptx::tmem_st32(t_o + c0, oa);
          ptx::tmem_ld32_wait(ob);
          if (c0 + 64 < D) ptx::tmem_ld32_issue(t_o + c0 + 64, oa);
#pragma unroll
          for (int c = 0; c < 32; ++c) ob[c] = __float_as_uint(__uint_as_float(ob[c]) * alpha);
          ptx::tmem_st32(t_o + c0 + 32, ob);
          if (c0 + 64 < D) ptx::tmem_ld32_wait(oa);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + F_P_FULL + x);
    }
    // epilogue: O / l as bf16, LSE = (m + log2 l) * ln 2
    if (ntt > 0) {
      const int last = ntt - 1;
      if (ok) ok = ptx::warp_wait(bars + F_PV_DONE + x, last & 1, abort_flag, tmo);
      const size_t row = (size_t)b * p.S + (size_t)qt * kTile + r;
      if (ok) {
        ptx::tc_fence_after();
        const float inv = 1.f / l;
        __nv_bfloat16* dst = p.o + (row * p.H + h) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float v[32];
          ptx::tmem_ld32(t_o + c0, v);
          uint4* d4 = (uint4*)(dst + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            d4[k] = make_uint4(ptx::pack_bf16(v[8 * k] * inv, v[8 * k + 1] * inv),
                               ptx::pack_bf16(v[8 * k + 2] * inv, v[8 * k + 3] * inv),
                               ptx::pack_bf16(v[8 * k + 4] * inv, v[8 * k + 5] * inv),
                               ptx::pack_bf16(v[8 * k + 6] * inv, v[8 * k + 7] * inv));
        }
        p.lse[(size_t)bh * p.S + (size_t)qt * kTile + r] = (m + __log2f(l)) * kLn2;
      } else {
        p.lse[(size_t)bh * p.S + (size_t)qt * kTile + r] = __int_as_float(0x7fc00000);   // NaN
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag && p.status) atomicCAS(p.status, 0, kStatusSyncTimeout);
}

}  // namespace tc
}  // namespace dash
