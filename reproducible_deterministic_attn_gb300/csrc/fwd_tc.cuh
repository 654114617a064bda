// Forward pass on the 5th-generation tensor cores: O = softmax(scale * Q K^T) V and the
// natural-log LSE per row, the inputs from which the backward recomputes P.
//
// One CTA per (128-row Q tile, batch * head); the longest causal rows are launched first.
// Per KV tile j (128 keys):
//   S_j = Q K_j^T        M = 128 q, N = 128 kv, K = D     TMEM cols [128 (j & 1), +128)
//   running max m, P_j = exp2(S_j * scale*log2e - m)      packed bf16 over S_j's first 64
//                                                         columns (kv 2c, 2c + 1 in col c)
//   O  += P_j V_j        M = 128 q, N = D, K = 128 kv     TMEM cols [256, 256 + D), A = P_j
//                                                         read from TMEM
// S is double-buffered, so S_{j+1} runs on the tensor pipe while the softmax warps work on
// S_j; S_{j+2} reuses the buffer once P_j V_j has read P_j from it. Each softmax thread
// reads its row's scores from TMEM twice: for the row maximum, then 64 at a time for
// P (holding all 128 in registers at once measured ~20 % slower). When a row's running max
// grows, its O row is rescaled in TMEM (after P_{j-1} V_{j-1} has landed) before P_j V_j
// accumulates onto it; rows whose max did not change are left alone. At the end O / l goes
// to global memory as bf16 and LSE = (m + log2 l) * ln 2.
//
// Warp roles (256 threads): 0 = TMA producer (Q once, K and V in two stages), 1 = MMA
// issuer, 2..3 idle, 4..7 = softmax (thread = one Q row = one TMEM lane). Every wait is
// bounded; a CTA that gives up writes NaN into its LSE rows and, when the caller passed a
// status word, records DASH_ERR_SYNC_TIMEOUT there, so the failure cannot pass unnoticed.
#pragma once

#include "tc_shared.cuh"

namespace dash {
namespace tc {

template <int D>
struct FwdL {
  static constexpr int TILE = kTile * D * 2;                  // one 128-row bf16 tile
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = Q_OFF + TILE;                 // stage s: K at +2s*TILE, V next
  static constexpr int BAR_OFF = KV_OFF + 4 * TILE;
  static constexpr int TOTAL = BAR_OFF + 256;
  static constexpr int ALLOC = TOTAL + 1024;                  // slack for 1024 alignment
  static_assert(ALLOC <= 232448, "shared memory budget");
  static constexpr int T_S = 0, T_O = 256;                     // TMEM columns
};

enum {
  F_Q_FULL = 0, F_KV_FULL, F_KV_EMPTY = F_KV_FULL + 2, F_S_FULL = F_KV_EMPTY + 2,
  F_P_FULL = F_S_FULL + 2, F_PV_DONE = F_P_FULL + 2, F_DRAIN = F_PV_DONE + 2, F_COUNT
};

constexpr int kFwdThreads = 256;

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_tc_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ TmaMaps maps) {
  using L = FwdL<D>;
  extern __shared__ uint8_t smem_fwd[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_fwd + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR_OFF);
  uint32_t* tmem_slot = (uint32_t*)(sm + L::BAR_OFF + 8 * F_COUNT);
  volatile int* abort_flag = (volatile int*)(sm + L::BAR_OFF + 8 * F_COUNT + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tmo = p.timeout_ns;   // per wait: far beyond any legitimate wait

  const int n = p.S / kTile;
  const int qt = n - 1 - (int)blockIdx.x;          // longest causal rows first
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int nt = p.causal ? qt + 1 : n;            // KV tiles this Q tile sees
  const int q0 = qt * kTile;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bars + F_Q_FULL, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bars + F_KV_FULL + s, 1);
      ptx::mbar_init(bars + F_KV_EMPTY + s, 1);
      ptx::mbar_init(bars + F_S_FULL + s, 1);
      ptx::mbar_init(bars + F_P_FULL + s, 4);
      ptx::mbar_init(bars + F_PV_DONE + s, 1);
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

  if (warp == 0) {
    // ===================================== TMA producer =====================================
    if (lane == 0) {
      ptx::mbar_expect_tx(bars + F_Q_FULL, L::TILE);
      for (int cb = 0; cb < D / 64; ++cb)
        ptx::tma_load_3d(sm + L::Q_OFF + cb * kTile * 128, &maps.q, cb * 64, h, b * p.S + q0,
                         bars + F_Q_FULL);
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
    }
  } else if (warp == 1) {
    // ====================================== MMA issuer ======================================
    if (lane == 0) {
      const uint32_t sQ = ptx::smem_u32(sm + L::Q_OFF), sKV = ptx::smem_u32(sm + L::KV_OFF);
      const uint32_t dQ_k = ptx::sdesc_lo(sQ, 16);
      constexpr uint32_t ID_S = ptx::idesc_bf16(128, 128, 0, 0);   // S = Q K^T
      constexpr uint32_t ID_O = ptx::idesc_bf16(128, D, 0, 1);     // O += P V (V MN-major)
      constexpr uint32_t TILE16 = L::TILE >> 4;
      auto kstep = [](int ks) -> uint32_t { return ((ks >> 2) * kTile * 128 + (ks & 3) * 32) >> 4; };
      constexpr uint32_t MN_STEP = 2048 >> 4;
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        if (!ptx::mbar_wait(bars + F_KV_FULL + s, (j >> 1) & 1, abort_flag, tmo)) return false;
        // the buffer's last reader: P_{j-2} V_{j-2} (which came after the softmax's reads)
        if (j >= 2 && !ptx::mbar_wait(bars + F_PV_DONE + s, ((j >> 1) - 1) & 1, abort_flag, tmo))
          return false;
        ptx::tc_fence_after();
        const uint32_t dK_k = ptx::sdesc_lo(sKV, 16) + 2 * s * TILE16;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          ptx::mma_lo(tmem + L::T_S + 128 * s, dQ_k + kstep(ks), dK_k + kstep(ks), ID_S, ks > 0);
        ptx::mma_commit(bars + F_S_FULL + s);
        return true;
      };
      bool ok = ptx::mbar_wait(bars + F_Q_FULL, 0, abort_flag, tmo) && issue_s(0);
      for (int j = 0; ok && j < nt; ++j) {
        const int s = j & 1;
        if (j + 1 < nt && !(ok = issue_s(j + 1))) break;
        if (!(ok = ptx::mbar_wait(bars + F_P_FULL + s, (j >> 1) & 1, abort_flag, tmo))) break;
        ptx::tc_fence_after();
        // O += P_j V_j: A = P_j from TMEM (16 kv = 8 packed columns per step), B = V
        // (MN-major over d)
        const uint32_t dV_mn = ptx::sdesc_lo(sKV + (2 * s + 1) * L::TILE, kTile * 128);
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          ptx::mma_ts(tmem + L::T_O, tmem + L::T_S + 128 * s + 8 * ks, dV_mn + ks * MN_STEP, ID_O,
                      (j > 0 || ks > 0) ? 1u : 0u);
        ptx::mma_commit(bars + F_PV_DONE + s);
        ptx::mma_commit(bars + F_KV_EMPTY + s);
      }
      ptx::mma_commit(bars + F_DRAIN);
      ptx::mbar_drain(bars + F_DRAIN, 0, 1000000000ll);
    }
  } else if (warp >= 4) {
    // ======================================= softmax ========================================
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // Q row within the tile = TMEM lane
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    float m = -INFINITY, l = 0.f;                     // running max (log2 units) and sum
    bool ok = true;
    for (int j = 0; ok && j < nt; ++j) {
      const int s = j & 1;
      ok = ptx::warp_wait(bars + F_S_FULL + s, (j >> 1) & 1, abort_flag, tmo);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_s = tmem + lane_addr + L::T_S + 128 * s;
      const bool diag = p.causal && j == qt;           // keys after row r are masked there
      float mx = -INFINITY;
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 32) {
        float t[32];
        ptx::tmem_ld32(t_s + c0, t);
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (!diag || c0 + c <= r) mx = fmaxf(mx, t[c]);
      }
      const float m_new = fmaxf(m, mx * p.scale_log2);
      float lt = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 64) {
        float v[64];
        {
          float t[32];
          ptx::tmem_ld32(t_s + c0, t);
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = t[c];
          ptx::tmem_ld32(t_s + c0 + 32, t);
#pragma unroll
          for (int c = 0; c < 32; ++c) v[32 + c] = t[c];
        }
        uint32_t u[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int c = c0 + 2 * k;
          float e0 = ptx::ex2(fmaf(v[2 * k], p.scale_log2, -m_new));
          float e1 = ptx::ex2(fmaf(v[2 * k + 1], p.scale_log2, -m_new));
          e0 = (!diag || c <= r) ? e0 : 0.f;
          e1 = (!diag || c + 1 <= r) ? e1 : 0.f;
          lt += e0;
          lt += e1;
          u[k] = ptx::pack_bf16(e0, e1);
        }
        ptx::tmem_st32(t_s + c0 / 2, u);
      }
      const float alpha = ptx::ex2(m - m_new);        // 0 on the first tile (m = -inf)
      l = l * alpha + lt;
      m = m_new;
      // rescale this warp's O rows when any of their maxima grew (after P_{j-1} V_{j-1})
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        ok = ptx::warp_wait(bars + F_PV_DONE + (s ^ 1), ((j - 1) >> 1) & 1, abort_flag, tmo);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          ptx::tmem_ld32(tmem + lane_addr + L::T_O + c0, o);
          uint32_t uo[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) uo[c] = __float_as_uint(o[c] * alpha);
          ptx::tmem_st32(tmem + lane_addr + L::T_O + c0, uo);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + F_P_FULL + s);
    }
    // epilogue: O / l as bf16, LSE = (m + log2 l) * ln 2
    const int last = nt - 1;
    if (ok) ok = ptx::warp_wait(bars + F_PV_DONE + (last & 1), (last >> 1) & 1, abort_flag, tmo);
    const size_t row = (size_t)b * p.S + q0 + r;
    if (ok) {
      ptx::tc_fence_after();
      const float inv = 1.f / l;
      __nv_bfloat16* dst = p.o + (row * p.H + h) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        ptx::tmem_ld32(tmem + lane_addr + L::T_O + c0, v);
        uint4* d4 = (uint4*)(dst + c0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          d4[k] = make_uint4(ptx::pack_bf16(v[8 * k] * inv, v[8 * k + 1] * inv),
                             ptx::pack_bf16(v[8 * k + 2] * inv, v[8 * k + 3] * inv),
                             ptx::pack_bf16(v[8 * k + 4] * inv, v[8 * k + 5] * inv),
                             ptx::pack_bf16(v[8 * k + 6] * inv, v[8 * k + 7] * inv));
      }
      p.lse[(size_t)bh * p.S + q0 + r] = (m + __log2f(l)) * kLn2;
    } else {
      p.lse[(size_t)bh * p.S + q0 + r] = __int_as_float(0x7fc00000);   // NaN: this tile failed
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
