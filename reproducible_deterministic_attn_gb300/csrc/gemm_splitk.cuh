// Split-K GEMM with the same ordered cross-SM reduction as the attention backward's dQ:
// C (fp32, [M, N]) += A B^T for bf16 A [M, K] and B [N, K] (both K-major), the K extent cut
// into `splits` chunks. The pages list split-K GEMMs among the kernels the reduction-order
// principle applies to (Pith review, "Where Pith is reading between the lines"); the task
// grid is (output tile, K chunk) and each output tile is one reduction chain.
//
// A unit is one (TM x 128 output tile, K chunk), TM = 256 rows of C when M allows it, else
// 128; units are dealt tile-major, round robin, to a persistent grid (cooperative launch in
// deterministic mode), so a tile's chunks run side by side on neighbouring SMs. Tiles are
// numbered in groups of 8 m-tiles (gemm_tile_mn), so that concurrent units share their A
// and B panels in L2. Per unit:
//   C^T tile partial = B_tile A_tile^T    M = 128 (n), N = TM (m), K = chunk   -> TMEM
// (TMEM lane = n, so one warp's red.global covers 32 consecutive n of one row of C: a full
// 128-byte line). The MMA is TM columns wide: at TM = 256 it runs at the tensor core's full
// rate, at 128 at half of it (an instruction costs the same issue slot either way).
// Deterministic mode adds the partials of a tile in ascending chunk order
// (the dealing order, so the waits cannot form a cycle): the tile's semaphore counts the
// read-out warps that have finished adding; chunk s's warps add once it reaches 4 s and
// each adds 1 with release semantics after its adds. Non-deterministic mode adds as soon as
// the partial is ready.
//
// Warp roles (256 threads): 0 = TMA producer (A and B tiles of 64 K-columns, 4 stages), 1 =
// MMA issuer, 2..3 idle, 4..7 = read-out and reduction (64 columns of the accumulator at a
// time). TMEM: two TM-column accumulators, so the next unit's MMAs run while this one is
// read out.
#pragma once

#include "tc_shared.cuh"

namespace dash {
namespace tc {

struct GemmParams {
  float* c;                 // [M, N] fp32, accumulated into (zeroed before the launch)
  int* sems;                // [M/128 * N/128] zeroed before the launch (deterministic mode)
  int* status;              // workspace header: 0 = ok, kStatusSyncTimeout on a timed-out wait
  int M, N, K, splits, kchunk;
  int deterministic;
  long long timeout_ns;
};

struct GemmMaps {
  CUtensorMap a, b;         // 2-D bf16 [rows][K], boxes {64, TM} (a) and {64, 128} (b), 128-byte swizzle
};

constexpr int kGemmThreads = 256;
constexpr int kGemmStages = 4;

template <int TM>
struct GemmL {
  static constexpr int TILE_A = TM * 64 * 2;                 // TM rows x 64 K bf16
  static constexpr int TILE_B = 128 * 64 * 2;                // 128 rows x 64 K bf16 = 16 KB
  static constexpr int STAGE = TILE_A + TILE_B;
  static constexpr int BAR_OFF = kGemmStages * STAGE;
  static constexpr int ALLOC = BAR_OFF + 256 + 1024;
  static constexpr int TMEM_COLS = 2 * TM;                   // two accumulators
  static_assert(ALLOC <= 232448, "shared memory budget");
};

enum { G_FULL = 0, G_EMPTY = G_FULL + kGemmStages, G_ACC_FULL = G_EMPTY + kGemmStages,
       G_ACC_EMPTY = G_ACC_FULL + 2, G_DRAIN = G_ACC_EMPTY + 2, G_COUNT };

// Output tile `tile` -> its (m, n) tile indices, in groups of kGemmGroupM m-tiles: within a
// group consecutive tiles step through the group's m-tiles first, then n. The grid's
// concurrent units then share a few A and B panels (8 A + 19 B at one chunk per tile on
// 152 CTAs) that stay in L2, instead of sweeping all of B for each row of A. A bijection
// onto [0, tiles_m) x [0, tiles_n); a tile's arithmetic and reduction order do not depend
// on it.
constexpr int kGemmGroupM = 8;
__device__ __forceinline__ void gemm_tile_mn(int tile, int tiles_m, int tiles_n, int& mi, int& ni) {
  const int per_group = kGemmGroupM * tiles_n;
  const int first_m = (tile / per_group) * kGemmGroupM;
  const int gm = min(kGemmGroupM, tiles_m - first_m);
  const int r = tile % per_group;
  mi = first_m + r % gm;
  ni = r / gm;
}

template <int TM>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_splitk_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ GemmMaps maps) {
  using L = GemmL<TM>;
  extern __shared__ uint8_t smem_gemm[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_gemm + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR_OFF);
  uint32_t* tmem_slot = (uint32_t*)(sm + L::BAR_OFF + 8 * G_COUNT);
  volatile int* abort_flag = (volatile int*)(sm + L::BAR_OFF + 8 * G_COUNT + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tmo = p.timeout_ns;
  const int tiles_n = p.N / 128;
  const int units = (p.M / TM) * tiles_n * p.splits;
  const int ksteps = p.kchunk / 64;                        // 64-column K blocks per unit

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      ptx::mbar_init(bars + G_FULL + s, 1);
      ptx::mbar_init(bars + G_EMPTY + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bars + G_ACC_FULL + a, 1);
      ptx::mbar_init(bars + G_ACC_EMPTY + a, 4);
    }
    ptx::mbar_init(bars + G_DRAIN, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, L::TMEM_COLS);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ===================================== TMA producer =====================================
    if (lane == 0) {
      long long kb = 0;                                     // K blocks issued so far
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const int tile = u / p.splits, split = u % p.splits;
        int mi, ni;
        gemm_tile_mn(tile, p.M / TM, tiles_n, mi, ni);
        const int m0 = mi * TM, n0 = ni * 128;
        for (int k = 0; k < ksteps; ++k, ++kb) {
          const int s = (int)(kb % kGemmStages);
          if (kb >= kGemmStages &&
              !(ok = ptx::mbar_wait(bars + G_EMPTY + s, (int)((kb / kGemmStages) - 1) & 1, abort_flag, tmo)))
            break;
          const int kx = split * p.kchunk + k * 64;
          ptx::mbar_expect_tx(bars + G_FULL + s, L::STAGE);
          ptx::tma_load_2d(sm + s * L::STAGE, &maps.a, kx, m0, bars + G_FULL + s);
          ptx::tma_load_2d(sm + s * L::STAGE + L::TILE_A, &maps.b, kx, n0, bars + G_FULL + s);
        }
      }
      for (long long k = (kb > kGemmStages ? kb - kGemmStages : 0); k < kb; ++k)
        ptx::mbar_drain(bars + G_FULL + (int)(k % kGemmStages), (int)(k / kGemmStages) & 1, 100000000ll);
    }
  } else if (warp == 1) {
    // ====================================== MMA issuer ======================================
    if (lane == 0) {
      constexpr uint32_t ID = ptx::idesc_bf16(128, TM, 0, 0);    // both K-major
      const uint32_t s0 = ptx::smem_u32(sm);
      long long kb = 0;
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++it) {
        const int acc = it & 1;
        // the read-out must have taken this accumulator's previous unit
        if (it >= 2 && !(ok = ptx::mbar_wait(bars + G_ACC_EMPTY + acc, ((it >> 1) - 1) & 1, abort_flag, tmo)))
          break;
        ptx::tc_fence_after();
        for (int k = 0; k < ksteps; ++k, ++kb) {
          const int s = (int)(kb % kGemmStages);
          if (!(ok = ptx::mbar_wait(bars + G_FULL + s, (int)(kb / kGemmStages) & 1, abort_flag, tmo))) break;
          ptx::tc_fence_after();
          // C^T partial: A operand = B tile (rows n), B operand = A tile (rows m)
          const uint32_t b_lo = ptx::sdesc_lo(s0 + s * L::STAGE + L::TILE_A, 16);
          const uint32_t a_lo = ptx::sdesc_lo(s0 + s * L::STAGE, 16);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            ptx::mma_lo(tmem + acc * TM, b_lo + ks * 2, a_lo + ks * 2, ID, (k > 0 || ks > 0) ? 1u : 0u);
          ptx::mma_commit(bars + G_EMPTY + s);
        }
        if (!ok) break;
        ptx::mma_commit(bars + G_ACC_FULL + acc);
      }
      ptx::mma_commit(bars + G_DRAIN);
      ptx::mbar_drain(bars + G_DRAIN, 0, 1000000000ll);
    }
  } else if (warp >= 4) {
    // ================================ read-out and reduction ================================
    const int quarter = warp & 3;
    const int nr = quarter * 32 + lane;                     // n within the tile = TMEM lane
    const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++it) {
      const int acc = it & 1;
      const int tile = u / p.splits, split = u % p.splits;
      int mi, ni;
      gemm_tile_mn(tile, p.M / TM, tiles_n, mi, ni);
      const int m0 = mi * TM, n0 = ni * 128;
      ok = ptx::warp_wait(bars + G_ACC_FULL + acc, (it >> 1) & 1, abort_flag, tmo);
      if (!ok) break;
      ptx::tc_fence_after();
      if (p.deterministic) {
        // The tile's semaphore counts finished read-out warps: chunk `split` may add once
        // all four warps of every earlier chunk have (count >= 4 * split); it cannot be
        // overtaken, since chunk split + 1 needs 4 * (split + 1).
        int got = 1;
        if (lane == 0) {
          got = wait_at_least(p.sems + tile, 4 * split, p.status, tmo, tile, split) ? 1 : 0;
          if (!got) *abort_flag = 1;
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) break;
      }
      // 64 columns (rows m of C) at a time: load them, then add them
      float* dst = p.c + (size_t)m0 * p.N + n0 + nr;
#pragma unroll 1
      for (int c0 = 0; c0 < TM; c0 += 64) {
        float v0[32], v1[32];                                // C[m0 + c0 + c][n0 + nr]
        ptx::tmem_ld32(tmem + lane_addr + acc * TM + c0, v0);
        ptx::tmem_ld32(tmem + lane_addr + acc * TM + c0 + 32, v1);
#pragma unroll
        for (int c = 0; c < 32; ++c) ptx::red_add_f32(dst + (size_t)(c0 + c) * p.N, v0[c]);
#pragma unroll
        for (int c = 0; c < 32; ++c) ptx::red_add_f32(dst + (size_t)(c0 + 32 + c) * p.N, v1[c]);
      }
      // the accumulator has been read: the MMA may reuse it
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + G_ACC_EMPTY + acc);
      if (p.deterministic) {
        // each warp adds 1 after its adds: the tile's semaphore reads 4 * (split + 1) once
        // all four warps of this unit are done, which is the next chunk's turn
        __syncwarp();
        if (lane == 0) red_release_add_gpu(p.sems + tile, 1);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(p.status, 0, kStatusSyncTimeout);
}

}  // namespace tc
}  // namespace dash
