// First-generation kernels on the CUDA cores (fp32 FMA): forward, backward main loop
// with the ordered dQ reduction, preprocess and dQ convert. They carry the whole
// protocol of the backward (persistent grid, schedule tables, bounded semaphores) and
// serve as the correctness baseline for the tensor-core kernels.
#pragma once

#include "common.cuh"

namespace dash {

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------------------------
// Forward: one CTA per (64-row Q tile, batch*head). Online softmax over 64-key chunks.
// ---------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fwd_simt_kernel(FwdParams p) {
  constexpr int BQ = 64, BK = 64, NT = 256;
  constexpr int PER = BQ * D / NT;       // O entries per thread
  extern __shared__ float smem[];
  float* Qs = smem;                      // [BQ][D]
  float* Ks = Qs + BQ * D;               // [BK][D]
  float* Vs = Ks + BK * D;               // [BK][D]
  float* Ss = Vs + BK * D;               // [BQ][BK + 1]
  float* m_s = Ss + BQ * (BK + 1);
  float* l_s = m_s + BQ;
  float* a_s = l_s + BQ;

  const int tid = threadIdx.x;
  const int q0 = blockIdx.x * BQ;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const size_t rs = (size_t)p.H * D;                       // row stride (elements)
  const size_t base = ((size_t)b * p.S * p.H + h) * D;     // (b, 0, h, 0)

  for (int e = tid; e < BQ * D; e += NT) {
    const int r = e / D, c = e % D;
    Qs[e] = bf(p.q[base + (size_t)(q0 + r) * rs + c]);
  }
  if (tid < BQ) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  const int my_r = tid / 4;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;

  const int kv_end = p.causal ? q0 + BQ : p.S;
  for (int k0 = 0; k0 < kv_end; k0 += BK) {
    __syncthreads();
    for (int e = tid; e < BK * D; e += NT) {
      const int r = e / D, c = e % D;
      Ks[e] = bf(p.k[base + (size_t)(k0 + r) * rs + c]);
      Vs[e] = bf(p.v[base + (size_t)(k0 + r) * rs + c]);
    }
    __syncthreads();
    for (int e = tid; e < BQ * BK; e += NT) {
      const int r = e / BK, c = e % BK;
      float s = 0.f;
#pragma unroll 8
      for (int x = 0; x < D; ++x) s += Qs[r * D + x] * Ks[c * D + x];
      s *= p.scale;
      if (p.causal && k0 + c > q0 + r) s = -INFINITY;
      Ss[r * (BK + 1) + c] = s;
    }
    __syncthreads();
    if (tid < BQ) {
      const float m_old = m_s[tid];
      float mx = m_old;
      for (int c = 0; c < BK; ++c) mx = fmaxf(mx, Ss[tid * (BK + 1) + c]);
      const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - mx);
      float sum = 0.f;
      for (int c = 0; c < BK; ++c) {
        const float pv = expf(Ss[tid * (BK + 1) + c] - mx);
        Ss[tid * (BK + 1) + c] = pv;
        sum += pv;
      }
      l_s[tid] = l_s[tid] * alpha + sum;
      m_s[tid] = mx;
      a_s[tid] = alpha;
    }
    __syncthreads();
    const float alpha = a_s[my_r];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int c = (tid % 4) + 4 * k;
      float s = acc[k] * alpha;
      for (int x = 0; x < BK; ++x) s += Ss[my_r * (BK + 1) + x] * Vs[x * D + c];
      acc[k] = s;
    }
  }
  __syncthreads();
  const float inv_l = 1.f / l_s[my_r];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int c = (tid % 4) + 4 * k;
    p.o[base + (size_t)(q0 + my_r) * rs + c] = __float2bfloat16(acc[k] * inv_l);
  }
  if (tid < BQ) p.lse[(size_t)bh * p.S + q0 + tid] = m_s[tid] + logf(l_s[tid]);
}

// ---------------------------------------------------------------------------------
// Preprocess: D = rowsum(dO * O) (one warp per row, fixed shuffle tree), clear the
// semaphores and the status header, and (non-deterministic mode) the dQ accumulator.
// ---------------------------------------------------------------------------------
__global__ void bwd_preprocess_kernel(BwdParams p) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long rows = (long long)p.B * p.H * p.S;
  for (long long r = warp; r < rows; r += nwarps) {
    // r enumerates (b, h, s) so that Dsum is written contiguously
    const int s = (int)(r % p.S);
    const long long bh = r / p.S;
    const int h = (int)(bh % p.H), b = (int)(bh / p.H);
    const size_t off = (((size_t)b * p.S + s) * p.H + h) * p.D;
    float acc = 0.f;
    for (int c = lane; c < p.D; c += 32) acc += bf(p.dO[off + c]) * bf(p.o[off + c]);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (lane == 0) p.Dsum[r] = acc;
  }
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nth = (long long)gridDim.x * blockDim.x;
  const long long nsem = (long long)p.B * p.H * p.n;
  for (long long e = tid; e < nsem; e += nth) p.sems[e] = 0;
  if (tid < (long long)(kWsHeaderBytes / sizeof(int))) p.ws_header[tid] = 0;
  if (!p.deterministic) {
    const long long nacc = (long long)p.B * p.H * p.S * p.D;
    for (long long e = tid; e < nacc; e += nth) p.dq_acc[e] = 0.f;
  }
}

// dQ = bf16(scale * accumulator), for the non-deterministic path.
__global__ void dq_convert_kernel(BwdParams p) {
  const long long n = (long long)p.B * p.H * p.S * p.D;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(e % p.D);
    const long long row = e / p.D;             // (b*H + h) * S + s
    const int s = (int)(row % p.S);
    const long long bh = row / p.S;
    const int h = (int)(bh % p.H), b = (int)(bh / p.H);
    p.dq[(((size_t)b * p.S + s) * p.H + h) * p.D + c] = __float2bfloat16(p.scale * p.dq_acc[e]);
  }
}

// ---------------------------------------------------------------------------------
// Backward main loop, persistent: CTA c runs units c, c + grid, ... ; a unit is one
// chain (schedule slot) of one (batch, head). For each task (KV_i, Q_j) it computes
// P, dS and the dK/dV updates in 32-row Q sub-tiles, collects the 128-row dQ_j partial
// in shared memory, then adds it into dQ_j: in the schedule's order (deterministic) or
// with atomics. The last contributor of a block writes the bf16 dQ directly.
// ---------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(512, 1) bwd_simt_kernel(BwdParams p) {
  constexpr int T = kTile, SQ = 32, NT = 512, PER = D / 4;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem_raw);   // [T][D]
  __nv_bfloat16* Vs = Ks + T * D;                                     // [T][D]
  __nv_bfloat16* Qs = Vs + T * D;                                     // [SQ][D]
  __nv_bfloat16* dOs = Qs + SQ * D;                                   // [SQ][D]
  float* Ps = reinterpret_cast<float*>(dOs + SQ * D);                 // [SQ][T + 1]
  float* dSs = Ps + SQ * (T + 1);                                     // [SQ][T + 1]
  float* dQs = dSs + SQ * (T + 1);                                    // [T][D]
  float* lse_s = dQs + T * D;                                         // [SQ]
  float* Dd_s = lse_s + SQ;                                           // [SQ]
  __shared__ int go;

  const int tid = threadIdx.x;
  const int my_r = tid / 4;               // kv row owned for dK/dV
  const size_t rs = (size_t)p.H * D;
  float dk[PER], dv[PER];

  for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    const int bh = u / p.num_slots, slot = u % p.num_slots;
    const int b = bh / p.H, h = bh % p.H;
    const size_t base = ((size_t)b * p.S * p.H + h) * D;
    const int t_beg = p.slot_off[slot], t_end = p.slot_off[slot + 1];
    int cur_i = -1;
    for (int t = t_beg; t <= t_end; ++t) {
      const int i = (t < t_end) ? (p.tasks[t] >> 16) : -2;
      const int j = (t < t_end) ? (p.tasks[t] & 0xffff) : 0;
      if (i != cur_i) {
        if (cur_i >= 0) {                                   // flush dK/dV of tile cur_i
#pragma unroll
          for (int k = 0; k < PER; ++k) {
            const int c = (tid % 4) + 4 * k;
            const size_t g = base + (size_t)(cur_i * T + my_r) * rs + c;
            p.dk[g] = __float2bfloat16(p.scale * dk[k]);
            p.dv[g] = __float2bfloat16(dv[k]);
          }
        }
        if (t == t_end) break;
        __syncthreads();
        for (int e = tid; e < T * D; e += NT) {
          const int r = e / D, c = e % D;
          Ks[e] = p.k[base + (size_t)(i * T + r) * rs + c];
          Vs[e] = p.v[base + (size_t)(i * T + r) * rs + c];
        }
#pragma unroll
        for (int k = 0; k < PER; ++k) dk[k] = dv[k] = 0.f;
        cur_i = i;
      }
      for (int sc = 0; sc < T / SQ; ++sc) {
        const int q0 = j * T + sc * SQ;
        __syncthreads();
        for (int e = tid; e < SQ * D; e += NT) {
          const int r = e / D, c = e % D;
          Qs[e] = p.q[base + (size_t)(q0 + r) * rs + c];
          dOs[e] = p.dO[base + (size_t)(q0 + r) * rs + c];
        }
        if (tid < SQ) {
          lse_s[tid] = p.lse[(size_t)bh * p.S + q0 + tid] * kLog2e;
          Dd_s[tid] = p.Dsum[(size_t)bh * p.S + q0 + tid];
        }
        __syncthreads();
        for (int e = tid; e < SQ * T; e += NT) {
          const int qr = e / T, kc = e % T;
          float pv = 0.f, ds = 0.f;
          if (!(p.causal && i * T + kc > q0 + qr)) {
            float s = 0.f, dp = 0.f;
#pragma unroll 8
            for (int x = 0; x < D; ++x) {
              s += bf(Qs[qr * D + x]) * bf(Ks[kc * D + x]);
              dp += bf(dOs[qr * D + x]) * bf(Vs[kc * D + x]);
            }
            pv = exp2f(s * p.scale_log2 - lse_s[qr]);
            ds = pv * (dp - Dd_s[qr]);
          }
          Ps[qr * (T + 1) + kc] = pv;
          dSs[qr * (T + 1) + kc] = ds;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < PER; ++k) {
          const int c = (tid % 4) + 4 * k;
          float a = dv[k], g = dk[k];
          for (int qr = 0; qr < SQ; ++qr) {
            a += Ps[qr * (T + 1) + my_r] * bf(dOs[qr * D + c]);
            g += dSs[qr * (T + 1) + my_r] * bf(Qs[qr * D + c]);
          }
          dv[k] = a;
          dk[k] = g;
        }
        for (int e = tid; e < SQ * D; e += NT) {
          const int qr = e / D, c = e % D;
          float a = 0.f;
          for (int kc = 0; kc < T; ++kc) a += dSs[qr * (T + 1) + kc] * bf(Ks[kc * D + c]);
          dQs[(sc * SQ + qr) * D + c] = a;
        }
      }
      __syncthreads();
      // ---- reduction phase R(i, j) ----
      float* acc = p.dq_acc + ((size_t)bh * p.S + (size_t)j * T) * D;
      if (p.deterministic) {
        const int o = p.ord[i * p.n + j];
        const int last = p.cnt[j] - 1;
        int* sem = p.sems + (size_t)bh * p.n + j;
        if (tid == 0)
          go = wait_turn(sem, o + p.ordinal_skew, p.ws_header, p.timeout_ns, bh, j) ? 1 : 0;
        __syncthreads();
        if (!go) return;                                   // uniform across the CTA
        for (int e = tid; e < T * D; e += NT) {
          const float x = dQs[e];
          const int r = e / D, c = e % D;
          const size_t g = base + (size_t)(j * T + r) * rs + c;
          if (o == last) {
            const float tot = (o == 0) ? x : __ldcg(acc + e) + x;
            p.dq[g] = __float2bfloat16(p.scale * tot);
          } else if (o == 0) {
            __stcg(acc + e, x);
          } else {
            __stcg(acc + e, __ldcg(acc + e) + x);
          }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release_gpu(sem, o + 1 + p.ordinal_skew);
      } else {
        for (int e = tid; e < T * D; e += NT) atomicAdd(acc + e, dQs[e]);
      }
    }
  }
}

}  // namespace dash
