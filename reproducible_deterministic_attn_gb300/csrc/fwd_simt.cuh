// Forward pass on the CUDA cores (fp32 FMA): O and LSE for the backward to recompute P
// from. One CTA per (64-row Q tile, batch * head), online softmax over 64-key chunks.
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

}  // namespace dash
