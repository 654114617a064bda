// Backward helper kernels around the main kernel: the preprocess (D = rowsum(dO * O),
// clearing of the semaphores, status header and fp32 dQ accumulator) and the final
// dQ convert. Both are memory-bound passes with fixed reduction trees (deterministic).
#pragma once

#include "common.cuh"

namespace dash {

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------------------------
// Preprocess: D = rowsum(dO * O) (one warp per row, fixed shuffle tree) and -LSE*log2(e)
// per row, clear the semaphores, the status header and the fp32 dQ accumulator.
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
    if (lane == 0) {
      p.Dsum[r] = acc;
      p.nlse2[r] = -p.lse[r] * kLog2e;
    }
  }
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nth = (long long)gridDim.x * blockDim.x;
  for (long long e = tid; e < p.num_sems; e += nth) p.sems[e] = 0;
  if (tid < (long long)(kWsHeaderBytes / sizeof(int))) p.ws_header[tid] = 0;
  const long long nacc4 = (long long)p.chains * p.B * p.H * p.S * p.D / 4;   // copies in use
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (long long e = tid; e < nacc4; e += nth) acc4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * accumulator).
__global__ void dq_convert_kernel(BwdParams p) {
  const long long n = (long long)p.B * p.H * p.S * p.D;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(e % p.D);
    const long long row = e / p.D;             // (b*H + h) * S + s
    const int s = (int)(row % p.S);
    const long long bh = row / p.S;
    const int h = (int)(bh % p.H), b = (int)(bh / p.H);
    // k interleaved chains: the copies added in index order
    float a = p.dq_acc[e];
    for (int c = 1; c < p.chains; ++c) a += p.dq_acc[e + (long long)c * n];
    p.dq[(((size_t)b * p.S + s) * p.H + h) * p.D + c] = __float2bfloat16(p.scale * a);
  }
}

}  // namespace dash
