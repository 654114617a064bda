// Backward helper kernels around the main kernel: the preprocess (D = rowsum(dO * O),
// clearing of the semaphores, status header and fp32 dQ accumulator) and the final
// dQ convert. Both are memory-bound passes with fixed reduction trees (deterministic).
#pragma once

#include "common.cuh"

namespace dash {

// x as hi + mid + lo, each rounded to bf16 in turn (their sum equals x to ~2^-24 |x|),
// packed as K columns 0, 1, 2 of a row of the score-offset block; columns 3..7 zero.
__device__ __forceinline__ uint4 split3_bf16(float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  return make_uint4((uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(mid) << 16),
                    (uint32_t)__bfloat16_as_ushort(lo), 0u, 0u);
}

// ---------------------------------------------------------------------------------
// Preprocess: D = rowsum(dO * O) and -LSE*log2(e) per row (and, for head dimension 128,
// the score-offset blocks of -LSE/scale and -D); clear the semaphores, the split-tile
// flags, the status header and the fp32 dQ accumulator copies in use. A row of D elements is read
// by D/8 consecutive lanes of one warp, 8 bf16 (16 bytes) of dO and of O each; each lane
// sums its 8 products in order, then a fixed shuffle tree over the row's lanes
// (deterministic).
// Index arithmetic is 32-bit: B*S*H*D < 2^31 is a precondition of every entry point.
// ---------------------------------------------------------------------------------
__global__ void bwd_preprocess_kernel(BwdParams p) {
  const int lanes = p.D >> 3;                     // lanes per row: 8 (D = 64) or 16 (D = 128)
  const int rpw = 32 / lanes;                     // whole rows per warp and pass
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nth = gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31;
  const int sub = lane % lanes;                   // this lane's 8-element chunk of its row
  const int rows = p.B * p.H * p.S;
  // the loop bound depends on the warp only, so every lane reaches the shuffles
  for (int base = (tid >> 5) * rpw; base < rows; base += (nth >> 5) * rpw) {
    const int r = base + lane / lanes;            // enumerates (b, h, s): Dsum is contiguous
    float acc = 0.f;
    if (r < rows) {
      const int s = r % p.S, bh = r / p.S;
      const int h = bh % p.H, b = bh / p.H;
      const size_t off = (((size_t)b * p.S + s) * p.H + h) * p.D + sub * 8;
      const uint4 g = *reinterpret_cast<const uint4*>(p.dO + off);
      const uint4 o = *reinterpret_cast<const uint4*>(p.o + off);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 gf = __bfloat1622float2(g2[k]), of = __bfloat1622float2(o2[k]);
        acc += gf.x * of.x;
        acc += gf.y * of.y;
      }
    }
    // fixed tree over the row's lanes (xor partners stay inside the row's aligned group)
    for (int w = lanes >> 1; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (r < rows && sub == 0) {
      p.Dsum[r] = acc;
      p.nlse2[r] = -p.lse[r] * kLog2e;
      if (p.qx) {
        // row rr of 128-row tile t of head bh; 8-row group g, K columns 0..7 at byte
        // 256 g + 16 (rr % 8), K columns 8..15 128 bytes further (all zero)
        const int s = r % p.S, bh = r / p.S;
        const int rr = s % kTile;
        const size_t off = (((size_t)bh * (p.S / kTile) + s / kTile) * 4096 +
                            (size_t)(rr >> 3) * 256 + (rr & 7) * 16) / sizeof(uint4);
        reinterpret_cast<uint4*>(p.qx)[off] = split3_bf16(-p.lse[r] / p.scale);
        reinterpret_cast<uint4*>(p.qx)[off + 8] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(p.dox)[off] = split3_bf16(-acc);
        reinterpret_cast<uint4*>(p.dox)[off + 8] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  for (int e = tid; e < p.num_sems; e += nth) p.sems[e] = 0;
  for (int e = tid; e < kSplitTiles * kSplitFlags; e += nth) p.split_flags[e] = 0;
  if (tid < (int)(kWsHeaderBytes / sizeof(int))) p.ws_header[tid] = 0;
  const long long nacc4 = (long long)p.chains * p.B * p.H * p.S * p.D / 4;   // copies in use
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (long long e = tid; e < nacc4; e += nth) acc4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * accumulator), 8 elements per thread: two 16-byte loads per copy in
// use (the copies added in index order), one 16-byte store. 32-bit index arithmetic.
__global__ void dq_convert_kernel(BwdParams p) {
  const int n = p.B * p.H * p.S * p.D;
  const int n8 = n >> 3;
  const float4* acc4 = reinterpret_cast<const float4*>(p.dq_acc);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
    const int e = i << 3;                      // first element: (b*H + h)*S*D + s*D + c
    const int c = e % p.D, row = e / p.D;
    const int s = row % p.S, bh = row / p.S;
    const int h = bh % p.H, b = bh / p.H;
    float4 a0 = acc4[2 * i], a1 = acc4[2 * i + 1];
    for (int k = 1; k < p.chains; ++k) {
      const float4 b0 = acc4[2 * i + (size_t)k * (n >> 2)], b1 = acc4[2 * i + 1 + (size_t)k * (n >> 2)];
      a0.x += b0.x; a0.y += b0.y; a0.z += b0.z; a0.w += b0.w;
      a1.x += b1.x; a1.y += b1.y; a1.z += b1.z; a1.w += b1.w;
    }
    const float sc = p.scale;
    __nv_bfloat162 q[4] = {__floats2bfloat162_rn(sc * a0.x, sc * a0.y), __floats2bfloat162_rn(sc * a0.z, sc * a0.w),
                           __floats2bfloat162_rn(sc * a1.x, sc * a1.y), __floats2bfloat162_rn(sc * a1.z, sc * a1.w)};
    *reinterpret_cast<uint4*>(p.dq + (((size_t)b * p.S + s) * p.H + h) * p.D + c) =
        *reinterpret_cast<const uint4*>(q);
  }
}

}  // namespace dash
