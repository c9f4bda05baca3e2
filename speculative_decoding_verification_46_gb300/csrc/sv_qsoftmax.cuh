// q from the draft's logits ("11.1 核心原理", section 11.1.2: temperature
// (and truncation) apply to the draft's distribution q_i as to the target's
// p_i, and q_i must be the draft's actual proposal).  One CTA of kQsThreads
// threads per draft row writes q_i(v) = 2^((x_v - m) c) / S in float32, where
// m is the row maximum and S the two-float sum of the same weights; the
// verify path then reads that q as it reads a caller's q.
//
// Three passes over the row (the first from HBM, the others mostly from L2):
// the maximum (and NaN / +inf detection), the sum, the write.  The weight of
// every token is formed by the same code in passes two and three, so
// sum_v q(v) is 1 up to the float32 rounding of each q(v).  A row holding
// NaN or +inf, or only -inf, defines no distribution: its q is written as 0
// everywhere (the step then flags q_i(d_i) <= 0 where it tests that row).
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kQsThreads = 1024;
constexpr int kQsWarps = kQsThreads / 32;

// The weight 2^((x - m) c) of one token (c = log2(e) / T as c + c_lo): x - m
// is exact for 16-bit logits; -inf is clamped to an exponent whose ex2.approx
// flushes to 0; ex2.approx with a first-order correction for the exponent's
// low part.
__device__ __forceinline__ float qs_weight(float x, float m, float c, float c_lo) {
  const float dh = fmaxf(x - m, -1.0e4f);
  const float p = dh * c;
  const float e = fmaf(dh, c_lo, fmaf(dh, c, -p));
  const float y = ex2_approx(p);
  return fmaf(y * 6.931471825e-01f, e, y);
}

__device__ __forceinline__ float qs_block_max(float v, float* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  float t = sm[0];
  for (int w = 1; w < kQsWarps; ++w) t = fmaxf(t, sm[w]);
  __syncthreads();
  return t;
}

__device__ __forceinline__ int qs_block_or(int v, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __any_sync(0xffffffffu, v) ? 1 : 0;
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < kQsWarps; ++w) t |= sm[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ F2 qs_block_sum(F2 v, F2* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = f2_add(v, f2_shfl_xor(v, o));
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  F2 t = sm[0];
  for (int w = 1; w < kQsWarps; ++w) t = f2_add(t, sm[w]);
  __syncthreads();
  return t;
}

// VEC: the row is read as 16-byte vectors (V a multiple of the vector width;
// the rows are then 16-byte aligned since the base is); else element by element.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kQsThreads) q_softmax_kernel(const T* __restrict__ ql, float* __restrict__ q, int V,
                                                               float c, float c_lo) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  __shared__ float s_f[kQsWarps];
  __shared__ int s_i[kQsWarps];
  __shared__ F2 s_f2[kQsWarps];
  const int tid = threadIdx.x;
  const T* src = ql + (size_t)blockIdx.x * V;
  float* dst = q + (size_t)blockIdx.x * V;
  const int NV = V / VW;

  // pass 1: maximum; NaN or +inf anywhere makes the row bad
  float m = -INFINITY;
  int bad = 0;
  if (VEC) {
#pragma unroll 4
    for (int j = tid; j < NV; j += kQsThreads) {
      const uint4 x = ldg_v4(src + (size_t)j * VW);
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        const float v = TR::get(x, t);
        bad |= (v != v) | (v == INFINITY);
        m = fmaxf(m, v);
      }
    }
  } else {
    for (int v0 = tid; v0 < V; v0 += kQsThreads) {
      const float v = TR::get(load_slot<T>(src, v0, 1, false), 0);
      bad |= (v != v) | (v == INFINITY);
      m = fmaxf(m, v);
    }
  }
  m = qs_block_max(m, s_f);
  bad = qs_block_or(bad, s_i) || !(m > -INFINITY);

  // pass 2: S = sum of the weights (two-float)
  float sh = 0.f, sl = 0.f;
  if (!bad) {
    if (VEC) {
#pragma unroll 4
      for (int j = tid; j < NV; j += kQsThreads) {
        const uint4 x = ldg_v4(src + (size_t)j * VW);
#pragma unroll
        for (int t = 0; t < VW; ++t) RunAcc::acc2(sh, sl, qs_weight(TR::get(x, t), m, c, c_lo), 0.f);
      }
    } else {
      for (int v0 = tid; v0 < V; v0 += kQsThreads)
        RunAcc::acc2(sh, sl, qs_weight(TR::get(load_slot<T>(src, v0, 1, false), 0), m, c, c_lo), 0.f);
    }
  }
  const F2 S = qs_block_sum(f2_norm(sh, sl), s_f2);
  const float Sf = S.hi + S.lo;

  // pass 3: q(v) = weight / S
  if (VEC) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll 2
    for (int j = tid; j < NV; j += kQsThreads) {
      float w[VW];
      if (!bad) {
        const uint4 x = ldg_v4(src + (size_t)j * VW);
#pragma unroll
        for (int t = 0; t < VW; ++t) w[t] = __fdiv_rn(qs_weight(TR::get(x, t), m, c, c_lo), Sf);
      } else {
#pragma unroll
        for (int t = 0; t < VW; ++t) w[t] = 0.f;
      }
#pragma unroll
      for (int h = 0; h < VW / 4; ++h)
        d4[(size_t)j * (VW / 4) + h] = make_float4(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
    }
  } else {
    for (int v0 = tid; v0 < V; v0 += kQsThreads)
      dst[v0] = bad ? 0.f : __fdiv_rn(qs_weight(TR::get(load_slot<T>(src, v0, 1, false), 0), m, c, c_lo), Sf);
  }
}

}  // namespace sv
