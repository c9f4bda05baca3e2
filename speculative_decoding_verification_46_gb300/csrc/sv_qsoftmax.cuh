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

// The weight 2^((x - m) c) of one token: the final draw's q_weight.
__device__ __forceinline__ float qs_weight(float x, float m, float c, float c_lo) { return q_weight(x, m, c, c_lo); }

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

namespace sv {

// ---- q with truncation: top-k (value desc, index asc) then top-p over the
// renormalised top-k, q renormalised over what is kept, zero elsewhere - the
// transform the target's p gets.  One CTA of kQsThreads threads per draft
// row, k <= kQsThreads:
//   1. the row maximum and NaN / +inf detection;
//   2. tau = the k-th largest of the threads' maxima, a lower bound of the
//      k-th largest value (k distinct elements reach it): one pass collects
//      every element >= tau (usually a few times k).  Only if more than
//      kQtCap do, K = the exact k-th largest value key by a radix select over
//      the row (one pass per 8-bit digit of the order-preserving key;
//      warp-private histograms, lanes with equal digits add once), then
//   3. the values above K and the ties at K; more than kQtCap of those (a
//      flood of ties) keeps the lowest-index ties directly (threads own
//      contiguous index ranges, a scan of their tie counts keeps index order);
//   4. a bitonic sort of the (value, index) keys, largest first: the first k
//      are the top-k with ties to the lowest index;
//   5. softmax weights over the k, top-p prefix J, renormalised over J;
//   6. the J kept probabilities written (the row holds zeros otherwise).
// Every pass reads the row with coalesced 16-byte loads when V is a multiple
// of the vector width.
constexpr int kQtCap = 4096;

struct QtSmem {
  unsigned long long cand[kQtCap];
  int hist[kQsWarps][256];
  int iscan[kQsWarps];
  F2 f2scan[kQsWarps];
  float fred[kQsWarps];
  int ired[kQsWarps];
  int count;
  int digit;
  int rank;
  int J;
};

__device__ __forceinline__ F2 block_excl_f2_qs(F2 v, F2* sm, F2* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const F2 inc = warp_incl_scan_f2(v);
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  F2 base{0.f, 0.f}, tot{0.f, 0.f};
  for (int w = 0; w < kQsWarps; ++w) {
    if (w < warp) base = f2_add(base, sm[w]);
    tot = f2_add(tot, sm[w]);
  }
  __syncthreads();
  *total = tot;
  F2 excl = f2_shfl_up(inc, 1);
  if (lane == 0) excl = F2{0.f, 0.f};
  return f2_add(base, excl);
}

__device__ __forceinline__ int qt_block_excl_int(int v, int* sm, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  int base = 0, tot = 0;
  for (int w = 0; w < kQsWarps; ++w) {
    if (w < warp) base += sm[w];
    tot += sm[w];
  }
  __syncthreads();
  *total = tot;
  return base + inc - v;
}

// The k-th largest of the kQsThreads keys (one per thread), by a radix select
// over 8-bit digits from the top; hist holds 256 ints.
__device__ __forceinline__ uint32_t qt_kth_largest_key(uint32_t key, int k, int* hist, int* s_digit, int* s_rank) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0u;
  int rank = k;
  for (int lo = 24; lo >= 0; lo -= 8) {
    const uint32_t upper = lo == 24 ? 0u : ~((1u << (lo + 8)) - 1u);
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    if ((key & upper) == prefix) atomicAdd(&hist[(key >> lo) & 255u], 1);
    __syncthreads();
    if (tid == 0) {
      int run = 0, dg = 0;
      for (int d = 255; d >= 0; --d) {
        if (run + hist[d] >= rank) {
          dg = d;
          break;
        }
        run += hist[d];
      }
      *s_digit = dg;
      *s_rank = rank - run;
    }
    __syncthreads();
    prefix |= (uint32_t)*s_digit << lo;
    rank = *s_rank;
    __syncthreads();
  }
  return prefix;
}

// Bitonic sort of cand[0, P) (P a power of two, at most kQtCap), largest first.
__device__ __forceinline__ void qt_sort_desc(unsigned long long* cand, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P; i += kQsThreads) {
        const int partner = i ^ stride;
        if (partner > i) {
          const unsigned long long a = cand[i], b2 = cand[partner];
          const bool desc = (i & size) == 0;
          if (desc ? (a < b2) : (a > b2)) {
            cand[i] = b2;
            cand[partner] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// q is written only where it is kept: the row must hold zeros on entry (the
// workspace contract) and q_clear_kernel restores them after the call, from
// the list of kept indices (plus one; 0 = none) written here.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kQsThreads) q_truncate_kernel(const T* __restrict__ ql, float* __restrict__ q, int V,
                                                                int k, float top_p, float c, float c_lo,
                                                                int* __restrict__ kept_list) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  extern __shared__ __align__(16) unsigned char qt_raw[];
  QtSmem& sm = *reinterpret_cast<QtSmem*>(qt_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T* src = ql + (size_t)blockIdx.x * V;
  float* dst = q + (size_t)blockIdx.x * V;
  const int NV = V / VW;
  auto val = [&](int v) { return TR::get(load_slot<T>(src, v, 1, false), 0); };
  // every element once, coalesced: fn(value, index)
  auto each = [&](auto&& fn) {
    if (VEC) {
#pragma unroll 4
      for (int j = tid; j < NV; j += kQsThreads) {
        const uint4 x = ldg_v4(src + (size_t)j * VW);
#pragma unroll
        for (int t = 0; t < VW; ++t) fn(TR::get(x, t), j * VW + t);
      }
    } else {
      for (int v = tid; v < V; v += kQsThreads) fn(val(v), v);
    }
  };
  k = min(k, V);

  // 1. maximum (this thread's, then the row's), bad row
  float m = -INFINITY;
  int bad = 0;
  each([&](float x, int) {
    bad |= (x != x) | (x == INFINITY);
    m = fmaxf(m, x);
  });
  const float m_thread = m;
  m = qs_block_max(m, sm.fred);
  bad = qs_block_or(bad, sm.ired) || !(m > -INFINITY);
  if (bad) return;   // no distribution: q stays 0

  // 2a. tau = the k-th largest thread maximum: k distinct elements reach it,
  // so every top-k element does; collect all elements >= tau (usually a few
  // times k) and sort them
  const uint32_t tau = qt_kth_largest_key(okey(m_thread), k, &sm.hist[0][0], &sm.digit, &sm.rank);
  if (tid == 0) sm.count = 0;
  __syncthreads();
  each([&](float x, int v) {
    if (okey(x) >= tau) {
      const int pos = atomicAdd(&sm.count, 1);
      if (pos < kQtCap) sm.cand[pos] = comp_key(x, v);
    }
  });
  __syncthreads();
  int N = sm.count;
  int P = 2;
  if (N <= kQtCap) {
    while (P < N) P <<= 1;
  } else {
  // 2b. too many elements at or above tau: K = the k-th largest value key by
  // a radix select (digits from the top, 8 bits a pass; the key bits below
  // KEY_LOW_BIT carry nothing for 16-bit types and are masked)
  const uint32_t kmask = ~((1u << TR::KEY_LOW_BIT) - 1u);
  uint32_t prefix = 0u;
  int rank = k;   // rank sought among the keys matching prefix
  for (int hi = 31; hi >= TR::KEY_LOW_BIT; hi -= 8) {
    const int lo = hi - 7 > TR::KEY_LOW_BIT ? hi - 7 : TR::KEY_LOW_BIT;
    const int nb = hi - lo + 1;
    const uint32_t upper = hi == 31 ? 0u : ~((1u << (hi + 1)) - 1u);
    for (int e = tid; e < kQsWarps * 256; e += kQsThreads) (&sm.hist[0][0])[e] = 0;
    __syncthreads();
    each([&](float x, int) {
      const uint32_t key = okey(x) & kmask;
      const bool match = (key & upper) == prefix;
      const uint32_t dg = (key >> lo) & ((1u << nb) - 1u);
      const unsigned act = __activemask();
      const unsigned same = __match_any_sync(act, match ? dg : 0xffffffffu);
      if (match && lane == __ffs(same) - 1) atomicAdd(&sm.hist[warp][dg], __popc(same));
    });
    __syncthreads();
    if (tid < 256) {
      int t = 0;
      for (int w = 0; w < kQsWarps; ++w) t += sm.hist[w][tid];
      sm.hist[0][tid] = t;
    }
    __syncthreads();
    if (tid == 0) {
      int run = 0, dg = 0;
      for (int d = (1 << nb) - 1; d >= 0; --d) {
        if (run + sm.hist[0][d] >= rank) {
          dg = d;
          break;
        }
        run += sm.hist[0][d];
      }
      sm.digit = dg;
      sm.rank = rank - run;
    }
    __syncthreads();
    prefix |= (uint32_t)sm.digit << lo;
    rank = sm.rank;
    __syncthreads();
  }
  const uint32_t K = prefix;

  // 3. candidates: the values above K and the ties at K, sorted below
  if (tid == 0) sm.count = 0;
  __syncthreads();
  each([&](float x, int v) {
    if ((okey(x) & kmask) >= K) {
      const int pos = atomicAdd(&sm.count, 1);
      if (pos < kQtCap) sm.cand[pos] = comp_key(x, v);
    }
  });
  __syncthreads();
  N = sm.count;
  P = kQsThreads;
  if (N <= kQtCap) {
    while (P < N) P <<= 1;
  } else {
    // a flood of ties: the values above K, then the first `rank` ties in index order
    __syncthreads();
    if (tid == 0) sm.count = 0;
    const int chunk = (V + kQsThreads - 1) / kQsThreads;
    const int v0 = tid * chunk, v1 = min(v0 + chunk, V);
    int eq = 0;
    for (int v = v0; v < v1; ++v) eq += (okey(val(v)) & kmask) == K;
    int tot_eq;
    const int eq_base = qt_block_excl_int(eq, sm.iscan, &tot_eq);
    for (int v = v0, seen = eq_base; v < v1; ++v) {
      const float x = val(v);
      const uint32_t key = okey(x) & kmask;
      bool take = key > K;
      if (key == K) take = seen++ < rank;
      if (take) {
        const int pos = atomicAdd(&sm.count, 1);
        if (pos < kQsThreads) sm.cand[pos] = comp_key(x, v);
      }
    }
    __syncthreads();
    N = min(sm.count, kQsThreads);
    P = kQsThreads;
  }
  }
  for (int i = N + tid; i < P; i += kQsThreads) sm.cand[i] = 0ull;   // padding sorts last
  __syncthreads();

  // 4. sort, largest key first; the first k are kept
  qt_sort_desc(sm.cand, P);
  N = min(N, k);

  // 5. weights over the k, top-p prefix, renormalised over it
  const float x = tid < N ? comp_val(sm.cand[tid]) : -INFINITY;
  const float w = tid < N ? q_weight(x, m, c, c_lo) : 0.f;
  F2 tot;
  const F2 excl = block_excl_f2_qs(F2{w, 0.f}, sm.f2scan, &tot);
  int J = N;
  if (top_p < 1.0f) {
    // the first rank whose cumulative renormalised mass reaches top_p
    const float cum = (float)(((double)excl.hi + (double)excl.lo + (double)w) / ((double)tot.hi + (double)tot.lo));
    if (tid == 0) sm.J = N;
    __syncthreads();
    if (tid < N && cum >= top_p) atomicMin(&sm.J, tid + 1);
    __syncthreads();
    J = sm.J;
  }
  F2 kept;
  (void)block_excl_f2_qs(F2{tid < J ? w : 0.f, 0.f}, sm.f2scan, &kept);
  const float Sk = kept.hi + kept.lo;

  // 6. the kept entries (the rest of the row is zero) and their list
  if (tid < J) {
    const int idx = comp_idx(sm.cand[tid]);
    if (idx >= 0 && idx < V) {
      dst[idx] = __fdiv_rn(w, Sk);
      kept_list[(size_t)blockIdx.x * k + tid] = idx + 1;
    }
  }
}

// After the call: the kept entries back to zero, and the list with them.
__global__ void q_clear_kernel(float* __restrict__ q, int* __restrict__ kept_list, int V, int k) {
  for (int t = threadIdx.x; t < k; t += blockDim.x) {
    int* e = kept_list + (size_t)blockIdx.x * k + t;
    const int idx = *e - 1;
    if (idx >= 0 && idx < V) {
      q[(size_t)blockIdx.x * V + idx] = 0.f;
      *e = 0;
    }
  }
}

}  // namespace sv
