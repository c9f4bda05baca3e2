// Top-k / top-p sampling verify: persistent kernel, one row per CTA at a time.
//
// Per row (temperature, then top-k ranked by (logit desc, index asc), then
// top-p over the renormalised top-k, as in "11.1 核心原理" section 11.1.2):
//
//   pass 1  stream the row from HBM (16-byte loads, L2 evict-last hint) and
//           keep each thread's maximum.  The k-th largest of the 512 thread
//           maxima, tau, is a lower bound of the row's k-th largest value:
//           the k threads holding those maxima each own an element >= tau.
//           It is found exactly by bisection over the order-preserving key
//           (one __syncthreads_count per key bit).
//   pass 2  stream the row again (now mostly an L2 hit, evict-first hint) and
//           append only the elements >= tau to per-warp candidate buffers.
//           For LM-like rows that is k plus a handful of elements; a vector
//           is skipped after one packed max-compare.
//   select  rank the candidates by (value desc, index asc) - a total order,
//           so ties at the k-th value are resolved by index exactly as the
//           oracle does - and keep the first k, in order.
//   top-p   softmax(./T) over the k (exp2 in float32, sums in float64), keep
//           the shortest prefix whose mass reaches top_p, renormalise, store
//           the kept (index, probability) list; look up p(d_i), gather q(d_i)
//           and store a_i = min(1, p/q).
//
// The last row of a sequence to finish (an atomic ticket; no CTA waits) runs
// the acceptance scan and the final draw over the kept list of row n (the
// residual max(p - q, 0) needs q only at the kept indices) or row gamma.
//
// If a warp's candidate buffer overflows (massive ties at tau), the row falls
// back to an exact bisection over 64-bit (value, index) keys, re-reading the
// row once per key bit: slow, but only for such rows.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkU = 4;
constexpr int kTkWarpCap = 256;
constexpr int kTkCap = kTkWarps * kTkWarpCap;

struct TopkSmem {
  unsigned long long cand[kTkCap];   // per-warp candidate buffers (warp w: [w*cap, (w+1)*cap))
  unsigned long long sel[kMaxK];     // the row's top-k, descending
  double w[kMaxK];
  int widx[kMaxK];
  unsigned long long mout[kMaxK];
  int wcount[kTkWarps];
  int ired[kTkWarps];
  double dred[kTkWarps];
  int flag;
  int count;
  int n;
  int status;
  int token;
  int J;
  double WJ;
  double pd;
};

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ldg_v4_hint(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}

__device__ __forceinline__ int block_sum_int_n(int v, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < nw; ++w) t += sm[w];
  return t;
}

// Final step of a sequence (run by the CTA that finished its last row).
__device__ void topk_finish_sequence(const Params& p, int b, TopkSmem& sm) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int k = p.top_k, G = p.gamma, G1 = G + 1, V = p.V;
  if (tid == 0) {
    int n = G;
    for (int i = 0; i < G; ++i) {
      const float u = __ldg(p.uniforms + b * G1 + i);
      if (!((double)u < __ldcg(p.acc + b * G + i))) { n = i; break; }
    }
    sm.n = n;
    sm.status = __ldcg(&p.seq[b].status);
  }
  __syncthreads();
  const int n = sm.n;
  const int2* kept = p.rowres + (size_t)(b * G1 + n) * (k + 1);
  const int J = __ldcg(kept).x;
  const bool resid = n < G;
  const float* qrow = resid ? p.q + ((size_t)b * G + n) * V : nullptr;
  for (int e = tid; e < J; e += nt) {
    const int2 en = __ldcg(kept + 1 + e);
    sm.widx[e] = en.x;
    sm.w[e] = (double)__int_as_float(en.y);
  }
  __syncthreads();
  // order the kept entries by token index; r_j = max(p_j - q_j, 0) or p_j
  double* rs = reinterpret_cast<double*>(sm.cand);
  for (int e = tid; e < J; e += nt) {
    const int me = sm.widx[e];
    int rank = 0;
    for (int j = 0; j < J; ++j) rank += sm.widx[j] < me;
    double r = sm.w[e];
    if (resid) r = fmax(r - (double)__ldg(qrow + me), 0.0);
    sm.mout[rank] = (unsigned long long)me;
    rs[rank] = r;
    rs[kMaxK + rank] = sm.w[e];
  }
  __syncthreads();
  if (tid == 0) {
    int status = sm.status;
    double R = 0.0;
    for (int e = 0; e < J; ++e) R += rs[e];
    if (resid && !(R > 0.0)) {
      status |= SEQ_RESID0;   // zero residual mass (rounding only): draw from p_n
      R = 0.0;
      for (int e = 0; e < J; ++e) {
        rs[e] = rs[kMaxK + e];
        R += rs[e];
      }
    }
    const double t = (double)__ldg(p.uniforms + b * G1 + G) * R;
    int tok = -1, lastpos = -1;
    double C = 0.0;
    for (int e = 0; e < J; ++e) {
      C += rs[e];
      if (rs[e] > 0.0) lastpos = e;
      if (C > t) { tok = (int)sm.mout[e]; break; }
    }
    if (tok < 0) tok = lastpos >= 0 ? (int)sm.mout[lastpos] : (J > 0 ? (int)sm.mout[0] : 0);
    if (tok < 0 || tok >= V) tok = 0;
    sm.token = tok;
    p.out_n[b] = n;
    if (p.out_status) p.out_status[b] = status;
    p.seq[b].status = 0;
  }
  __syncthreads();
  for (int j = tid; j < G1; j += nt)
    p.out_tokens[b * G1 + j] = j < n ? __ldg(p.draft + b * G + j) : (j == n ? sm.token : -1);
  // the kept lists and acceptance probabilities have been consumed: zero them
  for (int e = tid; e < G1 * (k + 1); e += nt) p.rowres[(size_t)b * G1 * (k + 1) + e] = make_int2(0, 0);
  for (int e = tid; e < G; e += nt) p.acc[b * G + e] = 0.0;
}

template <typename T>
__global__ void __launch_bounds__(kTkThreads, 2)
topk_rows_kernel(const Params p) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.gamma, G1 = G + 1, V = p.V, k = p.top_k;
  const int R = p.B * G1;
  const int NV = V / VW;                       // V % VW == 0 on this path
  const uint64_t pol_last = policy_evict_last();
  const uint64_t pol_first = policy_evict_first();

  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int b = r / G1, i = r - b * G1;
    const T* row = static_cast<const T*>(p.logits) + (size_t)r * V;
    __syncthreads();   // the previous row's shared state is no longer in use
    if (tid < kTkWarps) sm.wcount[tid] = 0;
    // the row's draft token and q(d): needed only at the end, fetched now
    int d_row = -1;
    float q_row = 0.f;
    if (tid == 0 && i < G) {
      d_row = __ldg(p.draft + b * G + i);
      if (d_row >= 0 && d_row < V) q_row = __ldg(p.q + ((size_t)b * G + i) * V + d_row);
    }

    // ---- pass 1: thread maxima (NaN ignored here; pass 2 flags NaN)
    float tmax = -INFINITY;
    int any = 0;
    for (int v0 = tid; v0 < NV; v0 += kTkThreads * kTkU) {
      uint4 buf[kTkU];
#pragma unroll
      for (int u = 0; u < kTkU; ++u) {
        const int vi = v0 + u * kTkThreads;
        if (vi < NV) buf[u] = ldg_v4_hint(row + (size_t)vi * VW, pol_last);
      }
#pragma unroll
      for (int u = 0; u < kTkU; ++u) {
        if (v0 + u * kTkThreads < NV) {
          tmax = fmaxf(tmax, TR::template vmax<false>(buf[u]));
          any = 1;
        }
      }
    }
    // ---- tau: k-th largest thread maximum, by bisection on its key
    const uint32_t tkey = any ? okey(tmax) : 0u;
    uint32_t K = 0u;
    if (NV * VW > k) {
      for (int bit = 31; bit >= TR::KEY_LOW_BIT; --bit) {
        const uint32_t Kt = K | (1u << bit);
        if (__syncthreads_count(tkey >= Kt) >= k) K = Kt;
      }
    } else {
      __syncthreads();
    }
    const float tau = K == 0u ? -INFINITY : key_to_float(K);

    // ---- pass 2: candidates >= tau
    int nan_seen = 0;
    unsigned long long* wbuf = sm.cand + warp * kTkWarpCap;
    for (int v0 = tid; v0 < NV; v0 += kTkThreads * kTkU) {
      uint4 buf[kTkU];
#pragma unroll
      for (int u = 0; u < kTkU; ++u) {
        const int vi = v0 + u * kTkThreads;
        if (vi < NV) buf[u] = ldg_v4_hint(row + (size_t)vi * VW, pol_first);
      }
#pragma unroll
      for (int u = 0; u < kTkU; ++u) {
        const int vi = v0 + u * kTkThreads;
        if (vi < NV) {
          const float m = TR::template vmax<true>(buf[u]);
          if (!(m < tau)) {
#pragma unroll
            for (int t = 0; t < VW; ++t) {
              const float x = TR::get(buf[u], t);
              if (x != x) {
                nan_seen = 1;
              } else if (x >= tau) {
                const int pos = atomicAdd(&sm.wcount[warp], 1);
                if (pos < kTkWarpCap) wbuf[pos] = comp_key(x, vi * VW + t);
              }
            }
          }
        }
      }
    }
    const int bad_nan = __syncthreads_or(nan_seen);
    int overflow = 0, N = 0;
    for (int w = 0; w < kTkWarps; ++w) {
      overflow |= sm.wcount[w] > kTkWarpCap;
      N += min(sm.wcount[w], kTkWarpCap);
    }
    if (overflow) {
      // exact k-th largest (value, index) key by bisection over the row
      unsigned long long K64 = 0ull;
      for (int bit = 63; bit >= 0; --bit) {
        const unsigned long long Kt = K64 | (1ull << bit);
        int mine = 0;
        for (int vi = tid; vi < NV; vi += kTkThreads) {
          const uint4 v = ldg_v4(row + (size_t)vi * VW);
#pragma unroll
          for (int t = 0; t < VW; ++t) {
            const float x = TR::get(v, t);
            mine += (x == x && comp_key(x, vi * VW + t) >= Kt);
          }
        }
        if (block_sum_int_n(mine, sm.ired) >= k) K64 = Kt;
      }
      __syncthreads();
      if (tid == 0) sm.count = 0;
      __syncthreads();
      for (int vi = tid; vi < NV; vi += kTkThreads) {
        const uint4 v = ldg_v4(row + (size_t)vi * VW);
#pragma unroll
        for (int t = 0; t < VW; ++t) {
          const float x = TR::get(v, t);
          if (x == x) {
            const unsigned long long ck = comp_key(x, vi * VW + t);
            if (ck >= K64) {
              const int pos = atomicAdd(&sm.count, 1);
              if (pos < kTkCap) sm.cand[pos] = ck;
            }
          }
        }
      }
      __syncthreads();
      N = min(sm.count, kTkCap);
      // the candidates now sit contiguously in cand[0, N)
      for (int e = tid; e < N; e += kTkThreads) {
        const unsigned long long me = sm.cand[e];
        int rank = 0;
        for (int j = 0; j < N; ++j) rank += sm.cand[j] > me;
        if (rank < k) sm.sel[rank] = me;
      }
    } else {
      // rank the candidates held in the per-warp buffers
      for (int w = 0; w < kTkWarps; ++w) {
        const int cw = min(sm.wcount[w], kTkWarpCap);
        for (int s = tid; s < cw; s += kTkThreads) {
          const unsigned long long me = sm.cand[w * kTkWarpCap + s];
          int rank = 0;
          for (int w2 = 0; w2 < kTkWarps; ++w2) {
            const int c2 = min(sm.wcount[w2], kTkWarpCap);
            const unsigned long long* src = sm.cand + w2 * kTkWarpCap;
            for (int j = 0; j < c2; ++j) rank += src[j] > me;
          }
          if (rank < k) sm.sel[rank] = me;
        }
      }
    }
    __syncthreads();
    const int kk = min(k, N);

    // ---- softmax(./T) over the top-k, then the top-p cut (float64 sums)
    const float m0 = kk > 0 ? comp_val(sm.sel[0]) : -INFINITY;
    const bool bad = bad_nan || !(m0 > -INFINITY && m0 < INFINITY);
    for (int e = tid; e < kk; e += kTkThreads) {
      sm.w[e] = bad ? 0.0 : (double)exp2f((comp_val(sm.sel[e]) - m0) * p.c);
      sm.widx[e] = comp_idx(sm.sel[e]);
    }
    __syncthreads();
    if (warp == 0) {
      double W = 0.0;
      for (int e = lane; e < kk; e += 32) W += sm.w[e];
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) W += __shfl_xor_sync(0xffffffffu, W, m);
      int J = kk;
      double WJ = W;
      if (bad || kk == 0) {
        J = kk > 0 ? 1 : 0;
        WJ = 1.0;
        if (lane == 0 && kk > 0) sm.w[0] = 1.0;
      } else if (p.top_p < 1.0f) {
        const double target = (double)p.top_p * W;   // cum / W >= top_p
        double carry = 0.0;
        J = kk;
        for (int c0 = 0; c0 < kk; c0 += 32) {
          const int e = c0 + lane;
          const double we = e < kk ? sm.w[e] : 0.0;
          const double inc = carry + warp_incl_scan_d(we);
          const unsigned hit = __ballot_sync(0xffffffffu, e < kk && inc >= target);
          if (hit) {
            const int first = __ffs(hit) - 1;
            J = c0 + first + 1;
            WJ = __shfl_sync(0xffffffffu, inc, first);
            break;
          }
          carry = __shfl_sync(0xffffffffu, inc, 31);
        }
      }
      if (lane == 0) {
        sm.J = J;
        sm.WJ = WJ;
        if (bad) atomicOr(&p.seq[b].status, SEQ_BADROW);
      }
    }
    __syncthreads();
    const int J = sm.J;
    const double WJ = sm.WJ;
    int2* out = p.rowres + (size_t)r * (k + 1);
    if (tid == 0) out[0] = make_int2(J, 0);
    for (int e = tid; e < J; e += kTkThreads)
      out[1 + e] = make_int2(sm.widx[e], __float_as_int((float)(sm.w[e] / WJ)));
    // ---- acceptance probability of this row's draft
    if (i < G) {
      if (tid == 0) {
        sm.pd = 0.0;
        sm.token = d_row;
      }
      __syncthreads();
      const int d = sm.token;
      if (d >= 0 && d < V)
        for (int e = tid; e < J; e += kTkThreads)
          if (sm.widx[e] == d) sm.pd = sm.w[e] / WJ;
      __syncthreads();
      if (tid == 0) {
        double a = 0.0;
        int st = 0;
        if (d < 0 || d >= V) {
          st |= SEQ_OOB;
        } else {
          const double pd = sm.pd;
          const float qd = q_row;
          if (qd > 0.0f) {
            a = fmin(1.0, pd / (double)qd);
          } else {
            a = pd > 0.0 ? 1.0 : 0.0;
            st |= SEQ_QBAD;
          }
        }
        if (st) atomicOr(&p.seq[b].status, st);
        p.acc[b * G + i] = a;
        if (p.out_a) p.out_a[b * G + i] = (float)a;
      }
    }
    if (arrive_last(p.seq_ticket + b, G1, &sm.flag)) topk_finish_sequence(p, b, sm);
  }
}

}  // namespace sv
