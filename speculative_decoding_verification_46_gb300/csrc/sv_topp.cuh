// Top-p without top-k, for any vocabulary ("11.1 核心原理", section 11.1.2:
// top-p is applied to p before the test; the kept set is the shortest prefix
// of the ranking by (logit descending, index ascending) whose renormalised
// mass reaches top_p, the crossing token included).
//
// topp_row_kernel: one CTA per row of logits.  The kept set is
//   { v : key(v) > K }  U  { v : key(v) = K and v <= idx }
// with key the order-preserving key of the logit.  K and idx are found
// exactly, without sorting:
//   1. the row maximum M (a row holding NaN or +inf, or only -inf, defines no
//      distribution);
//   2. mass-weighted bisection over the key: each pass reads the row, adds
//      the weight w = 2^((x - M) c) of every token whose key lies in the
//      current key range into one of 16 buckets (a thread-private column of a
//      shared-memory histogram: no atomics, a fixed order of additions), sums
//      the columns in two-float and keeps the bucket where the mass above it
//      plus the bucket's own first reaches top_p * (total); 4 key bits per
//      pass until a single key K remains (bf16: 4 passes; float16 5; float32
//      8);
//   3. the tokens with key K all have one weight w_K: the first
//      j = ceil((top_p * total - mass above K) / w_K) of them in index order
//      are kept (a block scan of per-thread counts over contiguous index
//      ranges finds the j-th), idx = its index.
// The kept mass W (two-float), and for a drafted row its acceptance
// probability a_i = min(1, (w(d_i) / W) / q_i(d_i)) (0 if d_i is not kept),
// go to the row's record; final_draw_kernel<T, true> then scans, and draws
// from max(p~_n - q_n, 0) (or p~_gamma) with the same mask.
#pragma once

#include <cooperative_groups.h>

#include "sv_device.cuh"

namespace sv {

constexpr int kTpThreads = 512;
constexpr int kTpBits = 4;
constexpr int kTpBuckets = 1 << kTpBits;
constexpr int kTpU = 8;   // vectors per thread whose loads are in flight together

// Per-row result of topp_row_kernel.
struct TpRow {
  float M;         // row maximum
  uint32_t K;      // crossing key (okey(x) >> KEY_LOW_BIT)
  int idx;         // last kept index among the tokens with key K
  float a;         // acceptance probability of the row's draft (rows i < gamma_b)
  float Wh, Wl;    // kept mass: sum over kept v of 2^((x_v - M) c), two-float
  int status;      // SEQ_OOB / SEQ_QBAD of the row's test; SEQ_BADROW
  int pad;
};

struct TpSmem {
  float hist[kTpBuckets][kTpThreads];   // thread-private bucket columns
  F2 tot[kTpBuckets];
  F2 wred[kTpThreads / 32];
  float fred[kTpThreads / 32];
  int ired[kTpThreads / 32];
  uint32_t lo;
  int width, pick, bad;
  F2 above;
  int cnt_base[kTpThreads / 32];
  int idx;
  float weq;
};

// Order-preserving key of a logit of type T (the bits that can differ).
template <typename T>
__device__ __forceinline__ uint32_t tp_key(float x) {
  return okey(x) >> Tr<T>::KEY_LOW_BIT;
}
// A conservative test of a whole 16-byte vector against a key range
// [klo, khi]: false only when none of its values can have a key in the
// range.  Bounds are the range's end values rounded outwards to T (keys past
// those of -inf / +inf open the bound), compared with native packed compares,
// so that a pass skips the vectors outside its range for a few instructions
// per 8 logits; the exact key test stays with the tokens that pass.
template <typename T>
struct TpFilter;
template <>
struct TpFilter<float> {
  float lo, hi;
  __device__ __forceinline__ void set(float flo, float fhi) {
    lo = flo;
    hi = fhi;
  }
  __device__ __forceinline__ bool any(const uint4& v) const {
    const float a = __uint_as_float(v.x), b = __uint_as_float(v.y), c = __uint_as_float(v.z), d = __uint_as_float(v.w);
    return (a >= lo && a <= hi) || (b >= lo && b <= hi) || (c >= lo && c <= hi) || (d >= lo && d <= hi);
  }
};
template <>
struct TpFilter<__nv_bfloat16> {
  __nv_bfloat162 lo, hi;
  __device__ __forceinline__ void set(float flo, float fhi) {
    lo = __bfloat162bfloat162(__float2bfloat16_rd(flo));
    hi = __bfloat162bfloat162(__float2bfloat16_ru(fhi));
  }
  __device__ __forceinline__ bool any(const uint4& v) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    unsigned m = 0u;
#pragma unroll
    for (int t = 0; t < 4; ++t) m |= __hge2_mask(h[t], lo) & __hle2_mask(h[t], hi);
    return m != 0u;
  }
};
template <>
struct TpFilter<__half> {
  __half2 lo, hi;
  __device__ __forceinline__ void set(float flo, float fhi) {
    lo = __half2half2(__float2half_rd(flo));
    hi = __half2half2(__float2half_ru(fhi));
  }
  __device__ __forceinline__ bool any(const uint4& v) const {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
    unsigned m = 0u;
#pragma unroll
    for (int t = 0; t < 4; ++t) m |= __hge2_mask(h[t], lo) & __hle2_mask(h[t], hi);
    return m != 0u;
  }
};
// The logit whose key (okey >> KEY_LOW_BIT) is k: the dropped low bits of an
// order-preserving key are all ones for a negative value, zeros otherwise.
template <typename T>
__device__ __forceinline__ float tp_key_value(uint32_t k) {
  constexpr int LOW = Tr<T>::KEY_LOW_BIT;
  const uint32_t full = (k << LOW) | ((k >> (31 - LOW)) & 1u ? 0u : (uint32_t)((1ull << LOW) - 1));
  return key_to_float(full);
}
template <typename T>
__device__ __forceinline__ TpFilter<T> tp_filter(uint32_t klo, uint32_t khi) {
  constexpr int LOW = Tr<T>::KEY_LOW_BIT;
  const uint32_t kninf = okey(-INFINITY) >> LOW, kpinf = okey(INFINITY) >> LOW;
  const float flo = klo <= kninf ? -INFINITY : tp_key_value<T>(klo);
  const float fhi = khi >= kpinf ? INFINITY : tp_key_value<T>(khi);
  TpFilter<T> f;
  f.set(flo, fhi);
  return f;
}

// Is token v (logit x) in the kept set (K, idx)?
template <typename T>
__device__ __forceinline__ bool tp_kept(float x, int v, uint32_t K, int idx) {
  const uint32_t k = tp_key<T>(x);
  return k > K || (k == K && v <= idx);
}

template <typename T>
__global__ void __launch_bounds__(kTpThreads) topp_row_kernel(const Params p, TpRow* rows) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  constexpr int NB = 32 - TR::KEY_LOW_BIT;   // key bits
  extern __shared__ __align__(16) unsigned char tp_dyn[];
  TpSmem& sm = *reinterpret_cast<TpSmem*>(tp_dyn);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = kTpThreads / 32;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int r = blockIdx.x;
  const int b = r / G1, i = r - b * G1;
  const int gb = seq_gamma(p, b);
  if (i > gb) return;   // not part of this round (uniform over the block)
  const T* row = static_cast<const T*>(p.logits) + (size_t)r * V;
  const bool vec = (V % VW) == 0;
  const int NVv = (V + VW - 1) / VW;   // 16-byte slots (the last one partial when !vec)
  auto slot = [&](int j) -> uint4 {
    const int e = j * VW;
    const int nv = min(VW, V - e);
    return load_slot<T>(row, e, nv, vec && nv == VW);
  };
  // the row in batches of kTpU vectors per thread, their loads issued
  // together (the passes re-read the row from L2; one load at a time per
  // thread would leave them latency-bound)
  auto sweep = [&](auto&& body) {
    for (int j0 = tid; j0 < NVv; j0 += kTpThreads * kTpU) {
      uint4 x[kTpU];
#pragma unroll
      for (int u = 0; u < kTpU; ++u) {
        const int j = j0 + u * kTpThreads;
        x[u] = j < NVv ? slot(j) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kTpU; ++u) {
        const int j = j0 + u * kTpThreads;
        if (j < NVv) body(j, x[u]);
      }
    }
  };
  // the draft's inputs, before anything else (their loads overlap the passes)
  int d = -1;
  float qd = 0.f, ld = 0.f;
  if (tid == 0 && i < gb) {
    d = __ldg(p.draft + b * G + i);
    if (d >= 0 && d < V) {
      ld = TR::get(load_slot<T>(row, d, 1, false), 0);
      qd = p.q ? __ldg(p.q + ((size_t)b * G + i) * V + d) : 1.f;   // NULL: one-hot draft
    }
  }
  // ---- 1. maximum; NaN / +inf / only -inf: no distribution
  float m = -INFINITY;
  int nan = 0;
  sweep([&](int j, const uint4& v) {
    const float vm = TR::template vmax<true>(v);
    nan |= (vm != vm);
    m = fmaxf(m, vm);
  });
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    nan |= __shfl_xor_sync(0xffffffffu, nan, o);
  }
  if (lane == 0) {
    sm.fred[warp] = m;
    sm.ired[warp] = nan;
  }
  __syncthreads();
  float M = sm.fred[0];
  int anynan = sm.ired[0];
  for (int w = 1; w < nw; ++w) {
    M = fmaxf(M, sm.fred[w]);
    anynan |= sm.ired[w];
  }
  const bool bad = anynan || !(M > -INFINITY && M < INFINITY);
  if (bad) {
    if (tid == 0) {
      TpRow o{};
      o.M = 0.f;
      o.a = 0.f;
      o.status = SEQ_BADROW | ((i < gb && (d < 0 || d >= V)) ? SEQ_OOB : 0);
      rows[r] = o;
    }
    return;
  }
  const float Mc = M * p.c;
  // ---- 2. mass-weighted bisection over the key
  uint32_t lo = 0u;
  int width = NB;
  F2 above{0.f, 0.f};
  F2 total{0.f, 0.f};
  F2 target{0.f, 0.f};
  bool first = true;
  while (width > 0) {
    const int bits = min(kTpBits, width);
    const int sh = width - bits;
    const uint64_t span = 1ull << width;
#pragma unroll
    for (int k = 0; k < kTpBuckets; ++k) sm.hist[k][tid] = 0.f;
    sweep([&](int j, const uint4& v) {
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        if (j * VW + t < V) {
          const float x = TR::get(v, t);
          const uint32_t key = tp_key<T>(x);
          if (key >= lo && (uint64_t)(key - lo) < span) {
            const float w = ex2_approx(fmaf(x, p.c, -Mc));
            sm.hist[(key - lo) >> sh][tid] += w;
          }
        }
      }
    });
    __syncthreads();
    // bucket totals: warp w sums bucket w (nw == kTpBuckets) over the columns
    {
      F2 acc{0.f, 0.f};
      for (int c = lane; c < kTpThreads; c += 32) acc = f2_add(acc, F2{sm.hist[warp][c], 0.f});
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc = f2_add(acc, f2_shfl_xor(acc, o));
      if (lane == 0) sm.tot[warp] = acc;
    }
    __syncthreads();
    if (first) {
      // the first pass covers every key: the row's total mass
      total = F2{0.f, 0.f};
      for (int k = 0; k < kTpBuckets; ++k) total = f2_add(total, sm.tot[k]);
      target = f2_scale(total, p.top_p);
      first = false;
    }
    // the crossing bucket, from the top: the first whose mass, added to the
    // mass above it, reaches the target (if rounding leaves none, the lowest
    // bucket with mass)
    int pick = -1, lowest = 0;
    F2 cum = above, cum_low = above;
    for (int k = (1 << bits) - 1; k >= 0; --k) {
      if (f2_pos(sm.tot[k])) {
        lowest = k;
        cum_low = cum;
      }
      const F2 nc = f2_add(cum, sm.tot[k]);
      if (!f2_lt(nc, target)) {
        pick = k;
        break;
      }
      cum = nc;
    }
    if (pick < 0) {
      pick = lowest;
      cum = cum_low;
    }
    above = cum;
    lo += (uint32_t)pick << sh;
    width = sh;
    __syncthreads();   // every thread has read tot before the next pass writes hist
  }
  const uint32_t K = lo;
  // ---- 3. ties at K: the j-th in index order; contiguous ranges of whole
  // vectors per thread (token order), loaded kTpU at a time
  const int Lv = (NVv + kTpThreads - 1) / kTpThreads;
  const int j0 = min(tid * Lv, NVv), j1 = min(j0 + Lv, NVv);
  // visit(e, x) for every token e of this thread's range in order; stops when it returns true
  auto ranged = [&](auto&& visit) {
    for (int jb = j0; jb < j1; jb += kTpU) {
      uint4 xv[kTpU];
#pragma unroll
      for (int u = 0; u < kTpU; ++u) xv[u] = jb + u < j1 ? slot(jb + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < kTpU; ++u) {
        if (jb + u < j1) {
#pragma unroll
          for (int t = 0; t < VW; ++t) {
            const int e = (jb + u) * VW + t;
            if (e < V && visit(e, TR::get(xv[u], t))) return;
          }
        }
      }
    }
  };
  int cnt = 0;
  float weq = 0.f;
  ranged([&](int e, float x) {
    if (tp_key<T>(x) == K) {
      ++cnt;
      weq = ex2_approx(fmaf(x, p.c, -Mc));
    }
    return false;
  });
  // exclusive prefix of the counts
  int inc = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sm.ired[warp] = inc;
  if (cnt > 0) sm.weq = weq;   // every tied token has this weight
  if (tid == 0) sm.idx = V - 1;
  __syncthreads();
  int base = 0, neq = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) base += sm.ired[w];
    neq += sm.ired[w];
  }
  base += inc - cnt;
  const float wK = sm.weq;
  const F2 need = f2_add(target, f2_neg(above));
  int jk = (int)ceilf((need.hi + need.lo) / wK);
  jk = max(1, min(jk, neq));
  // the thread holding the jk-th tied token finds its index
  if (cnt > 0 && base < jk && jk <= base + cnt) {
    int seen = base;
    ranged([&](int e, float x) {
      if (tp_key<T>(x) == K && ++seen == jk) {
        sm.idx = e;
        return true;
      }
      return false;
    });
  }
  __syncthreads();
  if (tid == 0) {
    const int idx = sm.idx;
    const F2 W = f2_add(above, f2_scale(F2{wK, 0.f}, (float)jk));
    TpRow o{};
    o.M = M;
    o.K = K;
    o.idx = idx;
    o.Wh = W.hi;
    o.Wl = W.lo;
    int st = 0;
    float a = 0.f;
    if (i < gb) {
      if (d < 0 || d >= V) {
        st |= SEQ_OOB;
      } else {
        const bool kept = tp_kept<T>(ld, d, K, idx);
        const float pd = kept ? exp2f((ld - M) * p.c) / (W.hi + W.lo) : 0.f;
        if (qd > 0.f) {
          a = fminf(1.f, pd / qd);
        } else {
          a = pd > 0.f ? 1.f : 0.f;
          st |= SEQ_QBAD;
        }
      }
    }
    o.a = a;
    o.status = st;
    rows[r] = o;
  }
}


// ---- cluster variant: the same kept set, with a row's logits resident in
// the shared memory of a thread-block cluster of C CTAs.  Rank c holds the
// tokens [c Vc, min(V, (c + 1) Vc)) (Vc a multiple of the 16-byte vector),
// loaded from HBM once; the bisection and tie passes read shared memory.
// Each pass's bucket totals, the slice maxima and the tie counts are pushed
// to every CTA of the cluster (distributed shared memory) and summed in rank
// order, so that every CTA takes the same decisions from the same numbers.
// Passes after the first skip the vectors outside their key range with the
// packed test (TpFilter).  Rank 0 writes the row's record.
constexpr int kTcMaxC = 8;                  // CTAs per cluster (portable size)
constexpr int kTcSliceBytes = 64 << 10;     // a CTA's share of the row: two CTAs per SM

struct TcSmem {
  float hist[kTpBuckets][kTpThreads];       // thread-private bucket columns
  F2 ctot[2][kTcMaxC][kTpBuckets];          // bucket totals by rank, by pass parity
  F2 tot[kTpBuckets];                       // the cluster's bucket totals
  float cmax[kTcMaxC];                      // slice maxima by rank
  int cnan[kTcMaxC];
  int ccnt[kTcMaxC];                        // tie counts by rank
  float fred[kTpThreads / 32];
  int ired[kTpThreads / 32];
  int cidx;                                 // rank 0: the index of the chosen tie
};
__host__ __device__ constexpr size_t tc_head_bytes() { return (sizeof(TcSmem) + 127) & ~(size_t)127; }

template <typename T>
__global__ void __launch_bounds__(kTpThreads, 2) topp_cluster_kernel(const Params p, TpRow* rows, int Vc) {
  namespace cg = cooperative_groups;
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  constexpr int NB = 32 - TR::KEY_LOW_BIT;
  extern __shared__ __align__(128) unsigned char tc_dyn[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(tc_dyn);
  uint4* sl = reinterpret_cast<uint4*>(tc_dyn + tc_head_bytes());
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = kTpThreads / 32;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int r = (int)blockIdx.x / C;
  const int b = r / G1, i = r - b * G1;
  const int gb = seq_gamma(p, b);
  if (i > gb) return;   // not part of this round (uniform over the cluster)
  const T* row = static_cast<const T*>(p.logits) + (size_t)r * V;
  const int e0 = min(V, rank * Vc), e1 = min(V, e0 + Vc);
  const int nvec = (e1 - e0) / VW;   // V and Vc are multiples of VW
  // the draft's inputs (rank 0), before anything else
  int d = -1;
  float qd = 0.f, ld = 0.f;
  if (rank == 0 && tid == 0 && i < gb) {
    d = __ldg(p.draft + b * G + i);
    if (d >= 0 && d < V) {
      ld = TR::get(load_slot<T>(row, d, 1, false), 0);
      qd = p.q ? __ldg(p.q + ((size_t)b * G + i) * V + d) : 1.f;   // NULL: one-hot draft
    }
  }
  // ---- 1. the slice into shared memory (kTpU loads in flight per thread) and its maximum
  float m = -INFINITY;
  int nan = 0;
  for (int j0 = tid; j0 < nvec; j0 += kTpThreads * kTpU) {
    uint4 x[kTpU];
#pragma unroll
    for (int u = 0; u < kTpU; ++u) {
      const int j = j0 + u * kTpThreads;
      x[u] = j < nvec ? ldg_v4(row + e0 + (size_t)j * VW) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kTpU; ++u) {
      const int j = j0 + u * kTpThreads;
      if (j < nvec) {
        sl[j] = x[u];
        const float vm = TR::template vmax<true>(x[u]);
        nan |= (vm != vm);
        m = fmaxf(m, vm);
      }
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    nan |= __shfl_xor_sync(0xffffffffu, nan, o);
  }
  if (lane == 0) {
    sm.fred[warp] = m;
    sm.ired[warp] = nan;
  }
  __syncthreads();
  if (warp == 0) {
    float mc = lane < nw ? sm.fred[lane] : -INFINITY;
    int nc = lane < nw ? sm.ired[lane] : 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
      nc |= __shfl_xor_sync(0xffffffffu, nc, o);
    }
    if (lane < C) {
      *cl.map_shared_rank(&sm.cmax[rank], lane) = mc;
      *cl.map_shared_rank(&sm.cnan[rank], lane) = nc;
    }
  }
  if (rank == 0 && tid == 0) sm.cidx = V - 1;   // the chosen tie's index unless a rank reports it
  cl.sync();
  float M = sm.cmax[0];
  int anynan = sm.cnan[0];
  for (int c = 1; c < C; ++c) {
    M = fmaxf(M, sm.cmax[c]);
    anynan |= sm.cnan[c];
  }
  const bool bad = anynan || !(M > -INFINITY && M < INFINITY);
  if (bad) {
    if (rank == 0 && tid == 0) {
      TpRow o{};
      o.M = 0.f;
      o.a = 0.f;
      o.status = SEQ_BADROW | ((i < gb && (d < 0 || d >= V)) ? SEQ_OOB : 0);
      rows[r] = o;
    }
    return;   // (no shared-memory traffic between the CTAs after the barrier)
  }
  const float Mc = M * p.c;
  // ---- 2. mass-weighted bisection over the key, on the resident slice
  uint32_t lo = 0u;
  int width = NB;
  F2 above{0.f, 0.f};
  F2 total{0.f, 0.f};
  F2 target{0.f, 0.f};
  bool first = true;
  int pass = 0;
  while (width > 0) {
    const int bits = min(kTpBits, width);
    const int sh = width - bits;
    const uint64_t span = 1ull << width;
#pragma unroll
    for (int k = 0; k < kTpBuckets; ++k) sm.hist[k][tid] = 0.f;
    if (first) {
      // every key is in range (lo = 0)
      for (int j = tid; j < nvec; j += kTpThreads) {
        const uint4 v = sl[j];
#pragma unroll
        for (int t = 0; t < VW; ++t) {
          const float x = TR::get(v, t);
          sm.hist[tp_key<T>(x) >> sh][tid] += ex2_approx(fmaf(x, p.c, -Mc));
        }
      }
    } else {
      const TpFilter<T> flt = tp_filter<T>(lo, (uint32_t)((uint64_t)lo + span - 1));
      for (int j = tid; j < nvec; j += kTpThreads) {
        const uint4 v = sl[j];
        if (!flt.any(v)) continue;
#pragma unroll
        for (int t = 0; t < VW; ++t) {
          const float x = TR::get(v, t);
          const uint32_t key = tp_key<T>(x);
          if (key >= lo && (uint64_t)(key - lo) < span) {
            const float w = ex2_approx(fmaf(x, p.c, -Mc));
            sm.hist[(key - lo) >> sh][tid] += w;
          }
        }
      }
    }
    __syncthreads();
    // this CTA's bucket totals (warp w sums bucket w over the columns), pushed to every rank
    {
      F2 a0{0.f, 0.f}, a1{0.f, 0.f};   // two chains: half the dependent additions
      for (int c = lane; c < kTpThreads; c += 64) {
        a0 = f2_add(a0, F2{sm.hist[warp][c], 0.f});
        a1 = f2_add(a1, F2{sm.hist[warp][c + 32], 0.f});
      }
      F2 acc = f2_add(a0, a1);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc = f2_add(acc, f2_shfl_xor(acc, o));
      if (lane < C) *cl.map_shared_rank(&sm.ctot[pass & 1][rank][warp], lane) = acc;
    }
    cl.sync();
    if (tid < kTpBuckets) {
      F2 t = sm.ctot[pass & 1][0][tid];
      for (int c = 1; c < C; ++c) t = f2_add(t, sm.ctot[pass & 1][c][tid]);
      sm.tot[tid] = t;
    }
    __syncthreads();
    // the crossing bucket, in every warp at once: lane l holds bucket 15 - l
    // (from the top), a two-float scan gives the mass above each bucket and
    // through it; the pick is the first bucket whose cumulative mass reaches
    // the target (if rounding leaves none, the lowest bucket with mass)
    const F2 tk = lane < kTpBuckets ? sm.tot[kTpBuckets - 1 - lane] : F2{0.f, 0.f};
    const F2 inc = warp_incl_scan_f2(tk);
    if (first) {
      total = F2{__shfl_sync(0xffffffffu, inc.hi, kTpBuckets - 1), __shfl_sync(0xffffffffu, inc.lo, kTpBuckets - 1)};
      target = f2_scale(total, p.top_p);
      first = false;
    }
    F2 excl{__shfl_up_sync(0xffffffffu, inc.hi, 1), __shfl_up_sync(0xffffffffu, inc.lo, 1)};
    if (lane == 0) excl = F2{0.f, 0.f};
    const F2 cin = f2_add(above, inc), cex = f2_add(above, excl);
    const unsigned hit = __ballot_sync(0xffffffffu, lane < kTpBuckets && !f2_lt(cin, target));
    const unsigned pos = __ballot_sync(0xffffffffu, lane < kTpBuckets && f2_pos(tk));
    const int pl = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    const int pick = pl >= 0 ? kTpBuckets - 1 - pl : 0;
    if (pl >= 0) above = F2{__shfl_sync(0xffffffffu, cex.hi, pl), __shfl_sync(0xffffffffu, cex.lo, pl)};
    lo += (uint32_t)pick << sh;
    width = sh;
    ++pass;
    __syncthreads();   // every thread has read tot (and its columns) before the next pass
  }
  const uint32_t K = lo;
  const float wK = ex2_approx(fmaf(tp_key_value<T>(K), p.c, -Mc));   // the weight of every tied token
  // ---- 3. ties at K: contiguous runs of the slice's vectors per thread (token order)
  const TpFilter<T> keq = tp_filter<T>(K, K);
  const int Lv = (nvec + kTpThreads - 1) / kTpThreads;
  const int j0 = min(tid * Lv, nvec), j1 = min(j0 + Lv, nvec);
  int cnt = 0;
  for (int j = j0; j < j1; ++j) {
    const uint4 v = sl[j];
    if (!keq.any(v)) continue;
#pragma unroll
    for (int t = 0; t < VW; ++t) cnt += tp_key<T>(TR::get(v, t)) == K;
  }
  int inc = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sm.ired[warp] = inc;
  __syncthreads();
  int base = 0, ctot = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) base += sm.ired[w];
    ctot += sm.ired[w];
  }
  base += inc - cnt;
  if (tid < C) *cl.map_shared_rank(&sm.ccnt[rank], tid) = ctot;
  cl.sync();
  int rbase = 0, neq = 0;
  for (int c = 0; c < C; ++c) {
    if (c < rank) rbase += sm.ccnt[c];
    neq += sm.ccnt[c];
  }
  const F2 need = f2_add(target, f2_neg(above));
  int jk = (int)ceilf((need.hi + need.lo) / wK);
  jk = max(1, min(jk, neq));
  // the thread holding the jk-th tied token reports its index to rank 0
  if (cnt > 0 && rbase + base < jk && jk <= rbase + base + cnt) {
    int seen = rbase + base;
    for (int j = j0; j < j1; ++j) {
      const uint4 v = sl[j];
      bool done = false;
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        if (!done && tp_key<T>(TR::get(v, t)) == K && ++seen == jk) {
          *cl.map_shared_rank(&sm.cidx, 0) = e0 + j * VW + t;
          done = true;
        }
      }
      if (done) break;
    }
  }
  cl.sync();
  if (rank == 0 && tid == 0) {
    const int idx = sm.cidx;
    const F2 W = f2_add(above, f2_scale(F2{wK, 0.f}, (float)jk));
    TpRow o{};
    o.M = M;
    o.K = K;
    o.idx = idx;
    o.Wh = W.hi;
    o.Wl = W.lo;
    int st = 0;
    float a = 0.f;
    if (i < gb) {
      if (d < 0 || d >= V) {
        st |= SEQ_OOB;
      } else {
        const bool kept = tp_kept<T>(ld, d, K, idx);
        const float pd = kept ? exp2f((ld - M) * p.c) / (W.hi + W.lo) : 0.f;
        if (qd > 0.f) {
          a = fminf(1.f, pd / qd);
        } else {
          a = pd > 0.f ? 1.f : 0.f;
          st |= SEQ_QBAD;
        }
      }
    }
    o.a = a;
    o.status = st;
    rows[r] = o;
  }
}

}  // namespace sv
