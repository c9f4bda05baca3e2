// Latency path of libspecverify: one thread-block cluster per sequence.
//
// For small problems (a few sequences, every row of a sequence together a few
// hundred KB) the two-launch grid path is bound by launch and memory latency,
// not bandwidth.  Here one kernel does the whole step:
//
//   * the vocabulary is split over the CN (<= 16) CTAs of a cluster; each CTA
//     copies its slice of all gamma+1 logit rows - and, for sampling, of all
//     gamma q rows - into shared memory with cp.async, so every DRAM request
//     of the step is in flight at once;
//   * one warp per row reduces the slice (max / sum of 2^((L - m) c), or the
//     argmax) into a per-row partial in the CTA's shared memory;
//   * every CTA pushes its partials to all CTAs of the cluster; after a
//     cluster barrier each merges the CN partials of each row in rank order
//     (so all CTAs hold identical row statistics) and runs the acceptance
//     scan (the drafts' l(d_i), q(d_i) were loaded at the start);
//   * sampling: each thread sums (S, A, Q) of its run of the final-draw row
//     (residual max(p_n - q_n, 0), or p_gamma) and keeps them in registers;
//     the CTA's slice sums are pushed to all CTAs; after a second barrier warp
//     0 of every CTA forms the exact normaliser and agrees on the slice
//     holding the inverse-CDF step; its owner goes thread -> token with the
//     same sums.
//
// CTAs exchange data only by pushing it into each other's shared memory
// (distributed shared memory stores) before a cluster barrier and reading
// their own copy after it; no CTA reads another's shared memory, so a CTA may
// leave once the last barrier it takes part in has passed.  The barriers are
// hardware cluster barriers (barrier.cluster): every CTA of the cluster
// arrives at each of them unconditionally, so none can wait on a CTA that
// never arrives.  The first one (arrive at entry, wait before the first push)
// makes sure every CTA of the cluster runs before any remote store.
#pragma once

#include <cooperative_groups.h>

#include "sv_device.cuh"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kClusterMax = 16;
constexpr int kClusterMaxNS = 8;   // vectors per thread for a whole slice (final-draw runs <= 64 tokens)

struct ClusterParams {
  Params p;
  int CN;      // CTAs per cluster
  int W;       // slice width in elements (multiple of the vector width)
  int NS;      // vectors per thread for a whole slice (ceil(W / VW / 256))
  int EPT;     // final draw: tokens per thread run (NS * VW)
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

struct ClusterSmem {
  float tab[128];            // exp2_f2 table
  float4 allpart[kClusterMax][kMaxG1];   // every CTA's per-row partial (pushed by its owner):
                                         // (max, s_hi, s_lo) or (max, index)
  float ur[kMaxG1];          // this sequence's uniforms
  F2x3 allsub[kClusterMax];      // every CTA's (S, A, Q) of the final-draw row (pushed)
  F2x3 red[kWarps];
  F2 ds;
  float M[kMaxG1];
  double S[kMaxG1];
  float a[kMaxG1];
  int g[kMaxG1];
  int st[kMaxG1];          // per-row status bits
  int dr[kMaxG1];          // drafts with their logit and q value
  float dl[kMaxG1];
  float dq[kMaxG1];
  F2 f2red[kWarps];
  int n;
  int status;
  int use_p;
  int owner;      // rank owning the inverse-CDF step (-1 none)
  int othread;    // thread of the owner whose run holds it
  int lastpos;    // last thread with a positive mass
  int token;
  F2 base;
  F2 target;
  F2 tbase;       // the owning thread's exclusive prefix
};

// Merge the CN partials of row i held by lanes [0, CN) of a 16-lane group.
template <int MODE>
__device__ __forceinline__ float4 group_merge(float4 v, int CN, float c) {
  const int lane16 = threadIdx.x & 15;
  const bool live = lane16 < CN;
  if (MODE == MODE_GREEDY) {
    float bv = live ? v.x : -INFINITY;
    int bi = live ? __float_as_int(v.y) : 0x7fffffff;
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, m, 16);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, m, 16);
      if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    return make_float4(bv, __int_as_float(bi), 0.f, 0.f);
  }
  float M = live ? v.x : -INFINITY;
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m, 16));
  F2 s{0.f, 0.f};
  if (live && v.x > -INFINITY && M < INFINITY) {
    const float sc = exp2f((v.x - M) * c);
    s = f2_add(F2{v.y * sc, 0.f}, F2{v.z * sc, 0.f});
  }
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) {
    const F2 o{__shfl_xor_sync(0xffffffffu, s.hi, m, 16), __shfl_xor_sync(0xffffffffu, s.lo, m, 16)};
    s = f2_add(s, o);
  }
  return make_float4(M, s.hi, s.lo, 0.f);
}

// (S, A, Q) of one thread's run of the final-draw row held in shared memory
// (len tokens, a multiple of VW; q = nullptr for the bonus row or a
// deterministic draft, whose one-hot q is infinite at run offset xq - so that
// token is outside the residual support - and 0 elsewhere): the tail tokens
// in one sweep, the tokens near the maximum (bits of `top`) after.
// The tail sweep of a run for 16-bit logits (x - M exact): every token takes
// the same branch-free steps (the tail weight and its residual with one
// rounding); a token near the maximum (p > -8) adds nothing and is flagged.
// -inf is clamped to an exponent that ex2.approx flushes to 0.
template <typename T, bool USE_Q>
__device__ __forceinline__ uint64_t cluster_sweep16(const T* L, const float* Q, int xq, int len, float M, float c,
                                                    float c_lo, float s_a, RunAcc* acc) {
  constexpr int VW = Tr<T>::VW;
  uint64_t top = 0ull;
  for (int j = 0; j * VW < len; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(L + j * VW);
    float qv[VW];
#pragma unroll
    for (int h = 0; h < VW / 4; ++h) {
      const float4 q4 = (USE_Q && Q) ? *reinterpret_cast<const float4*>(Q + j * VW + 4 * h)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
      qv[4 * h + 0] = q4.x;
      qv[4 * h + 1] = q4.y;
      qv[4 * h + 2] = q4.z;
      qv[4 * h + 3] = q4.w;
    }
    uint32_t tv = 0u;
#pragma unroll
    for (int t = 0; t < VW; ++t) {
      const float dh = fmaxf(Tr<T>::get(v, t) - M, -1.0e4f);
      const float p = dh * c;
      const float e = fmaf(dh, c_lo, fmaf(dh, c, -p));
      const float y = ex2_approx(p);
      const bool near = p > -8.f;
      const float w = near ? 0.f : fmaf(y * 6.931471825e-01f, e, y);
      if (near) tv |= 1u << t;
      RunAcc::acc2(acc->sh, acc->sl, w, 0.f);
      if (USE_Q) {
        // on the residual support {w > s' q} (the sign of w - s' q rounded
        // once): w - s' q and q, else 0 (adding 0 leaves both sums as they were)
        const float qt = (j * VW + t == xq) ? INFINITY : qv[t];
        const float d = fmaf(-s_a, qt, w);
        RunAcc::acc2(acc->ah, acc->al, d > 0.f ? d : 0.f, 0.f);
        acc->q += d > 0.f ? qt : 0.f;
      }
    }
    top |= (uint64_t)tv << (j * VW);
  }
  return top;
}

template <typename T>
__device__ __forceinline__ void cluster_run(const T* L, const float* Q, int xq, int len, bool use_q, float M,
                                            float c, float c_lo, float s_a, RunAcc* acc, const float* tab) {
  constexpr int VW = Tr<T>::VW;
  constexpr bool EXACT = sizeof(T) == 2;
  uint64_t top = 0ull;
  if constexpr (EXACT) {
    top = use_q ? cluster_sweep16<T, true>(L, Q, xq, len, M, c, c_lo, s_a, acc)
                : cluster_sweep16<T, false>(L, Q, xq, len, M, c, c_lo, s_a, acc);
  } else {
    for (int j = 0; j * VW < len; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(L + j * VW);
      float qv[VW];
#pragma unroll
      for (int h = 0; h < VW / 4; ++h) {
        const float4 q4 = Q ? *reinterpret_cast<const float4*>(Q + j * VW + 4 * h) : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[4 * h + 0] = q4.x;
        qv[4 * h + 1] = q4.y;
        qv[4 * h + 2] = q4.z;
        qv[4 * h + 3] = q4.w;
      }
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        const float qt = (j * VW + t == xq) ? INFINITY : qv[t];
        if (run_tail<EXACT>(*acc, Tr<T>::get(v, t), qt, use_q, M, c, c_lo, s_a)) top |= 1ull << (j * VW + t);
      }
    }
  }
  while (top) {
    const int o = __ffsll((long long)top) - 1;
    top &= top - 1;
    const float x = Tr<T>::get(*reinterpret_cast<const uint4*>(L + (o / VW) * VW), o % VW);
    run_top<EXACT>(*acc, x, o == xq ? INFINITY : (Q ? Q[o] : 0.f), use_q, M, c, c_lo, s_a, tab);
  }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
cluster_kernel(const ClusterParams cp) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  const Params& p = cp.p;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ClusterSmem& sm = *reinterpret_cast<ClusterSmem*>(smem_raw);
  T* Ls = reinterpret_cast<T*>(smem_raw + ((sizeof(ClusterSmem) + 15) & ~size_t(15)));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CN = cp.CN, W = cp.W;
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / CN;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);   // this sequence's drafts (ragged rounds)
  const int v0 = rank * W;
  const int v1 = min(v0 + W, V);
  const int nvec = max(v1 - v0, 0) / VW;               // vectors in this slice (V % VW == 0 on this path)
  float* Qs = reinterpret_cast<float*>(Ls + (size_t)G1 * W);
  // distributed shared memory may only be written once every CTA of the
  // cluster runs: arrive now, wait just before the first remote store
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  load_exp2_table(sm.tab);

  // ---- issue every load of the step: logits slices, then q slices
  const T* Lg = static_cast<const T*>(p.logits) + (size_t)b * G1 * V;
  for (int i = 0; i < G1; ++i) {
    const T* src = Lg + (size_t)i * V + v0;
    T* dst = Ls + (size_t)i * W;
    for (int k = tid; k < nvec; k += kThreads) cp_async16(dst + k * VW, src + k * VW);
  }
  cp_async_commit();
  const int nq = max(v1 - v0, 0) / 4;
  if (MODE == MODE_SOFTMAX && p.q) {
    const float* Qg = p.q + (size_t)b * G * V;
    for (int i = 0; i < G; ++i) {
      const float* src = Qg + (size_t)i * V + v0;
      float* dst = Qs + (size_t)i * W;
      for (int k = tid; k < nq; k += kThreads) cp_async16(dst + k * 4, src + k * 4);
    }
  }
  cp_async_commit();
  // this sequence's drafts with their logit and q value (plain loads, in
  // flight together with the slices; every CTA needs them for the scan)
  int d_own = -1;
  uint32_t l_bits = 0u;   // the raw logit bits: converted where they are used
  float q_own = 0.f, u_own = 0.f;
  if (tid < gb) {
    d_own = __ldg(p.draft + b * G + tid);
    if (d_own >= 0 && d_own < V) {
      l_bits = Tr<T>::scalar_bits(Lg + (size_t)tid * V + d_own);
      if (MODE == MODE_SOFTMAX) q_own = p.q ? __ldg(p.q + ((size_t)b * G + tid) * V + d_own) : 1.f;
    }
  }
  if (MODE == MODE_SOFTMAX && tid < G1) u_own = __ldg(p.uniforms + b * G1 + tid);
  if (tid < G1) sm.ur[tid] = u_own;
  if (tid < G) sm.dr[tid] = d_own;
  cp_async_wait<1>();
  __syncthreads();

  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  // ---- per-row partials of this slice: one warp per row
  for (int i = warp; i < G1; i += kWarps) {
    const T* Lr = Ls + (size_t)i * W;
    if (MODE == MODE_GREEDY) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int k = lane; k < nvec; k += 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(Lr + k * VW);
        const float m = TR::template vmax<true>(v);
        if (argmax_better(m, 1, bv, 0) || bi == 0x7fffffff) {
#pragma unroll
          for (int t = VW - 1; t >= 0; --t) {
            const float x = TR::get(v, t);
            const bool hit = (m != m) ? (x != x) : (x == m);
            if (hit) { bv = m; bi = v0 + k * VW + t; }
          }
        }
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, m);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, m);
        if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      // push the row partial into every CTA of the cluster (lane r -> rank r)
      if (lane < CN) *cluster.map_shared_rank(&sm.allpart[rank][i], lane) = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
    } else {
      float M = -INFINITY;
      for (int k = lane; k < nvec; k += 32)
        M = fmaxf(M, TR::template vmax<false>(*reinterpret_cast<const uint4*>(Lr + k * VW)));
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
      float a[4] = {0.f, 0.f, 0.f, 0.f};   // independent chains
      if (M > -INFINITY) {
        const float Mc = M * p.c;
        for (int k = lane; k < nvec; k += 32) {
          const uint4 v = *reinterpret_cast<const uint4*>(Lr + k * VW);
#pragma unroll
          for (int t = 0; t < VW; ++t) a[t & 3] += ex2_approx(fmaf(TR::get(v, t), p.c, -Mc));
        }
      }
      F2 s{(a[0] + a[1]) + (a[2] + a[3]), 0.f};
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) s = f2_add(s, f2_shfl_xor(s, m));
      if (lane < CN) *cluster.map_shared_rank(&sm.allpart[rank][i], lane) = make_float4(M, s.hi, s.lo, 0.f);
    }
  }
  // the drafts' l(d_i), q(d_i): loaded at the start, consumed only now, so
  // their latency hides behind the slice loads and the row partials
  if (tid < G) {
    uint4 lv = make_uint4(0u, 0u, 0u, 0u);
    Tr<T>::put(lv, 0, l_bits);
    sm.dl[tid] = Tr<T>::get(lv, 0);
    sm.dq[tid] = q_own;
  }
  cluster.sync();

  // ---- merge the CN partials of every row (16 lanes per row); the merging
  // lane also forms the row's acceptance test, then warp 0 runs the scan
  for (int base = 0; base < G1; base += 2 * kWarps) {
    const int i = base + (tid >> 4);
    const bool rowok = i < G1;
    float4 v = make_float4(-INFINITY, 0.f, 0.f, 0.f);
    const int r = tid & 15;
    if (rowok && r < CN) v = sm.allpart[r][i];
    const float4 mg = group_merge<MODE>(v, CN, p.c);
    if (rowok && r == 0) {
      int st = 0;
      const int d = i < gb ? sm.dr[i] : 0;
      if (i < gb && (d < 0 || d >= V)) st |= SEQ_OOB;
      if (MODE == MODE_GREEDY) {
        const bool nan = mg.x != mg.x;
        const int bi = __float_as_int(mg.y);
        sm.g[i] = (nan || bi == 0x7fffffff) ? 0 : bi;
        if (nan && i <= gb) st |= SEQ_BADROW;
      } else {
        const double sd = (double)mg.y + (double)mg.z;
        const bool badrow = !(mg.x > -INFINITY && mg.x < INFINITY) || !(sd > 0.0 && sd < 1e300);
        sm.M[i] = mg.x;
        sm.S[i] = sd;
        if (badrow && i <= gb) st |= SEQ_BADROW;
        if (i < G) {
          float a = 0.f;
          if (i < gb && d >= 0 && d < V) {
            const float pd = badrow ? 0.f : exp2f((sm.dl[i] - mg.x) * p.c) / (float)sd;
            const float qd = sm.dq[i];
            if (qd > 0.0f) {
              a = fminf(1.f, pd / qd);
            } else {
              a = pd > 0.f ? 1.f : 0.f;
              st |= SEQ_QBAD;
            }
          }
          sm.a[i] = a;
        }
      }
      sm.st[i] = st;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int status = 0, n = gb;
    for (int c0 = 0; c0 < G1; c0 += 32) {
      const int i = c0 + lane;
      if (i <= gb) status |= sm.st[i];
      const bool rej = i < gb && (MODE == MODE_GREEDY ? sm.dr[i] != sm.g[i] : !(sm.ur[i] < sm.a[i]));
      const unsigned rb = __ballot_sync(0xffffffffu, rej);
      if (rb && n == gb) n = c0 + __ffs(rb) - 1;
    }
    status = __reduce_or_sync(0xffffffffu, status);
    if (lane == 0) {
      sm.n = n;
      sm.status = status;
      if (MODE == MODE_GREEDY) sm.token = sm.g[n];
    }
  }
  __syncthreads();
  const int n = sm.n;
  if (rank == 0) {
    for (int j = tid; j < G1; j += kThreads) {
      if (j < n) p.out_tokens[b * G1 + j] = sm.dr[j];
      else if (j > n) p.out_tokens[b * G1 + j] = -1;
      else if (MODE == MODE_GREEDY) p.out_tokens[b * G1 + j] = sm.token;
    }
    if (MODE == MODE_SOFTMAX && p.out_a)
      for (int j = tid; j < G; j += kThreads) p.out_a[b * G + j] = sm.a[j];
    if (tid == 0) {
      p.out_n[b] = n;
      if (MODE == MODE_GREEDY && p.out_status) p.out_status[b] = sm.status;
    }
  }
  if (MODE == MODE_GREEDY) {
    return;   // every remote access (the pushes) happened before the barrier
  }

  // ---- final draw: residual of row n, or the bonus from row gamma
  // (precise weights and the (S, A, Q) decomposition, as in final_draw_kernel;
  // thread t of a CTA owns the run of EPT tokens at t * EPT of its slice)
  const bool resid = n < gb;
  const bool bad = (sm.status & SEQ_BADROW) != 0;
  const T* Lf = Ls + (size_t)n * W;
  const float* Qf = (resid && p.q) ? Qs + (size_t)n * W : nullptr;
  // deterministic drafts (q == NULL): q_n is one-hot at d_n (slice index xq)
  const int xq = (resid && !p.q) ? sm.dr[n] - v0 : -1;
  const float M = sm.M[n];
  const float s_a = (float)sm.S[n];
  const int EPT = cp.EPT;
  const int r0 = tid * EPT;
  const int rlen = min(EPT, max(v1 - v0 - r0, 0));   // a multiple of VW
  int status = sm.status;
  cp_async_wait<0>();     // this thread's q copies have landed
  __syncthreads();        // ... and every thread's are visible to all
  // this thread's run sums stay in registers: the owner walks them again below
  RunAcc acc;
  acc.zero();
  if (!bad) cluster_run<T>(Lf + r0, Qf ? Qf + r0 : nullptr, xq - r0, rlen, resid, M, p.c, p.c_lo, s_a, &acc, sm.tab);
  {
    const F2x3 t = block_sum_f2x3_w0(F2x3{acc.S(), acc.A(), F2{acc.q, 0.f}}, sm.red);   // warp 0 pushes
    if (tid < CN) *cluster.map_shared_rank(&sm.allsub[rank], tid) = t;
  }
  cluster.sync();
  // warp 0 of every CTA: the exact normaliser s, the masses of the CN slices
  // (lane r = rank r) and the inverse-CDF step: the first slice whose
  // interval [prefix, prefix + mass) holds u * R (R = the total); if rounding
  // leaves none, the last slice with positive mass
  if (warp == 0) {
    F2 S_l{0.f, 0.f}, m_l{0.f, 0.f};
    float Q_l = 0.f;
    if (lane < CN) {
      const F2x3 r3 = sm.allsub[lane];
      S_l = r3.a;
      m_l = r3.b;
      Q_l = r3.c.hi;
    }
    const F2 sinc = warp_incl_scan_f2(S_l);
    const F2 s = F2{__shfl_sync(0xffffffffu, sinc.hi, 31), __shfl_sync(0xffffffffu, sinc.lo, 31)};
    const F2 ds = f2_add(s, F2{-s_a, 0.f});          // s - s', tiny
    bool use_q = resid;
    if (resid) {
      m_l = f2_add(m_l, f2_neg(f2_scale(ds, Q_l)));
      if (m_l.hi < 0.f) m_l = F2{0.f, 0.f};
    } else {
      m_l = S_l;
    }
    F2 inc = warp_incl_scan_f2(m_l);
    F2 R = F2{__shfl_sync(0xffffffffu, inc.hi, 31), __shfl_sync(0xffffffffu, inc.lo, 31)};
    if (resid && !bad && !f2_pos(R)) {
      // zero residual mass (only through rounding): draw from p_n instead
      status |= SEQ_RESID0;
      use_q = false;
      m_l = S_l;
      inc = sinc;
      R = s;
    }
    const F2 tgt = f2_scale(R, sm.ur[gb]);
    F2 excl = f2_shfl_up(inc, 1);
    if (lane == 0) excl = F2{0.f, 0.f};
    const bool live = lane < CN && f2_pos(m_l);
    const unsigned hit = __ballot_sync(0xffffffffu, live && !f2_lt(tgt, excl) && f2_lt(tgt, f2_add(excl, m_l)));
    const unsigned any = __ballot_sync(0xffffffffu, live);
    int sub = hit ? __ffs(hit) - 1 : (any ? 31 - __clz(any) : -1);
    if (bad || !f2_pos(R)) sub = -1;
    const int src = sub < 0 ? 0 : sub;
    const F2 base{__shfl_sync(0xffffffffu, excl.hi, src), __shfl_sync(0xffffffffu, excl.lo, src)};
    if (lane == 0) {
      sm.owner = sub;
      sm.base = base;
      sm.target = tgt;
      sm.token = -1;
      sm.use_p = use_q ? 0 : 1;
      sm.ds = ds;
      sm.othread = 0x7fffffff;
      sm.lastpos = -1;
      sm.status = status;
    }
  }
  __syncthreads();
  status = sm.status;
  if (sm.owner == rank) {
    const bool uq = sm.use_p == 0;
    F2 mine = acc.mass(uq, sm.ds);
    if (mine.hi < 0.f) mine = F2{0.f, 0.f};
    F2 total;
    const F2 ex = block_exclusive_f2(mine, sm.f2red, &total);
    const F2 tb = f2_add(sm.base, ex);
    const bool pos = f2_pos(mine);
    if (pos && !f2_lt(sm.target, tb) && f2_lt(sm.target, f2_add(tb, mine))) atomicMin(&sm.othread, tid);
    if (pos) atomicMax(&sm.lastpos, tid);
    __syncthreads();
    // rounding can leave no run above the target: take the last positive one
    const bool take_last = sm.othread == 0x7fffffff;
    const int owner_t = take_last ? sm.lastpos : sm.othread;
    if (tid == owner_t) sm.tbase = tb;
    __syncthreads();
    if (owner_t >= 0 && tid < 32) {
      // warp 0 walks the owning run, 32 tokens at a time
      const int o0 = owner_t * EPT;
      const int olen = min(EPT, max(v1 - v0 - o0, 0));
      F2 carry = sm.tbase;
      int pick = -1, lastp = -1;
      for (int c0 = 0; c0 < olen && pick < 0; c0 += 32) {
        const int e = o0 + c0 + lane;
        F2 m{0.f, 0.f};
        if (c0 + lane < olen) {
          const float x = TR::get(*reinterpret_cast<const uint4*>(Lf + (e / VW) * VW), e % VW);
          const float qv = uq ? (Qf ? Qf[e] : (e == xq ? INFINITY : 0.f)) : 0.f;
          m = token_mass<sizeof(T) == 2>(x, qv, uq, M, p.c, p.c_lo, s_a, sm.ds, sm.tab);
        }
        const F2 inc = warp_incl_scan_f2(m);
        F2 excl = f2_shfl_up(inc, 1);
        if (lane == 0) excl = F2{0.f, 0.f};
        const F2 lb = f2_add(carry, excl);
        const bool live = f2_pos(m);
        const unsigned hit = __ballot_sync(0xffffffffu, live && !take_last && !f2_lt(sm.target, lb) &&
                                                            f2_lt(sm.target, f2_add(lb, m)));
        const unsigned any = __ballot_sync(0xffffffffu, live);
        if (hit) pick = c0 + __ffs(hit) - 1;
        if (any) lastp = c0 + 31 - __clz(any);
        const F2 tot = F2{__shfl_sync(0xffffffffu, inc.hi, 31), __shfl_sync(0xffffffffu, inc.lo, 31)};
        carry = f2_add(carry, tot);
      }
      if (pick < 0) pick = lastp;
      if (lane == 0) sm.token = pick >= 0 ? v0 + o0 + pick : -1;
    }
    __syncthreads();
    if (tid == 0) {
      p.out_tokens[b * G1 + n] = sm.token < 0 ? 0 : sm.token;
      if (p.out_status) p.out_status[b] = status;
    }
  } else if (sm.owner < 0 && rank == 0 && tid == 0) {
    p.out_tokens[b * G1 + n] = 0;
    if (p.out_status) p.out_status[b] = status;
  }
}

}  // namespace sv
