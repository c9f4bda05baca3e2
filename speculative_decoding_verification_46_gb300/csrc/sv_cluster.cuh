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
//   * after a cluster barrier every CTA reads the CN partials of each row
//     through distributed shared memory, merges them in rank order (so all
//     CTAs hold identical row statistics), gathers l(d_i) and q(d_i) from the
//     owning CTA and runs the acceptance scan;
//   * sampling: each CTA sums the residual max(p_n - q_n, 0) (or p_gamma) over
//     its slice in 256-vector sub-ranges; after a second barrier the CTAs read
//     all sub-range masses, agree on the sub-range holding the inverse-CDF
//     step, and its owner walks it thread -> element with the same float32
//     partials.  A last barrier keeps every CTA's shared memory alive until
//     the others have finished reading it.
//
// The barriers are hardware cluster barriers (barrier.cluster): every CTA of
// the cluster arrives at each of them unconditionally, so none can wait on a
// CTA that never arrives.
#pragma once

#include <cooperative_groups.h>

#include "sv_device.cuh"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kClusterMax = 16;
constexpr int kClusterMaxNS = 8;   // 256-vector sub-ranges per CTA slice

struct ClusterParams {
  Params p;
  int CN;      // CTAs per cluster
  int W;       // slice width in elements (multiple of the vector width)
  int NS;      // sub-ranges of 256 vectors per slice
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

struct ClusterSmem {
  float4 part[kMaxG1];       // this CTA's per-row partial: (max, s_hi, s_lo) or (max, index)
  float ur[kMaxG1];          // this sequence's uniforms
  F2x3 sub3[kClusterMaxNS];                // this CTA's (S, A, Q) per sub-range
  F2 allmass[kClusterMax * kClusterMaxNS]; // every CTA's masses, in index order
  F2 allS[kClusterMax * kClusterMaxNS];
  float allQ[kClusterMax * kClusterMaxNS];
  F2x3 red[kWarps];
  F2 ds;
  float M[kMaxG1];
  double S[kMaxG1];
  float a[kMaxG1];
  int g[kMaxG1];
  int st[kMaxG1];
  int bad[kMaxG1];
  F2 f2red[kWarps];
  int n;
  int status;
  int use_p;
  int owner;      // rank owning the inverse-CDF step (-1 none)
  int sub;
  int token;
  F2 base;
  F2 target;
  LocateSmem loc;
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
  const int v0 = rank * W;
  const int v1 = min(v0 + W, V);
  const int nvec = max(v1 - v0, 0) / VW;               // vectors in this slice (V % VW == 0 on this path)
  float* Qs = reinterpret_cast<float*>(Ls + (size_t)G1 * W);

  // ---- issue every load of the step: logits slices, then q slices
  const T* Lg = static_cast<const T*>(p.logits) + (size_t)b * G1 * V;
  for (int e = tid; e < G1 * nvec; e += kThreads) {
    const int i = e / nvec, k = e - i * nvec;
    cp_async16(Ls + (size_t)i * W + k * VW, Lg + (size_t)i * V + v0 + k * VW);
  }
  cp_async_commit();
  const int nq = max(v1 - v0, 0) / 4;
  if (MODE == MODE_SOFTMAX) {
    const float* Qg = p.q + (size_t)b * G * V;
    for (int e = tid; e < G * nq; e += kThreads) {
      const int i = e / nq, k = e - i * nq;
      cp_async16(Qs + (size_t)i * W + k * 4, Qg + (size_t)i * V + v0 + k * 4);
    }
  }
  cp_async_commit();
  // this sequence's drafts with their logit and q value (plain loads, in
  // flight together with the slices; every CTA needs them for the scan)
  int d_own = -1;
  float l_own = 0.f, q_own = 0.f, u_own = 0.f;
  if (tid < G) {
    d_own = __ldg(p.draft + b * G + tid);
    if (d_own >= 0 && d_own < V) {
      l_own = Tr<T>::get(load_slot<T>(Lg + (size_t)tid * V, d_own, 1, false), 0);
      if (MODE == MODE_SOFTMAX) q_own = __ldg(p.q + ((size_t)b * G + tid) * V + d_own);
    }
  }
  if (MODE == MODE_SOFTMAX && tid < G1) u_own = __ldg(p.uniforms + b * G1 + tid);
  if (tid < G1) sm.ur[tid] = u_own;
  cp_async_wait<1>();
  __syncthreads();

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
      if (lane == 0) sm.part[i] = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
    } else {
      float M = -INFINITY;
      for (int k = lane; k < nvec; k += 32)
        M = fmaxf(M, TR::template vmax<false>(*reinterpret_cast<const uint4*>(Lr + k * VW)));
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
      float a0 = 0.f, a1 = 0.f;
      if (M > -INFINITY) {
        const float Mc = M * p.c;
        for (int k = lane; k < nvec; k += 32) {
          const uint4 v = *reinterpret_cast<const uint4*>(Lr + k * VW);
#pragma unroll
          for (int t = 0; t < VW; t += 2) {
            a0 += ex2_approx(fmaf(TR::get(v, t), p.c, -Mc));
            a1 += ex2_approx(fmaf(TR::get(v, t + 1), p.c, -Mc));
          }
        }
      }
      F2 s{a0 + a1, 0.f};
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) s = f2_add(s, f2_shfl_xor(s, m));
      if (lane == 0) sm.part[i] = make_float4(M, s.hi, s.lo, 0.f);
    }
  }
  cluster.sync();

  // ---- merge the CN partials of every row (16 lanes per row), then the scan
  for (int base = 0; base < G1; base += 2 * kWarps) {
    const int i = base + (tid >> 4);
    const bool rowok = i < G1;
    float4 v = make_float4(-INFINITY, 0.f, 0.f, 0.f);
    const int r = tid & 15;
    if (rowok && r < CN) v = *cluster.map_shared_rank(&sm.part[i], r);
    const float4 mg = group_merge<MODE>(v, CN, p.c);
    if (rowok && r == 0) {
      if (MODE == MODE_GREEDY) {
        const bool nan = mg.x != mg.x;
        const int bi = __float_as_int(mg.y);
        sm.g[i] = (nan || bi == 0x7fffffff) ? 0 : bi;
        sm.bad[i] = nan;
      } else {
        const double s = (double)mg.y + (double)mg.z;
        sm.M[i] = mg.x;
        sm.S[i] = s;
        sm.bad[i] = !(mg.x > -INFINITY && mg.x < INFINITY) || !(s > 0.0 && s < 1e300);
      }
    }
  }
  __syncthreads();
  if (MODE == MODE_SOFTMAX && tid < G) {
    const int d = d_own;
    float a = 0.f;
    int st = 0;
    if (d < 0 || d >= V) {
      st |= SEQ_OOB;
    } else {
      const float l = l_own;
      const float qd = q_own;
      const float pd = sm.bad[tid] ? 0.f : exp2f((l - sm.M[tid]) * p.c) / (float)sm.S[tid];
      if (qd > 0.0f) {
        a = fminf(1.f, pd / qd);
      } else {
        a = pd > 0.f ? 1.f : 0.f;
        st |= SEQ_QBAD;
      }
    }
    sm.a[tid] = a;
    sm.st[tid] = st;
  }
  __syncthreads();
  if (tid == 0) {
    int status = 0, n = G;
    for (int i = 0; i < G1; ++i)
      if (sm.bad[i]) status |= SEQ_BADROW;
    if (MODE == MODE_GREEDY) {
      for (int i = 0; i < G; ++i) {
        const int d = p.draft[b * G + i];
        if (d < 0 || d >= V) status |= SEQ_OOB;
      }
      for (int i = 0; i < G; ++i)
        if (p.draft[b * G + i] != sm.g[i]) { n = i; break; }
      sm.token = sm.g[n];
    } else {
      for (int i = 0; i < G; ++i) status |= sm.st[i];
      for (int i = 0; i < G; ++i)
        if (!(sm.ur[i] < sm.a[i])) { n = i; break; }
    }
    sm.n = n;
    sm.status = status;
  }
  __syncthreads();
  const int n = sm.n;
  if (rank == 0) {
    for (int j = tid; j < G1; j += kThreads) {
      if (j < n) p.out_tokens[b * G1 + j] = p.draft[b * G + j];
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
    cluster.sync();   // no CTA leaves while others may still read its partials
    return;
  }

  // ---- final draw: residual of row n, or the bonus from row gamma
  // (precise weights and the (S, A, Q) decomposition, as in residual_kernel)
  const bool resid = n < G;
  const bool bad = (sm.status & SEQ_BADROW) != 0;
  const T* Lf = Ls + (size_t)n * W;
  const float* Qf = resid ? Qs + (size_t)n * W : nullptr;
  const float M = sm.M[n];
  const float s_a = (float)sm.S[n];
  const int NS = cp.NS;
  int status = sm.status;
  cp_async_wait<0>();     // this thread's q copies have landed
  __syncthreads();        // ... and every thread's are visible to all
#pragma unroll
  for (int j = 0; j < kClusterMaxNS; ++j) {
    if (j < NS) {
      SlotRun run;
      run.zero();
      const int k = j * kThreads + tid;
      if (k < nvec && !bad) {
        const uint4 v = *reinterpret_cast<const uint4*>(Lf + k * VW);
        float qv[VW];
#pragma unroll
        for (int t = 0; t < VW; ++t) qv[t] = resid ? Qf[k * VW + t] : 0.f;
        run = slot_run<T>(v, qv, VW, resid, M, p.c, p.c_lo, s_a);
      }
      const F2x3 t = block_sum_f2x3(F2x3{run.S(), run.A(), F2{run.q, 0.f}}, sm.red);
      if (tid == 0) sm.sub3[j] = t;
    }
  }
  cluster.sync();
  // every CTA: the exact normaliser and the masses of all CN * NS sub-ranges
  F2 sl{0.f, 0.f};
  for (int e = tid; e < CN * NS; e += kThreads) {
    const F2x3 r3 = *cluster.map_shared_rank(&sm.sub3[e % NS], e / NS);
    sm.allS[e] = r3.a;
    sm.allmass[e] = r3.b;                 // A; corrected below once s is known
    sl = f2_add(sl, r3.a);
    sm.allQ[e] = r3.c.hi;
  }
  const F2 s = block_sum_f2(sl, sm.f2red);
  const F2 ds = f2_add(s, F2{-s_a, 0.f});
  for (int e = tid; e < CN * NS; e += kThreads) {
    if (resid) {
      F2 m = f2_add(sm.allmass[e], f2_neg(f2_scale(ds, sm.allQ[e])));
      if (m.hi < 0.f) m = F2{0.f, 0.f};
      sm.allmass[e] = m;
    } else {
      sm.allmass[e] = sm.allS[e];
    }
  }
  __syncthreads();
  {
    const float u = sm.ur[G];
    F2 R{0.f, 0.f}, base{0.f, 0.f}, tgt{0.f, 0.f};
    bool use_q = resid;
    int sub = locate(sm.allmass, CN * NS, u, &R, &base, &tgt, sm.loc, false);
    if (resid && !bad && !f2_pos(R)) {
      // zero residual mass (only through rounding): draw from p_n instead
      status |= SEQ_RESID0;
      use_q = false;
      sub = locate(sm.allS, CN * NS, u, &R, &base, &tgt, sm.loc, false);
    }
    if (tid == 0) {
      if (bad || !f2_pos(R)) sub = -1;
      sm.owner = sub < 0 ? -1 : sub / NS;
      sm.sub = sub < 0 ? -1 : sub % NS;
      sm.base = base;
      sm.target = tgt;
      sm.token = -1;
      sm.use_p = use_q ? 0 : 1;
      sm.ds = ds;
    }
  }
  __syncthreads();
  // every remote read of this CTA is done: arrive now, wait before leaving
  // (no CTA may exit while others can still read its shared memory)
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  if (sm.owner == rank) {
    const bool uq = sm.use_p == 0;
    const int k = sm.sub * kThreads + tid;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    float qv[VW];
#pragma unroll
    for (int t = 0; t < VW; ++t) qv[t] = 0.f;
    F2 mine{0.f, 0.f};
    if (k < nvec) {
      v = *reinterpret_cast<const uint4*>(Lf + k * VW);
#pragma unroll
      for (int t = 0; t < VW; ++t) qv[t] = uq ? Qf[k * VW + t] : 0.f;
      mine = slot_run<T>(v, qv, VW, uq, M, p.c, p.c_lo, s_a).mass(uq, sm.ds);
      if (mine.hi < 0.f) mine = F2{0.f, 0.f};
    }
    F2 total;
    const F2 ex = block_exclusive_f2(mine, sm.f2red, &total);
    const F2 tb = f2_add(sm.base, ex);
    int lastp = -1;
    if (k < nvec && f2_pos(mine) && !f2_lt(sm.target, tb) && f2_lt(sm.target, f2_add(tb, mine))) {
      const int f = slot_find<T>(v, qv, VW, uq, M, p.c, p.c_lo, s_a, sm.ds, tb, sm.target, &lastp);
      if (f >= 0) sm.token = v0 + k * VW + f;
    }
    __syncthreads();
    if (sm.token < 0) {
      int m = -1;
      if (k < nvec) {
        int lp = -1;
        slot_find<T>(v, qv, VW, uq, M, p.c, p.c_lo, s_a, sm.ds, F2{0.f, 0.f}, F2{INFINITY, 0.f}, &lp);
        if (lp >= 0) m = v0 + k * VW + lp;
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) sm.st[warp] = m;
      __syncthreads();
      if (tid == 0) {
        int mm = -1;
        for (int w = 0; w < kWarps; ++w) mm = max(mm, sm.st[w]);
        sm.token = mm;
      }
      __syncthreads();
    }
    if (tid == 0) {
      p.out_tokens[b * G1 + n] = sm.token < 0 ? 0 : sm.token;
      if (p.out_status) p.out_status[b] = status;
    }
  } else if (sm.owner < 0 && rank == 0 && tid == 0) {
    p.out_tokens[b * G1 + n] = 0;
    if (p.out_status) p.out_status[b] = status;
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace sv
