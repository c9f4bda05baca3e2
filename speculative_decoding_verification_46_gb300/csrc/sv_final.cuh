// Final draw of untruncated sampling: the one categorical draw per sequence,
// from the residual norm(max(p_n - q_n, 0)) after a rejection at n, or from
// p_gamma when every draft was accepted ("11.1 核心原理", section 11.1.2 and
// listing 10-1; the notes "Fast Inference from Transformers via Speculative
// Decoding", speculative-sampling paragraph).  The draw is the inverse CDF in
// token-index order: the smallest v with sum_{w <= v} r(w) > u * sum(r).
//
// Two kernels follow the row statistics (streaming kernel or rows kernel):
//
//   final_draw_kernel persistent; every WARP works through its own
//                     contiguous range of items (sequence b, 512 tokens of row
//                     n_b) with a lane-private cp.async ring of kFdStages
//                     items: no block barriers and no cross-warp waits.  When
//                     a warp reaches a new sequence it merges that
//                     sequence's per-warp row partials (streaming path; the
//                     rows path leaves the merged state), forms p_i(d_i) and
//                     a_i = min(1, p_i(d_i) / q_i(d_i)) and scans for the first
//                     rejection n (the drafts, their logits and q values are
//                     gathered before the dependency wait); the warp holding
//                     the sequence's first item writes every output but the
//                     drawn token.  Per item it sums (S, A, Q): the weights
//                     w = 2^((x - M) c), and over the residual support
//                     {w > s' q} the differences w - s' q and q (s' the float
//                     normaliser); lane 0 stores them.
//   final_pick_kernel one CTA per sequence: the inverse-CDF search item ->
//                     token over the item sums, then over the 512 tokens of
//                     the one item the target falls in (re-read from L2).
//
// Precision (the draw is compared with a float64 reference over up to 10^5
// CDF steps).  Tokens whose exponent (x - M) c is above -8 carry most of the
// mass: their weights and residuals are two-float (Tang's table exp2; the
// residual formed exactly).  Every other token's weight is ex2.approx with a
// first-order correction for the exponent's low part, and a lane adds its 16
// such tokens of an item in float32: each is below 2^-8 of the largest
// weight, so the rounding of these short sums stays at the level of the
// weights' own error.  Lane sums and everything above them are two-float.
// The exact normaliser s = sum S is formed at the end; the residual mass of
// an item is A - (s - s') Q.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kFdThreads = 256;            // 8 independent warps per CTA
constexpr int kFdWarps = kFdThreads / 32;
constexpr int kFdStages = 4;               // ring stages (items) per lane
constexpr int kFdTok = 512;                // tokens per item: 4 groups x 32 lanes x 4 tokens
constexpr int kPickThreads = 256;          // final_pick_kernel: 2 tokens of the item per thread

enum { FD_NONE = 0, FD_DENSE = 1, FD_DET = 2, FD_QL = 3, FD_SKIP = 4 };

// Ring bytes per lane per stage: 4 logits groups of 4 tokens ([group][lane],
// LB bytes each), then 4 q groups of 4 float32 or 4 draft logits ([group]
// [lane], QB bytes each).
template <typename T>
struct FdRing {
  static constexpr int LB = 4 * (int)sizeof(T);
  static constexpr int QB = 16;
  static constexpr int lane_bytes = 4 * LB + 4 * QB;
  static constexpr int stage_bytes = 32 * lane_bytes;   // one warp's stage
  static constexpr size_t bytes = (size_t)kFdWarps * kFdStages * stage_bytes;
};

__device__ __forceinline__ void fd_cp16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void fd_cp8(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void fd_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void fd_wait_ring() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kFdStages - 1) : "memory");
}

// What the final draw needs about one sequence: row n, how q is given, the
// row statistics and where the rows are.
template <typename T>
struct FdSeq {
  int n, gb, mode, status;
  float M, s_a;         // row n's maximum and float normaliser
  double s;             // row n's normaliser as merged
  int xq;               // deterministic draft: the rejected draft's token
  QLrow qlr;            // q formed from the draft's logits: row n's statistics
  const T* row;         // logits row n
  const float* qrow;    // q row n (FD_DENSE)
  const T* qlrow;       // draft logits row n (FD_QL)
};

// Row pointers and the mode of sequence b once n, status and the row
// statistics are known.
template <typename T>
__device__ __forceinline__ void fd_bind(const Params& p, int b, FdSeq<T>& s) {
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const bool resid = s.n < s.gb;
  s.row = static_cast<const T*>(p.logits) + ((size_t)b * G1 + s.n) * V;
  s.qrow = nullptr;
  s.qlrow = nullptr;
  s.xq = -1;
  if (s.status & SEQ_BADROW) {
    s.mode = FD_SKIP;   // outputs undefined (in range): nothing is read
  } else if (!resid) {
    s.mode = FD_NONE;
  } else if (p.ql) {
    s.mode = FD_QL;
    s.qlrow = static_cast<const T*>(p.ql) + ((size_t)b * G + s.n) * V;
  } else if (p.q) {
    s.mode = FD_DENSE;
    s.qrow = p.q + ((size_t)b * G + s.n) * V;
  } else {
    s.mode = FD_DET;
    s.xq = __ldg(p.draft + b * G + s.n);
  }
}

// The state a previous kernel left for sequence b (the rows path's finisher,
// or final_draw_kernel's scanning warp for final_pick_kernel).
template <typename T>
__device__ __forceinline__ void fd_load_state(const Params& p, int b, FdSeq<T>& s) {
  const SeqState* sp = p.seq + b;
  s.n = __ldcg(&sp->n);
  s.gb = seq_gamma(p, b);
  s.status = __ldcg(&sp->status);
  s.M = __ldcg(&sp->M);
  s.s = __ldcg(&sp->s);
  s.s_a = (float)s.s;
  s.qlr = QLrow{__ldcg(&sp->qm), __ldcg(&sp->qinv), __ldcg(&sp->qbad) != 0};
  fd_bind(p, b, s);
}

// Inputs of sequence b's acceptance tests for draft rows i = lane and
// lane + 32 (gamma <= 64): d_i, u_i, the target logit at d_i and q_i(d_i) (or
// the draft's logit at d_i).  Inputs only: gathered before the dependency
// wait when the sequence is known then.
struct FdDrafts {
  int d[2];
  float u[2], l[2], q[2];
};
template <typename T>
__device__ __forceinline__ void fd_gather(const Params& p, int b, FdDrafts& g) {
  const int lane = threadIdx.x & 31;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    g.d[h] = -1;
    g.u[h] = g.l[h] = g.q[h] = 0.f;
    if (i < gb) {
      const int d = __ldg(p.draft + b * G + i);
      g.d[h] = d;
      g.u[h] = __ldg(p.uniforms + b * G1 + i);
      if (d >= 0 && d < V) {
        g.l[h] = Tr<T>::get(load_slot<T>(static_cast<const T*>(p.logits) + ((size_t)b * G1 + i) * V, d, 1, false), 0);
        if (p.ql)
          g.q[h] = Tr<T>::get(load_slot<T>(static_cast<const T*>(p.ql) + ((size_t)b * G + i) * V, d, 1, false), 0);
        else
          g.q[h] = p.q ? __ldg(p.q + ((size_t)b * G + i) * V + d) : 1.f;   // NULL: one-hot draft
      }
    }
  }
}

// Merge the streaming kernel's per-warp partials of rows 0..nrows-1 (slot
// row * NP + j from `base`, NP = H * 8 slots per row, NP dividing 32; the
// first row is row r0g of the streaming kernel's; empty segment slots are
// skipped) into
// each row's maximum and two-float sum, delivered to lane (row mod 32) in
// entry (row / 32) of m / s / bad (a row with no maximum, an infinite one or
// no positive sum defines no distribution).  One aligned lane segment merges
// one row.
__device__ __forceinline__ void fd_merge_rows(const Params& p, const float4* base, long long r0g, int nrows,
                                              float m[2], F2 s[2], int bad[2]) {
  const int lane = threadIdx.x & 31;
  const int NP = stream_np(p);
  const int per = 32 / NP;   // rows merged per pass
  const int E = nrows * NP;
  m[0] = m[1] = -INFINITY;
  s[0] = s[1] = F2{0.f, 0.f};
  bad[0] = bad[1] = 1;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    const bool ok = e < E && seg_valid(p, r0g + e / NP, e % NP);
    const float4 v = ok ? __ldcg(base + e) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
    float M = v.x;
    for (int o = NP >> 1; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    F2 t{0.f, 0.f};
    if (ok && v.x > -INFINITY && M < INFINITY) {
      const float sc = ex2_approx((v.x - M) * p.c);
      t = f2_add(F2{v.y * sc, 0.f}, F2{v.z * sc, 0.f});
    }
    for (int o = NP >> 1; o >= 1; o >>= 1) t = f2_add(t, f2_shfl_xor(t, o));
    // row r0 + j's result is in lane j * NP; lane (row mod 32) takes it
    const int r0 = e0 / NP;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = lane + 32 * h;
      const int j = row - r0;
      const bool mine = j >= 0 && j < per && row < nrows;
      const int src = mine ? j * NP : 0;
      const float Mr = __shfl_sync(0xffffffffu, M, src);
      const float th = __shfl_sync(0xffffffffu, t.hi, src), tl = __shfl_sync(0xffffffffu, t.lo, src);
      if (mine) {
        m[h] = Mr;
        s[h] = F2{th, tl};
        const double sum = (double)th + (double)tl;
        bad[h] = !(Mr > -INFINITY && Mr < INFINITY) || !(sum > 0.0 && sum < 1e300);
      }
    }
  }
}

// The acceptance scan of sequence b by one warp (streaming path): row
// statistics merged from the partials, a_i for i < gamma_b, n = the first
// rejected position (gamma_b if none), the status bits, and row n's state
// in s.  `writer`: this warp holds the sequence's first item and writes the
// outputs (all but the drawn token) and the state final_pick_kernel reads.
template <typename T>
__device__ __forceinline__ void fd_scan(const Params& p, int b, const FdDrafts& g, bool writer, FdSeq<T>& s) {
  const int lane = threadIdx.x & 31;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);
  const int NP = stream_np(p);
  float rM[2], qM[2];
  F2 rS[2], qS[2];
  int rBad[2], qBad[2];
  fd_merge_rows(p, p.part + (size_t)b * G1 * NP, (long long)b * G1, gb + 1, rM, rS, rBad);
  if (p.ql) fd_merge_rows(p, p.qpart + (size_t)b * G * NP, (long long)p.B * G1 + (long long)b * G, gb, qM, qS, qBad);
  int bits = 0;
  float a[2] = {0.f, 0.f};
  unsigned rej[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    bool r = false;
    if (i < gb) {
      const int d = g.d[h];
      if (d < 0 || d >= V) {
        bits |= SEQ_OOB;
      } else {
        float qd = g.q[h];
        if (p.ql) {
          const double qs = (double)qS[h].hi + (double)qS[h].lo;
          qd = qBad[h] ? 0.f : q_weight(qd, qM[h], p.c, p.c_lo) * (float)(1.0 / qs);
        }
        const float ssum = (float)((double)rS[h].hi + (double)rS[h].lo);
        const float pd = rBad[h] ? 0.f : exp2f((g.l[h] - rM[h]) * p.c) / ssum;
        if (qd > 0.f) {
          a[h] = fminf(1.f, pd / qd);
        } else {
          a[h] = pd > 0.f ? 1.f : 0.f;
          bits |= SEQ_QBAD;
        }
      }
      r = !(g.u[h] < a[h]);
    }
    rej[h] = __ballot_sync(0xffffffffu, r);
  }
  const int n = rej[0] ? __ffs(rej[0]) - 1 : (rej[1] ? 32 + __ffs(rej[1]) - 1 : gb);
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (__any_sync(0xffffffffu, (lane <= gb && rBad[0]) || (lane + 32 <= gb && rBad[1]))) bits |= SEQ_BADROW;
  // row n's statistics (and its draft row's, with q from draft logits) from lane n mod 32
  const int hn = n >> 5, ln = n & 31;
  const float Mn = __shfl_sync(0xffffffffu, hn ? rM[1] : rM[0], ln);
  const float Sh = __shfl_sync(0xffffffffu, hn ? rS[1].hi : rS[0].hi, ln);
  const float Sl = __shfl_sync(0xffffffffu, hn ? rS[1].lo : rS[0].lo, ln);
  s.n = n;
  s.gb = gb;
  s.status = bits;
  s.M = Mn;
  s.s = (double)Sh + (double)Sl;
  s.s_a = (float)s.s;
  s.qlr = QLrow{0.f, 0.f, true};
  if (p.ql) {
    const float qm = __shfl_sync(0xffffffffu, hn ? qM[1] : qM[0], ln);
    const float qh = __shfl_sync(0xffffffffu, hn ? qS[1].hi : qS[0].hi, ln);
    const float ql = __shfl_sync(0xffffffffu, hn ? qS[1].lo : qS[0].lo, ln);
    const int qb = __shfl_sync(0xffffffffu, hn ? qBad[1] : qBad[0], ln);
    if (n < gb) s.qlr = QLrow{qm, (float)(1.0 / ((double)qh + (double)ql)), qb != 0};
  }
  fd_bind(p, b, s);
  if (writer) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      if (p.out_a && i < G) p.out_a[b * G + i] = i < gb ? a[h] : 0.f;
      if (i < G1 && i != n) p.out_tokens[b * G1 + i] = i < n ? g.d[h] : -1;
    }
    if (lane == 0) {
      p.out_n[b] = n;
      SeqState st;
      st.n = n;
      st.status = bits;
      st.M = s.M;
      st.s = s.s;
      st.qm = s.qlr.m;
      st.qinv = s.qlr.inv;
      st.qbad = s.qlr.bad ? 1 : 0;
      p.seq[b] = st;
    }
  }
}

// One 4-token group of an unaligned row (V % 4 != 0), token by token: the
// logits, and q or the draft's logits when given.  Tokens past the row's end
// are not read.
template <typename T>
__device__ __noinline__ void fd_scalar_group(const T* row, const float* qrow, const T* qlrow, int t0, int V,
                                             unsigned char* ld, unsigned char* qd) {
  for (int t = 0; t < 4; ++t) {
    if (t0 + t < V) {
      if (sizeof(T) == 4) reinterpret_cast<uint32_t*>(ld)[t] = Tr<T>::scalar_bits(row + t0 + t);
      else reinterpret_cast<unsigned short*>(ld)[t] = (unsigned short)Tr<T>::scalar_bits(row + t0 + t);
      if (qrow) {
        reinterpret_cast<float*>(qd)[t] = __ldg(qrow + t0 + t);
      } else if (qlrow) {
        if (sizeof(T) == 4) reinterpret_cast<uint32_t*>(qd)[t] = Tr<T>::scalar_bits(qlrow + t0 + t);
        else reinterpret_cast<unsigned short*>(qd)[t] = (unsigned short)Tr<T>::scalar_bits(qlrow + t0 + t);
      }
    }
  }
}

// Issue this lane's copies of item c of sequence s into one ring stage:
// logits groups g = 0..3 (tokens c*512 + 128 g + 4 lane .. + 3) and, for a
// residual, the matching q (or draft logit) groups.  vec: 4-token groups are
// aligned (V % 4 == 0); otherwise the in-range tokens are loaded one by one.
// Groups past the end of the row are not read (the sweep gives them weight 0).
template <typename T>
__device__ __forceinline__ void fd_issue(const FdSeq<T>& s, int c, int V, bool vec, unsigned char* st) {
  using R = FdRing<T>;
  if (s.mode == FD_SKIP) return;
  const int lane = threadIdx.x & 31;
  unsigned char* lg = st;
  unsigned char* qg = st + 4 * 32 * R::LB;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int t0 = c * kFdTok + 128 * g + 4 * lane;
    unsigned char* ld = lg + (g * 32 + lane) * R::LB;
    unsigned char* qd = qg + (g * 32 + lane) * R::QB;
    if (vec) {
      if (t0 < V) {
        if (R::LB == 16) fd_cp16(ld, s.row + t0); else fd_cp8(ld, s.row + t0);
        if (s.mode == FD_DENSE) {
          fd_cp16(qd, s.qrow + t0);
        } else if (s.mode == FD_QL) {
          if (R::LB == 16) fd_cp16(qd, s.qlrow + t0); else fd_cp8(qd, s.qlrow + t0);
        }
      }
    } else {
      fd_scalar_group(s.row, s.mode == FD_DENSE ? s.qrow : nullptr, s.mode == FD_QL ? s.qlrow : nullptr, t0, V, ld,
                      qd);
    }
  }
}

// The 4 tokens of a group held as raw little-endian bytes.
template <typename T>
__device__ __forceinline__ void fd_unpack(const unsigned char* grp, float x[4]) {
  if (sizeof(T) == 4) {
    const float4 v = *reinterpret_cast<const float4*>(grp);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(grp);
    if (std::is_same<T, __half>::value) {
      x[0] = __half2float(__ushort_as_half((unsigned short)(w.x & 0xffffu)));
      x[1] = __half2float(__ushort_as_half((unsigned short)(w.x >> 16)));
      x[2] = __half2float(__ushort_as_half((unsigned short)(w.y & 0xffffu)));
      x[3] = __half2float(__ushort_as_half((unsigned short)(w.y >> 16)));
    } else {
      x[0] = __uint_as_float(w.x << 16);
      x[1] = __uint_as_float(w.x & 0xffff0000u);
      x[2] = __uint_as_float(w.y << 16);
      x[3] = __uint_as_float(w.y & 0xffff0000u);
    }
  }
}

// q of the 4 tokens of a group starting at token t0 (mode-specific): dense
// float32 q, q formed from the draft's logits, or the deterministic draft's
// one-hot (+inf at the rejected draft's token takes it out of the residual
// support; 0 elsewhere).
template <typename T, int MODE>
__device__ __forceinline__ void fd_qgroup(const FdSeq<T>& s, const unsigned char* grp, int t0, float c, float c_lo,
                                          float q[4]) {
  if (MODE == FD_DENSE) {
    const float4 v = *reinterpret_cast<const float4*>(grp);
    q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
  } else if (MODE == FD_QL) {
    float x[4];
    fd_unpack<T>(grp, x);
#pragma unroll
    for (int t = 0; t < 4; ++t) q[t] = s.qlr.q(x[t], c, c_lo);
  } else if (MODE == FD_DET) {
#pragma unroll
    for (int t = 0; t < 4; ++t) q[t] = t0 + t == s.xq ? INFINITY : 0.f;
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) q[t] = 0.f;
  }
}

// Per-lane sums of one item: tail tokens in float32 (two of each, for even
// and odd tokens of a group: shorter dependency chains), tokens near the
// maximum in two-float.
struct FdAcc {
  float S[2], A[2], Q[2];
  RunAcc top;
};

// One item's 16 tokens of this lane.  The per-token formulas are those of
// run_tail / run_top, so token_mass reproduces each token's share.  FULL: the
// whole item lies inside the row.
template <typename T, int MODE, bool FULL>
__device__ __forceinline__ void fd_sweep(const FdSeq<T>& s, const unsigned char* st, int c, int V, float cc,
                                         float c_lo, const float* tab, FdAcc& acc) {
  using R = FdRing<T>;
  constexpr bool EXACT = sizeof(T) == 2;
  const int lane = threadIdx.x & 31;
  const unsigned char* lg = st;
  const unsigned char* qg = st + 4 * 32 * R::LB;
  const float M = s.M, s_a = s.s_a;
  uint32_t near = 0u;
  // rolled over the 4 groups (the 4 tokens of a group are independent): the
  // kernel holds 8 variants of this sweep, and unrolled they overflow the
  // instruction cache
#pragma unroll 1
  for (int g = 0; g < 4; ++g) {
    const int t0 = c * kFdTok + 128 * g + 4 * lane;
    float x[4], q[4];
    fd_unpack<T>(lg + (g * 32 + lane) * R::LB, x);
    fd_qgroup<T, MODE>(s, qg + (g * 32 + lane) * R::QB, t0, cc, c_lo, q);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (!FULL && t0 + t >= V) {
        x[t] = -INFINITY;
        q[t] = 0.f;
      }
      float e, p;
      if (EXACT) {
        const float dh = fmaxf(x[t] - M, -1.0e4f);   // exact for 16-bit logits; -inf flushes to 0 below
        p = dh * cc;
        e = fmaf(dh, c_lo, fmaf(dh, cc, -p));
      } else {
        p = tok_exponent<false>(x[t], M, cc, c_lo, &e);
      }
      const bool hi = p > -8.f;
      const float y = ex2_approx(p);
      float w = fmaf(y * 6.931471825e-01f, e, y);
      if (!EXACT) w = p > -1.0e30f ? w : 0.f;   // -inf (float32 logits)
      w = hi ? 0.f : w;
      near |= (uint32_t)hi << (4 * g + t);
      acc.S[t & 1] += w;
      if (MODE != FD_NONE) {
        // the residual support {w > s' q}: the sign of w - s' q rounded once
        const float d = fmaf(-s_a, q[t], w);
        acc.A[t & 1] += fmaxf(d, 0.f);
        acc.Q[t & 1] += d > 0.f ? q[t] : 0.f;
      }
    }
  }
  while (near) {
    const int o = __ffs(near) - 1;
    near &= near - 1;
    const int g = o >> 2, t = o & 3;
    const int t0 = c * kFdTok + 128 * g + 4 * lane;
    float x[4], q[4];
    fd_unpack<T>(lg + (g * 32 + lane) * R::LB, x);
    fd_qgroup<T, MODE>(s, qg + (g * 32 + lane) * R::QB, t0, cc, c_lo, q);
    run_top<EXACT>(acc.top, x[t], q[t], MODE != FD_NONE, M, cc, c_lo, s_a, tab);
  }
}

// One item's lane sums: S and A two-float, Q float32.
struct IT5 {
  F2 S{0.f, 0.f}, A{0.f, 0.f};
  float Q = 0.f;
  __device__ static __forceinline__ IT5 of(F2 s, F2 a, float q) {
    IT5 r;
    r.S = s;
    r.A = a;
    r.Q = q;
    return r;
  }
};
__device__ __forceinline__ IT5 it5_add(const IT5& a, const IT5& b) {
  return IT5::of(f2_add(a.S, b.S), f2_add(a.A, b.A), a.Q + b.Q);
}
__device__ __forceinline__ IT5 it5_sel(bool c, const IT5& a, const IT5& b) { return c ? a : b; }
__device__ __forceinline__ IT5 it5_shfl_xor(const IT5& v, int m) {
  return IT5::of(f2_shfl_xor(v.S, m), f2_shfl_xor(v.A, m), __shfl_xor_sync(0xffffffffu, v.Q, m));
}

// Warp totals of four items at once: a butterfly in which each exchange
// halves the items a lane keeps (xor 16: slots {0,1} or {2,3}; xor 8: one
// slot), then three plain levels.  Returns, in every lane of group
// g = lane / 8, the total of slot g.
__device__ __forceinline__ IT5 it5_reduce4(const IT5 slot[4]) {
  const int lane = threadIdx.x & 31;
  const bool up16 = (lane & 16) != 0, up8 = (lane & 8) != 0;
  IT5 h[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const IT5 keep = it5_sel(up16, slot[2 + j], slot[j]);
    const IT5 send = it5_sel(up16, slot[j], slot[2 + j]);
    h[j] = it5_add(keep, it5_shfl_xor(send, 16));
  }
  const IT5 keep = it5_sel(up8, h[1], h[0]);
  const IT5 send = it5_sel(up8, h[0], h[1]);
  IT5 t = it5_add(keep, it5_shfl_xor(send, 8));
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) t = it5_add(t, it5_shfl_xor(t, m));
  return t;
}

template <typename T>
__global__ void __launch_bounds__(kFdThreads, 2) final_draw_kernel(const Params p) {
  using R = FdRing<T>;
  extern __shared__ __align__(16) unsigned char fd_dyn[];
  __shared__ float tab[128];
  load_exp2_table(tab);
  __syncthreads();   // the only block barrier: the warps are independent from here on
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* ring = fd_dyn + (size_t)warp * kFdStages * R::stage_bytes;
  const int V = p.V, C = p.FC;
  const long long N = (long long)p.B * C;
  const long long NW = (long long)gridDim.x * kFdWarps;
  const long long g = (long long)blockIdx.x * kFdWarps + warp;
  const int i0 = (int)(g * N / NW), i1 = (int)((g + 1) * N / NW);
  if (i0 >= i1) {
    pdl_wait();
    return;
  }
  const bool vec = (V & 3) == 0;
  const bool scan = p.H > 0;   // streaming path: the row partials are merged here
  const int b0 = i0 / C;
  // inputs of the first sequence's acceptance tests, before the wait
  FdDrafts dr;
  int dr_b = -1;   // the sequence dr holds
  if (scan) {
    fd_gather<T>(p, b0, dr);
    dr_b = b0;
  }
  pdl_wait();   // the row statistics come from the previous kernel
  // The issuer runs up to kFdStages items ahead of the consumer; it reaches
  // each sequence first (and scans it), the consumer takes a copy of its state.
  FdSeq<T> is, cs;
  int is_b = -1, cs_b = -1;
  auto reach = [&](int b) {
    if (scan) {
      if (b != dr_b) {
        fd_gather<T>(p, b, dr);
        dr_b = b;
      }
      fd_scan<T>(p, b, dr, (long long)b * C >= i0, is);
    } else {
      fd_load_state<T>(p, b, is);
    }
    is_b = b;
  };
  int ki = i0;
#pragma unroll 1
  for (int st = 0; st < kFdStages; ++st) {
    if (ki < i1) {
      const int b = ki / C;
      if (b != is_b) reach(b);
      fd_issue(is, ki - b * C, V, vec, ring + st * R::stage_bytes);
      ++ki;
    }
    fd_commit();
  }
  int stage = 0;
  int cs_end = -1;   // first item past the consumer's sequence
  // Items are reduced across the warp four at a time (transposed butterfly):
  // the lane sums of the batch's items sit in slots 0..3 (slot 0 the latest).
  for (int kb = i0; kb < i1; kb += 4) {
    const int nb = min(4, i1 - kb);
    IT5 slot[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) slot[j] = IT5{};
#pragma unroll 1
    for (int kc = kb; kc < kb + nb; ++kc) {
      fd_wait_ring();
      if (kc >= cs_end) {
        // the consumer reaches a new sequence: the issuer is on it unless it
        // has already moved on (fewer than kFdStages items of this sequence
        // left in the range), in which case the state is rebuilt
        const int b = kc / C;
        if (b != is_b) {
          const int keep_b = is_b;
          FdSeq<T> keep = is;
          reach(b);
          cs = is;
          is = keep;
          is_b = keep_b;
        } else {
          cs = is;
        }
        cs_b = b;
        cs_end = (b + 1) * C;
      }
      const int c = kc - cs_b * C;
      unsigned char* st = ring + stage * R::stage_bytes;
      FdAcc acc;
      acc.S[0] = acc.S[1] = acc.A[0] = acc.A[1] = acc.Q[0] = acc.Q[1] = 0.f;
      acc.top.zero();
      const bool full = (c + 1) * kFdTok <= V;
      switch (cs.mode * 2 + (full ? 1 : 0)) {
        case FD_NONE * 2 + 1: fd_sweep<T, FD_NONE, true>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        case FD_NONE * 2: fd_sweep<T, FD_NONE, false>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        case FD_DENSE * 2 + 1: fd_sweep<T, FD_DENSE, true>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        case FD_DENSE * 2: fd_sweep<T, FD_DENSE, false>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        case FD_DET * 2 + 1: fd_sweep<T, FD_DET, true>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        case FD_DET * 2: fd_sweep<T, FD_DET, false>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        case FD_QL * 2 + 1: fd_sweep<T, FD_QL, true>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        case FD_QL * 2: fd_sweep<T, FD_QL, false>(cs, st, c, V, p.c, p.c_lo, tab, acc); break;
        default: break;   // a bad row: nothing was read
      }
      // this stage has been read: refill it with the item kFdStages ahead
      if (ki < i1) {
        const int b2 = ki / C;
        if (b2 != is_b) reach(b2);
        fd_issue(is, ki - b2 * C, V, vec, st);
        ++ki;
      }
      fd_commit();
      stage = stage + 1 == kFdStages ? 0 : stage + 1;
      slot[3] = slot[2];
      slot[2] = slot[1];
      slot[1] = slot[0];
      slot[0] = IT5::of(f2_add(f2_add(F2{acc.S[0], 0.f}, F2{acc.S[1], 0.f}), acc.top.S()),
                        f2_add(f2_add(F2{acc.A[0], 0.f}, F2{acc.A[1], 0.f}), acc.top.A()),
                        acc.Q[0] + acc.Q[1] + acc.top.q);
    }
    // slot j holds item kb + nb - 1 - j; after the butterfly every lane of
    // group g = lane / 8 holds slot g's warp total
    const IT5 tot = it5_reduce4(slot);
    const int g = lane >> 3;
    if ((lane & 7) == 0 && g < nb) {
      const int k = kb + nb - 1 - g;
      const int b = k / C, c = k - b * C;
      p.fd_part[(size_t)b * C + c] = make_float4(tot.S.hi, tot.S.lo, tot.A.hi, tot.A.lo);
      p.fd_q[(size_t)b * C + c] = tot.Q;
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- the search

struct PickSmem {
  float tab[128];
  F2 wsum[kPickThreads / 32];
  F2 carry;
  F2 base, lastbase;
  int found, last;
  int owner, lastpos;
  int token;
};

// Block-wide inverse-CDF search over NT two-float masses mass(k) in index
// order: the total R, then the first k whose running interval [prefix_k,
// prefix_k + m_k) holds t = u * R (both passes add in the same order), else
// the last k with positive mass.  Returns k (-1 if R <= 0) and its exclusive
// prefix in *base_out, R in *R_out and t in *t_out, in every thread.
template <typename F>
__device__ int pick_locate(F mass, int NT, float u, F2* R_out, F2* base_out, F2* t_out, PickSmem& ls) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = kPickThreads / 32;
  F2 R{0.f, 0.f}, t{0.f, 0.f};
  for (int pass = 0; pass < 2; ++pass) {
    t = f2_scale(R, u);
    __syncthreads();
    if (tid == 0) {
      ls.carry = F2{0.f, 0.f};
      ls.found = 0x7fffffff;
      ls.last = -1;
      ls.lastbase = F2{0.f, 0.f};
    }
    __syncthreads();
    for (int c0 = 0; c0 < NT; c0 += kPickThreads) {
      const int k = c0 + tid;
      const F2 m = k < NT ? mass(k) : F2{0.f, 0.f};
      const F2 inc = warp_incl_scan_f2(m);
      if (lane == 31) ls.wsum[warp] = inc;
      __syncthreads();
      F2 off = ls.carry, tot = ls.carry;
#pragma unroll
      for (int w = 0; w < nw; ++w) {
        if (w < warp) off = f2_add(off, ls.wsum[w]);
        tot = f2_add(tot, ls.wsum[w]);
      }
      F2 below = f2_shfl_up(inc, 1);
      if (lane == 0) below = F2{0.f, 0.f};
      const F2 excl = f2_add(off, below);
      if (pass == 1 && k < NT && f2_pos(m)) {
        if (!f2_lt(t, excl) && f2_lt(t, f2_add(excl, m))) atomicMin(&ls.found, k);
        atomicMax(&ls.last, k);
      }
      __syncthreads();
      if (pass == 1 && k < NT) {
        if (ls.found == k) ls.base = excl;
        if (ls.last == k) ls.lastbase = excl;
      }
      if (tid == 0) ls.carry = tot;
      __syncthreads();
      if (pass == 1 && ls.found != 0x7fffffff) break;
    }
    if (pass == 0) R = ls.carry;
  }
  __syncthreads();
  *R_out = R;
  *t_out = t;
  if (!f2_pos(R)) return -1;
  if (ls.found != 0x7fffffff) {
    *base_out = ls.base;
    return ls.found;
  }
  *base_out = ls.lastbase;
  return ls.last;
}

// The item search with every item's sums read once into registers (thread t
// holds items t, t + 256, ...; C <= 256 * kPickRegItems): the masses, one
// block-wide inclusive scan per 256 items chained by a carry (its total is
// R, so the search and the total agree), and the first item whose interval
// holds u * R, else the last positive one.  Same results as pick_locate.
template <int KP>
__device__ int pick_items_fast_t(const float4* SA, const float* QQ, int C, bool use_q, F2 ds, float u, F2* R_out,
                                 F2* base_out, F2* t_out, PickSmem& ls) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = kPickThreads / 32;
  F2 m[KP], ex[KP];
#pragma unroll
  for (int j = 0; j < KP; ++j) {
    const int k = j * kPickThreads + tid;
    m[j] = F2{0.f, 0.f};
    if (k < C) {
      const float4 v = __ldcg(SA + k);
      if (!use_q) {
        m[j] = F2{v.x, v.y};
      } else {
        m[j] = f2_add(F2{v.z, v.w}, f2_neg(f2_scale(ds, __ldcg(QQ + k))));
        if (m[j].hi < 0.f) m[j] = F2{0.f, 0.f};
      }
    }
  }
  F2 carry{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < KP; ++j) {
    if (j * kPickThreads >= C) break;
    const F2 inc = warp_incl_scan_f2(m[j]);
    __syncthreads();   // wsum of the previous round has been read
    if (lane == 31) ls.wsum[warp] = inc;
    __syncthreads();
    F2 off = carry, tot = carry;
#pragma unroll
    for (int w = 0; w < nw; ++w) {
      if (w < warp) off = f2_add(off, ls.wsum[w]);
      tot = f2_add(tot, ls.wsum[w]);
    }
    F2 below = f2_shfl_up(inc, 1);
    if (lane == 0) below = F2{0.f, 0.f};
    ex[j] = f2_add(off, below);
    carry = tot;
  }
  const F2 R = carry;
  const F2 t = f2_scale(R, u);
  if (tid == 0) {
    ls.found = 0x7fffffff;
    ls.last = -1;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < KP; ++j) {
    const int k = j * kPickThreads + tid;
    if (k < C && f2_pos(m[j])) {
      if (!f2_lt(t, ex[j]) && f2_lt(t, f2_add(ex[j], m[j]))) atomicMin(&ls.found, k);
      atomicMax(&ls.last, k);
    }
  }
  __syncthreads();
  const int found = ls.found, last = ls.last;
#pragma unroll
  for (int j = 0; j < KP; ++j) {
    const int k = j * kPickThreads + tid;
    if (k == found) ls.base = ex[j];
    if (k == last) ls.lastbase = ex[j];
  }
  __syncthreads();
  *R_out = R;
  *t_out = t;
  const int item = !f2_pos(R) ? -1 : (found != 0x7fffffff ? found : last);
  *base_out = found != 0x7fffffff ? ls.base : ls.lastbase;
  __syncthreads();   // ls may be reused right after
  return item;
}
constexpr int kPickRegItems = 4;
__device__ __forceinline__ int pick_items_fast(const float4* SA, const float* QQ, int C, bool use_q, F2 ds, float u,
                                               F2* R_out, F2* base_out, F2* t_out, PickSmem& ls) {
  if (C <= kPickThreads) return pick_items_fast_t<1>(SA, QQ, C, use_q, ds, u, R_out, base_out, t_out, ls);
  return pick_items_fast_t<kPickRegItems>(SA, QQ, C, use_q, ds, u, R_out, base_out, t_out, ls);
}

// One CTA per sequence after final_draw_kernel: the exact normaliser
// s = sum S, the item masses (A - (s - s') Q for a residual, S for the bonus
// or the fallback to p_n), the item holding u * R, then the token inside it
// (each thread two consecutive tokens of the item), the output, and the
// workspace zeroed behind it.
template <typename T>
__global__ void __launch_bounds__(kPickThreads) final_pick_kernel(const Params p) {
  constexpr bool EXACT = sizeof(T) == 2;
  __shared__ PickSmem sm;
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  const int G = p.gamma, G1 = G + 1, V = p.V, C = p.FC;
  load_exp2_table(sm.tab);
  const int gb = seq_gamma(p, b);
  const float u = __ldg(p.uniforms + b * G1 + gb);   // an input: before the wait
  pdl_wait();
  __syncthreads();
  FdSeq<T> s;
  fd_load_state<T>(p, b, s);
  const bool bad = s.mode == FD_SKIP;
  const bool resid = s.n < gb;
  float4* SA = p.fd_part + (size_t)b * C;
  float* QQ = p.fd_q + (size_t)b * C;
  int token = 0, resid0 = 0;
  if (!bad) {
    F2 sl{0.f, 0.f};
    for (int k = tid; k < C; k += kPickThreads) {
      const float4 v = __ldcg(SA + k);
      sl = f2_add(sl, F2{v.x, v.y});
    }
    const F2 sum = block_sum_f2(sl, sm.wsum);
    const F2 ds = f2_add(sum, F2{-s.s_a, 0.f});   // s - s', tiny
    bool use_q = resid;
    auto mass = [&](int k) -> F2 {
      const float4 v = __ldcg(SA + k);
      if (!use_q) return F2{v.x, v.y};
      F2 m = f2_add(F2{v.z, v.w}, f2_neg(f2_scale(ds, __ldcg(QQ + k))));
      if (m.hi < 0.f) m = F2{0.f, 0.f};
      return m;
    };
    F2 R{0.f, 0.f}, base{0.f, 0.f}, target{0.f, 0.f};
    int item;
    if (C <= kPickThreads * kPickRegItems) {
      item = pick_items_fast(SA, QQ, C, use_q, ds, u, &R, &base, &target, sm);
      if (resid && !f2_pos(R)) {
        resid0 = 1;   // zero residual mass (only through rounding): draw from p_n
        use_q = false;
        item = pick_items_fast(SA, QQ, C, use_q, ds, u, &R, &base, &target, sm);
      }
    } else {
      item = pick_locate(mass, C, u, &R, &base, &target, sm);
      if (resid && !f2_pos(R)) {
        resid0 = 1;
        use_q = false;
        item = pick_locate(mass, C, u, &R, &base, &target, sm);
      }
    }
    if (item >= 0) {
      // ---- the item's tokens: this thread's two, their masses
      const int mode = use_q ? s.mode : FD_NONE;
      const int t0 = item * kFdTok + 2 * tid;
      F2 tm[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int v = t0 + j;
        tm[j] = F2{0.f, 0.f};
        if (v < V) {
          const float x = Tr<T>::get(load_slot<T>(s.row, v, 1, false), 0);
          float qv = 0.f;
          if (mode == FD_DENSE) qv = __ldcg(s.qrow + v);
          else if (mode == FD_QL) qv = s.qlr.q(Tr<T>::get(load_slot<T>(s.qlrow, v, 1, false), 0), p.c, p.c_lo);
          else if (mode == FD_DET) qv = v == s.xq ? INFINITY : 0.f;
          tm[j] = token_mass<EXACT>(x, qv, use_q, s.M, p.c, p.c_lo, s.s_a, ds, sm.tab);
        }
      }
      const F2 mine = f2_add(tm[0], tm[1]);
      F2 total;
      const F2 ex = block_exclusive_f2(mine, sm.wsum, &total);
      const F2 tb = f2_add(base, ex);
      if (tid == 0) {
        sm.owner = 0x7fffffff;
        sm.lastpos = -1;
      }
      __syncthreads();
      const bool pos = f2_pos(mine);
      if (pos && !f2_lt(target, tb) && f2_lt(target, f2_add(tb, mine))) atomicMin(&sm.owner, tid);
      if (pos) atomicMax(&sm.lastpos, tid);
      __syncthreads();
      // rounding can leave no thread's interval holding the target: take the last positive one
      const bool take_last = sm.owner == 0x7fffffff;
      const int owner = take_last ? sm.lastpos : sm.owner;
      if (tid == owner) {
        int pick = -1, lastp = -1;
        F2 lb = tb;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (f2_pos(tm[j])) {
            if (pick < 0 && !take_last && !f2_lt(target, lb) && f2_lt(target, f2_add(lb, tm[j]))) pick = j;
            lastp = j;
          }
          lb = f2_add(lb, tm[j]);
        }
        sm.token = t0 + (pick >= 0 ? pick : lastp);
      }
      __syncthreads();
      token = owner >= 0 ? sm.token : 0;
    }
  }
  // the output; the item sums, the row partials and the state zeroed behind it
  for (int k = tid; k < C; k += kPickThreads) {
    SA[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    QQ[k] = 0.f;
  }
  if (p.H > 0) {
    const int E = G1 * stream_np(p);
    for (int e = tid; e < E; e += kPickThreads) p.part[(size_t)b * E + e] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.ql) {
      const int Eq = G * stream_np(p);
      for (int e = tid; e < Eq; e += kPickThreads) p.qpart[(size_t)b * Eq + e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (tid == 0) {
    p.out_tokens[b * G1 + s.n] = token;
    if (p.out_status) p.out_status[b] = s.status | (resid0 ? SEQ_RESID0 : 0);
    SeqState z;
    z.n = 0; z.status = 0; z.M = 0.f; z.qm = 0.f; z.s = 0.0; z.qinv = 0.f; z.qbad = 0;
    p.seq[b] = z;
  }
}

}  // namespace sv
