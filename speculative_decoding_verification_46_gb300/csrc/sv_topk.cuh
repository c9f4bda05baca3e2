// Top-k / top-p pieces shared by the streaming top-k kernel (sv_stream.cuh):
// shared-memory layout, the per-row epilogue
// (softmax(./T) over the row's top-k, the top-p cut, the kept list and the
// acceptance probability of the row's draft) and the per-sequence finisher
// (acceptance scan, final draw over the kept list of row n in token order,
// the residual max(p - q, 0) needing q only at the kept indices).
// Order of the transforms as in "11.1 核心原理" section 11.1.2: temperature,
// top-k by (logit desc, index asc), renormalise, top-p, renormalise.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kTkCap = kMaxK;   // candidates >= tau held per row (more: the exact fallback)
constexpr int kTkWarps = 256 / 32;

struct TopkSmem {
  unsigned long long cand[kTkCap];   // candidates >= tau; the finisher's two-float weights
  float w[kMaxK];                    // the row's top-k in rank order: logits, then exp2 weights
  int widx[kMaxK];                   // and their token indices
  int sidx[kMaxK];                   // finisher: kept indices in token order
  int rel[256];                      // threads whose maximum reaches tau
  int hist[256];                     // radix select of tau: one 8-bit digit's histogram
  int pick_digit;
  int pick_rank;
  int ired[kTkWarps];
  float fu[kMaxG1];                  // finisher: uniforms and acceptance probabilities
  float fa[kMaxG1];
  LocateSmem loc;
  int flag;
  int rows[4];                       // streaming: this CTA's rows j .. j + 3 (ring by j & 3)
  int count;
  int nrel;
  int n;
  int status;
  int token;
  int J;
  float WJ;
  float pd;
};
static_assert(sizeof(unsigned long long) * kTkCap >= sizeof(F2) * kMaxK, "finisher weights fit in cand");

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

// The probability a kept list ([0].x = J, then J (index, probability bits))
// gives token v: 0 if v is not kept.
__device__ __forceinline__ float kept_prob(const int2* list, int v) {
  const int J = __ldcg(list).x;
  float pv = 0.f;
  for (int e = 0; e < J; ++e) {
    const int2 en = __ldcg(list + 1 + e);
    if (en.x == v) pv = __int_as_float(en.y);
  }
  return pv;
}

// Final step of a sequence (run by the CTA that finished its last row): the
// acceptance scan, then the draw over the kept list of row n in token order.
// With q formed from the draft's logits (p.ql), q_i is draft row i's kept
// list: the acceptance tests are formed here, and q(v) of the final draw is
// looked up in draft row n's list.
__device__ void topk_finish_sequence(const Params& p, int b, TopkSmem& sm) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int k = p.top_k, G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);
  if (tid < G1) sm.fu[tid] = __ldg(p.uniforms + b * G1 + tid);
  if (tid < G) sm.fa[tid] = (float)__ldcg(p.acc + b * G + tid);
  if (tid == 0) sm.status = __ldcg(&p.seq[b].status);
  __syncthreads();
  if (p.ql) {
    if (tid < gb) {
      const int d = __ldg(p.draft + b * G + tid);
      float a = 0.f;
      int bits = 0;
      if (d < 0 || d >= V) {
        bits |= SEQ_OOB;
      } else {
        const float pd = kept_prob(p.rowres + (size_t)(b * G1 + tid) * (k + 1), d);
        const float qd = kept_prob(p.qrowres + (size_t)(b * G + tid) * (k + 1), d);
        if (qd > 0.f) {
          a = fminf(1.f, pd / qd);
        } else {
          a = pd > 0.f ? 1.f : 0.f;
          bits |= SEQ_QBAD;
        }
      }
      sm.fa[tid] = a;
      if (p.out_a) p.out_a[b * G + tid] = a;
      if (bits) atomicOr(&sm.status, bits);
    }
    __syncthreads();
  }
  if (tid == 0) {
    int n = gb;
    for (int i = 0; i < gb; ++i)
      if (!(sm.fu[i] < sm.fa[i])) { n = i; break; }
    sm.n = n;
  }
  __syncthreads();
  const int n = sm.n;
  const int2* kept = p.rowres + (size_t)(b * G1 + n) * (k + 1);
  const int J = __ldcg(kept).x;
  const bool resid = n < gb;
  const float* qrow = (resid && p.q) ? p.q + ((size_t)b * G + n) * V : nullptr;
  const int2* qlist = (resid && p.ql) ? p.qrowres + (size_t)(b * G + n) * (k + 1) : nullptr;
  // deterministic draft: q_n one-hot
  const int dn = (resid && !p.q && !p.ql) ? __ldg(p.draft + b * G + n) : -1;
  for (int e = tid; e < J; e += nt) {
    const int2 en = __ldcg(kept + 1 + e);
    sm.widx[e] = en.x;
    sm.w[e] = __int_as_float(en.y);
  }
  __syncthreads();
  // kept entries in token order; weights r_j = max(p_j - q_j, 0), or p_j
  F2* rs = reinterpret_cast<F2*>(sm.cand);
  for (int e = tid; e < J; e += nt) {
    const int me = sm.widx[e];
    int rank = 0;
    for (int j = 0; j < J; ++j) rank += sm.widx[j] < me;
    const float pe = sm.w[e];
    const float qm = qlist ? kept_prob(qlist, me) : qrow ? __ldg(qrow + me) : (me == dn ? 1.f : 0.f);
    const float r = resid ? fmaxf(__fsub_rn(pe, qm), 0.f) : pe;
    sm.sidx[rank] = me;
    rs[rank] = F2{r, 0.f};
  }
  __syncthreads();
  const float u = sm.fu[gb];
  F2 R{0.f, 0.f}, base{0.f, 0.f}, tgt{0.f, 0.f};
  int pos = locate(rs, J, u, &R, &base, &tgt, sm.loc, false);
  int status = sm.status;
  if (resid && !f2_pos(R)) {
    status |= SEQ_RESID0;   // zero residual mass (rounding only): draw from p_n
    for (int e = tid; e < J; e += nt) {
      const int me = sm.widx[e];
      int rank = 0;
      for (int j = 0; j < J; ++j) rank += sm.widx[j] < me;
      rs[rank] = F2{sm.w[e], 0.f};
    }
    __syncthreads();
    pos = locate(rs, J, u, &R, &base, &tgt, sm.loc, false);
  }
  if (tid == 0) {
    int tok = pos >= 0 ? sm.sidx[pos] : (J > 0 ? sm.sidx[0] : 0);
    if (tok < 0 || tok >= V) tok = 0;
    sm.token = tok;
    p.out_n[b] = n;
    if (p.out_status) p.out_status[b] = status;
    p.seq[b].status = 0;
  }
  __syncthreads();
  for (int j = tid; j < G1; j += nt)
    p.out_tokens[b * G1 + j] = j < n ? __ldg(p.draft + b * G + j) : (j == n ? sm.token : -1);
  if (p.out_a)
    for (int j = gb + tid; j < G; j += nt) p.out_a[b * G + j] = 0.f;   // beyond this sequence's drafts
  // the kept lists and acceptance probabilities have been consumed: zero them
  for (int e = tid; e < G1 * (k + 1); e += nt) p.rowres[(size_t)b * G1 * (k + 1) + e] = make_int2(0, 0);
  if (p.ql)
    for (int e = tid; e < G * (k + 1); e += nt) p.qrowres[(size_t)b * G * (k + 1) + e] = make_int2(0, 0);
  for (int e = tid; e < G; e += nt) p.acc[b * G + e] = 0.0;
}

// Per-row epilogue of the top-k path: softmax(./T) over the row's top-k (in
// sm.w / sm.widx [0, kk), descending by (logit, -index)), the top-p cut with
// two-float sums, the kept
// (index, probability) list written to rowres[r], and the acceptance
// probability of the row's draft (d_row, q_row prefetched by thread 0).
// out: where the kept list goes (rowres for a target row; for a draft row,
// with q formed from the draft's logits, its own list, which q is read from).
// A draft row with no distribution keeps nothing (q = 0); a draft row tests
// no draft, and with q from the draft's logits the acceptance tests move to
// the sequence finisher (q_i(d_i) comes from draft row i's list).
__device__ void topk_row_epilogue(const Params& p, int b, int i, int gb, int2* out, int kk, bool bad_nan, int d_row,
                                  float q_row, TopkSmem& sm, bool draft_row = false) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
  const int G = p.gamma, V = p.V;
    // ---- softmax(./T) over the top-k, then the top-p cut (two-float sums)
    const float m0 = kk > 0 ? sm.w[0] : -INFINITY;
    const bool bad = bad_nan || !(m0 > -INFINITY && m0 < INFINITY);
    __syncthreads();   // every thread has read w[0]
    for (int e = tid; e < kk; e += nt) sm.w[e] = bad ? 0.f : exp2f((sm.w[e] - m0) * p.c);
    __syncthreads();
    if (warp == 0) {
      // one inclusive two-float scan of the k weights in rank order: its last
      // value is the total W, and the prefixes (kept in cand, free by now)
      // give the top-p cut without a second pass of shuffles
      F2* pre = reinterpret_cast<F2*>(sm.cand);
      F2 carry{0.f, 0.f};
      for (int c0 = 0; c0 < kk; c0 += 32) {
        const int e = c0 + lane;
        const F2 inc = f2_add(carry, warp_incl_scan_f2(F2{e < kk ? sm.w[e] : 0.f, 0.f}));
        if (e < kk) pre[e] = inc;
        carry = F2{__shfl_sync(0xffffffffu, inc.hi, 31), __shfl_sync(0xffffffffu, inc.lo, 31)};
      }
      __syncwarp();
      const F2 W = carry;
      int J = kk;
      F2 WJ = W;
      if (bad || kk == 0) {
        J = (kk > 0 && !draft_row) ? 1 : 0;
        WJ = F2{1.f, 0.f};
        if (lane == 0 && J > 0) sm.w[0] = 1.f;
      } else if (p.top_p < 1.0f) {
        const F2 target = f2_scale(W, p.top_p);   // cumulative mass / W >= top_p
        for (int c0 = 0; c0 < kk; c0 += 32) {
          const int e = c0 + lane;
          const F2 inc = e < kk ? pre[e] : W;
          const unsigned hit = __ballot_sync(0xffffffffu, e < kk && !f2_lt(inc, target));
          if (hit) {
            const int first = __ffs(hit) - 1;
            J = c0 + first + 1;
            WJ = F2{__shfl_sync(0xffffffffu, inc.hi, first), __shfl_sync(0xffffffffu, inc.lo, first)};
            break;
          }
        }
      }
      const float wj = WJ.hi + WJ.lo;
      // the acceptance probability of this row's draft (thread 0 holds d_row, q_row)
      const int d = __shfl_sync(0xffffffffu, d_row, 0);
      float pd = 0.f;
      if (i < gb && !draft_row && !p.ql && d >= 0 && d < V) {
        for (int c0 = 0; c0 < J; c0 += 32) {
          const int e = c0 + lane;
          const unsigned hit = __ballot_sync(0xffffffffu, e < J && sm.widx[e] == d);
          if (hit) {
            const int l = __ffs(hit) - 1;
            pd = __shfl_sync(0xffffffffu, e < J ? sm.w[e] : 0.f, l) / wj;
            break;
          }
        }
      }
      if (lane == 0) {
        sm.J = J;
        sm.WJ = wj;
        if (bad && i <= gb && !draft_row) atomicOr(&p.seq[b].status, SEQ_BADROW);
        if (i < gb && !draft_row && !p.ql) {
          float a = 0.f;
          int st = 0;
          if (d < 0 || d >= V) {
            st |= SEQ_OOB;
          } else if (q_row > 0.0f) {
            a = fminf(1.f, pd / q_row);
          } else {
            a = pd > 0.f ? 1.f : 0.f;
            st |= SEQ_QBAD;
          }
          if (st) atomicOr(&p.seq[b].status, st);
          p.acc[b * G + i] = (double)a;
          if (p.out_a) p.out_a[b * G + i] = a;
        }
      }
    }
    __syncthreads();
    const int J = sm.J;
    const float WJ = sm.WJ;
    if (tid == 0) out[0] = make_int2(J, 0);
    for (int e = tid; e < J; e += nt) out[1 + e] = make_int2(sm.widx[e], __float_as_int(sm.w[e] / WJ));
}

// One entry of a vocabulary shard's candidate list (16 bytes): the
// comparison key of (logit, global index) (comp_key; 0 = empty) and, for a
// drafted row, q at that token.  Entry 0 of a row's record is its header:
// key = number of entries, q = q at the row's draft token (when the shard
// holds it), aux = SH_HAS_D | SH_NAN.
struct ShardCand {
  unsigned long long key;
  float q;
  int aux;
};

// Record of row r for the shard steps: the row's top min(k, N) in rank
// order (sm.w logits, sm.widx local indices) with q of draft row i at each
// (one-hot at d_i when q is NULL), then empty entries up to k.
__device__ void topk_shard_candidates(const Params& p, int r, int b, int i, int kk, bool bad_nan, int d_row,
                                      float q_row, TopkSmem& sm) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int k = p.top_k, G = p.gamma, V = p.V;
  ShardCand* rec = static_cast<ShardCand*>(p.sh_out) + (size_t)r * (k + 1);
  if (tid == 0) {
    const bool has = i < G && d_row >= 0 && d_row < V;
    ShardCand h;
    h.key = (unsigned long long)kk;
    h.q = has ? q_row : 0.f;
    h.aux = (has ? 1 : 0) | (bad_nan ? 2 : 0);   // SH_HAS_D, SH_NAN
    rec[0] = h;
    sm.token = d_row;
  }
  __syncthreads();
  const int dl = sm.token;
  const float* qrow = (i < G && p.q) ? p.q + ((size_t)b * G + i) * V : nullptr;
  for (int e = tid; e < k; e += nt) {
    ShardCand c;
    c.key = 0ull;
    c.q = 0.f;
    c.aux = 0;
    if (e < kk) {
      const int idx = sm.widx[e];
      c.key = comp_key(sm.w[e], p.v0 + idx);
      if (i < G) c.q = qrow ? __ldg(qrow + idx) : (idx == dl ? 1.f : 0.f);
    }
    rec[1 + e] = c;
  }
}

}  // namespace sv
