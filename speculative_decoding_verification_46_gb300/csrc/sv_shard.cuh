// Vocabulary-sharded verify: the logits and q of every row are split into
// contiguous token ranges, one per process (the layout a tensor-parallel
// output layer leaves).  The verify round ("11.1 核心原理", section 11.1.2:
// the acceptance test min(1, p/q), the first rejection, then one draw from
// norm(max(p_n - q_n, 0)) or from p_gamma) needs, per row, the softmax
// normaliser over the whole vocabulary and, for the final draw, the inverse
// CDF over the whole row n: both are sums over tokens, so each shard reduces
// its own range and the shards exchange a few numbers per row.
//
// Per call (every shard runs the same steps; the caller moves the records):
//   1. shard_stats_kernel: per row, this shard's maximum, sum of
//      2^((x - m) c) (two-float), first argmax, and the target logit and q at
//      the draft token if the token is in this shard's range.
//   2. (caller: all-gather of the records, shards in token order)
//   3. shard_scan_kernel: the rows' global statistics merged in shard order
//      (identically on every shard), a_i, n, every output but the final draw;
//      greedy is complete here.
//   4. final_draw_kernel in shard mode 1: the item sums of this shard's part
//      of row n and their totals (sum S, sum A, sum Q).
//   5. (caller: all-gather of the totals)
//   6. shard_pick_kernel: the global normaliser s = sum of the shards' S, each
//      shard's residual mass A - (s - s') Q, the target u R, and the shard
//      holding it; that shard searches its own items and writes the token,
//      every other shard writes -1 at that position.
//   7. (caller: element-wise maximum of out_tokens over the shards)
#pragma once

#include "sv_device.cuh"
#include "sv_final.cuh"
#include "sv_topk.cuh"

namespace sv {

constexpr int kShThreads = 256;
constexpr int kShWarps = kShThreads / 32;
constexpr int kMaxShards = 32;

// One row's record from one shard (32 bytes).
struct ShardStat {
  float m;          // maximum logit of the shard's range (NaN if one was NaN)
  float s_hi, s_lo; // sum over the range of 2^((x - m) c), two-float (sampling)
  int arg;          // first index (global) of the maximum (greedy)
  float ld, qd;     // target logit and q at the row's draft token, if it is in the range
  int flags;        // SH_HAS_D: ld, qd are set; SH_NAN: the range holds a NaN
  int pad;
};
enum { SH_HAS_D = 1, SH_NAN = 2 };

// Step 1: one CTA per row of this shard's logits [B][gamma+1][V] (V = the
// shard's range, tokens v0 .. v0 + V - 1 of the vocabulary).
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kShThreads) shard_stats_kernel(const Params p) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int r = blockIdx.x;
  const int b = r / G1, i = r - b * G1;
  const T* row = static_cast<const T*>(p.logits) + (size_t)r * V;
  const bool vec = (V % VW) == 0;
  const int NVv = (V + VW - 1) / VW;
  // the draft token's logit and q, loaded first (they overlap the row's read)
  int has_d = 0;
  float ld = 0.f, qd = 0.f;
  if (tid == 0 && i < G) {
    const int d = __ldg(p.draft + b * G + i);
    const int dl = d - p.v0;
    if (d >= 0 && dl >= 0 && dl < V) {
      has_d = 1;
      ld = TR::get(load_slot<T>(row, dl, 1, false), 0);
      if (!GREEDY) qd = p.q ? __ldg(p.q + ((size_t)b * G + i) * V + dl) : 1.f;   // NULL: one-hot draft
    }
  }
  float best = -INFINITY;
  int best_i = 0x7fffffff, nan = 0;
  float m = -INFINITY, s0 = 0.f, s1 = 0.f;
  for (int j = tid; j < NVv; j += kShThreads) {
    const int e = j * VW;
    const int nv = min(VW, V - e);
    const uint4 x = load_slot<T>(row, e, nv, vec && nv == VW);
    if (GREEDY) {
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        if (t < nv) {
          const float xv = TR::get(x, t);
          nan |= (xv != xv);
          if (argmax_better(xv, e + t, best, best_i)) {
            best = xv;
            best_i = e + t;
          }
        }
      }
    } else {
      float vm = -INFINITY;
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        if (t < nv) {
          const float xv = TR::get(x, t);
          nan |= (xv != xv);
          vm = fmaxf(vm, xv);
        }
      }
      if (vm > m) {
        const float sc = (m == -INFINITY) ? 0.f : ex2_approx((m - vm) * p.c);
        s0 *= sc;
        s1 *= sc;
        m = vm;
      }
      if (m > -INFINITY && m < INFINITY) {
        const float mc = m * p.c;
#pragma unroll
        for (int t = 0; t < VW; t += 2) {
          if (t < nv) s0 += ex2_approx(fmaf(TR::get(x, t), p.c, -mc));
          if (t + 1 < nv) s1 += ex2_approx(fmaf(TR::get(x, t + 1), p.c, -mc));
        }
      }
    }
  }
  __shared__ float4 red[kShWarps];
  nan = __syncthreads_or(nan);
  if (GREEDY) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
      if (argmax_better(ov, oi, best, best_i)) { best = ov; best_i = oi; }
    }
    if (lane == 0) red[warp] = make_float4(best, __int_as_float(best_i), 0.f, 0.f);
  } else {
    float M = m;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    F2 acc{0.f, 0.f};
    if (m > -INFINITY && M < INFINITY) {
      const float sc = ex2_approx((m - M) * p.c);
      acc = f2_add(F2{s0 * sc, 0.f}, F2{s1 * sc, 0.f});
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc = f2_add(acc, f2_shfl_xor(acc, o));
    if (lane == 0) red[warp] = make_float4(M, acc.hi, acc.lo, 0.f);
  }
  __syncthreads();
  if (tid == 0) {
    ShardStat o{};
    if (GREEDY) {
      float bv = red[0].x;
      int bi = __float_as_int(red[0].y);
      for (int w = 1; w < kShWarps; ++w) {
        const float ov = red[w].x;
        const int oi = __float_as_int(red[w].y);
        if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      o.m = bv;
      o.arg = bi == 0x7fffffff ? p.v0 : p.v0 + bi;
    } else {
      float Mb = red[0].x;
      for (int w = 1; w < kShWarps; ++w) Mb = fmaxf(Mb, red[w].x);
      F2 t{0.f, 0.f};
      if (Mb > -INFINITY && Mb < INFINITY) {
        for (int w = 0; w < kShWarps; ++w) {
          if (red[w].x > -INFINITY) {
            const float sc = ex2_approx((red[w].x - Mb) * p.c);
            t = f2_add(t, f2_add(F2{red[w].y * sc, 0.f}, F2{red[w].z * sc, 0.f}));
          }
        }
      }
      o.m = Mb;
      o.s_hi = t.hi;
      o.s_lo = t.lo;
      o.arg = 0;
    }
    o.ld = ld;
    o.qd = qd;
    o.flags = (has_d ? SH_HAS_D : 0) | (nan ? SH_NAN : 0);
    reinterpret_cast<ShardStat*>(p.sh_out)[r] = o;
  }
}

// Step 3: one warp per sequence.  Rows i = lane, lane + 32, lane + 64 (i <=
// gamma); each merges its S records in shard order: M = max m_r, s = sum
// s_r 2^((m_r - M) c), the argmax by (value, lowest index), and the draft's
// logit and q from the shard that holds the token.  Then the acceptance scan
// of the unsharded path; greedy writes every output, sampling every output
// but the final token and leaves row n's state in seq[b] for steps 4 and 6.
template <bool GREEDY>
__global__ void __launch_bounds__(kShThreads) shard_scan_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kShWarps + (threadIdx.x >> 5);
  if (b >= p.B) return;
  const int G = p.gamma, G1 = G + 1, S = p.nshard, Vg = p.Vg;
  const ShardStat* all = static_cast<const ShardStat*>(p.sh_in);
  const size_t stride = (size_t)p.B * G1;   // records of one shard
  float rM[3], ld[3], qd[3];
  F2 rS[3];
  int arg[3], nan[3], hasd[3];
#pragma unroll
  for (int h = 0; h < 3; ++h) {
    const int i = lane + 32 * h;
    rM[h] = -INFINITY;
    rS[h] = F2{0.f, 0.f};
    arg[h] = 0x7fffffff;
    nan[h] = 0;
    hasd[h] = 0;
    ld[h] = qd[h] = 0.f;
    if (i < G1) {
      const ShardStat* rec = all + (size_t)b * G1 + i;
      if (GREEDY) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int r = 0; r < S; ++r) {
          const ShardStat x = rec[r * stride];
          nan[h] |= (x.flags & SH_NAN) != 0;
          if (argmax_better(x.m, x.arg, bv, bi)) { bv = x.m; bi = x.arg; }
          if (x.flags & SH_HAS_D) hasd[h] = 1;
        }
        rM[h] = bv;
        arg[h] = bi;
      } else {
        float M = -INFINITY;
        for (int r = 0; r < S; ++r) {
          const ShardStat x = rec[r * stride];
          nan[h] |= (x.flags & SH_NAN) != 0;
          M = fmaxf(M, x.m);
          if (x.flags & SH_HAS_D) {
            hasd[h] = 1;
            ld[h] = x.ld;
            qd[h] = x.qd;
          }
        }
        F2 t{0.f, 0.f};
        if (M > -INFINITY && M < INFINITY) {
          for (int r = 0; r < S; ++r) {
            const ShardStat x = rec[r * stride];
            if (x.m > -INFINITY) t = f2_add(t, f2_scale(F2{x.s_hi, x.s_lo}, ex2_approx((x.m - M) * p.c)));
          }
        }
        rM[h] = M;
        rS[h] = t;
      }
    }
  }
  const int gb = G;
  int bits = 0;
  unsigned rej[2] = {0u, 0u};
  float a[2] = {0.f, 0.f};
  int bad_any = 0;
#pragma unroll
  for (int h = 0; h < 3; ++h) {
    const int i = lane + 32 * h;
    bool badrow = false;
    if (i <= gb) {
      if (GREEDY) badrow = nan[h] != 0;
      else badrow = nan[h] != 0 || !(rM[h] > -INFINITY && rM[h] < INFINITY) || !(rS[h].hi > 0.f && rS[h].hi < INFINITY);
    }
    bad_any |= badrow;
    if (h < 2) {
      bool r = false;
      if (i < gb) {
        const int d = __ldg(p.draft + b * G + i);
        if (d < 0 || d >= Vg || !hasd[h]) {
          bits |= SEQ_OOB;
          r = true;
        } else if (GREEDY) {
          const int g = (nan[h] || arg[h] == 0x7fffffff) ? 0 : arg[h];
          r = d != g;
        } else {
          const float ssum = rS[h].hi + rS[h].lo;
          const float pd = badrow ? 0.f : exp2f((ld[h] - rM[h]) * p.c) / ssum;
          if (qd[h] > 0.f) {
            a[h] = fminf(1.f, pd / qd[h]);
          } else {
            a[h] = pd > 0.f ? 1.f : 0.f;
            bits |= SEQ_QBAD;
          }
          r = !(__ldg(p.uniforms + b * G1 + i) < a[h]);
        }
      }
      rej[h] = __ballot_sync(0xffffffffu, r);
    }
  }
  const int n = rej[0] ? __ffs(rej[0]) - 1 : (rej[1] ? 32 + __ffs(rej[1]) - 1 : gb);
  bits = __reduce_or_sync(0xffffffffu, bits);
  if (__any_sync(0xffffffffu, bad_any)) bits |= SEQ_BADROW;
  // row n's statistics from lane n mod 32
  const int hn = n >> 5, ln = n & 31;
  const float Mn = __shfl_sync(0xffffffffu, hn == 0 ? rM[0] : (hn == 1 ? rM[1] : rM[2]), ln);
  const float Sh = __shfl_sync(0xffffffffu, hn == 0 ? rS[0].hi : (hn == 1 ? rS[1].hi : rS[2].hi), ln);
  const float Sl = __shfl_sync(0xffffffffu, hn == 0 ? rS[0].lo : (hn == 1 ? rS[1].lo : rS[2].lo), ln);
  const int An = __shfl_sync(0xffffffffu, hn == 0 ? arg[0] : (hn == 1 ? arg[1] : arg[2]), ln);
  const int Nn = __shfl_sync(0xffffffffu, hn == 0 ? nan[0] : (hn == 1 ? nan[1] : nan[2]), ln);
#pragma unroll
  for (int h = 0; h < 3; ++h) {
    const int i = lane + 32 * h;
    if (!GREEDY && p.out_a && i < G) p.out_a[b * G + i] = i < gb ? a[h < 2 ? h : 0] : 0.f;
    if (i < G1 && i != n) p.out_tokens[b * G1 + i] = i < n ? __ldg(p.draft + b * G + i) : -1;
  }
  if (lane == 0) {
    p.out_n[b] = n;
    if (GREEDY) {
      p.out_tokens[b * G1 + n] = (Nn || An == 0x7fffffff) ? 0 : An;
      if (p.out_status) p.out_status[b] = bits;
    } else {
      SeqState st;
      st.n = n;
      st.status = bits;
      st.M = Mn;
      st.qm = 0.f;
      st.s = (double)(Sh + Sl);
      st.qinv = 0.f;
      st.qbad = 0;
      st.tpK = 0u;
      st.tpIdx = 0;
      p.seq[b] = st;
    }
  }
}

// Step 6: one CTA per sequence.  The shards' totals (8 floats each,
// [S][B][8]) give s = sum S_r, s - s', each shard's mass R_r (A_r - (s - s')
// Q_r clamped at 0 after a rejection, S_r for the bonus draw or when the
// residual has no mass), R = sum R_r and t = u R.  The owner is the last
// shard with R_r > 0 whose start (sum of the masses before it) is <= t; it
// searches its items with target t - start and writes v0 + token at
// out_tokens[b][n]; every other shard writes -1 there (the caller's maximum
// over shards keeps the owner's).  Status: the scan's bits, SEQ_RESID0 when
// the residual had no mass.  The items, the state and the ticket are zeroed
// behind.
template <typename T>
__global__ void __launch_bounds__(kFdThreads, 1) shard_pick_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char sh_dyn[];
  __shared__ FdSmem sm;
  __shared__ FdGiven gv;
  __shared__ int owner_s, resid0_s;
  load_exp2_table(sm.tab);
  const int tid = threadIdx.x, lane = tid & 31;
  const int b = blockIdx.x;
  const int G1 = p.gamma + 1, S = p.nshard, C = p.FC;
  FdSeq<T> s;
  fd_load_state<T>(p, b, s);
  if (tid < 32) {
    const float* tot = static_cast<const float*>(p.sh_in);
    F2 Sr{0.f, 0.f}, Ar{0.f, 0.f};
    float Qr = 0.f;
    if (lane < S) {
      const float4 x = *reinterpret_cast<const float4*>(tot + ((size_t)lane * p.B + b) * 8);
      Sr = F2{x.x, x.y};
      Ar = F2{x.z, x.w};
      Qr = tot[((size_t)lane * p.B + b) * 8 + 4];
    }
    F2 st = Sr;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) st = f2_add(st, f2_shfl_xor(st, o));
    const F2 ds = f2_add(st, F2{-s.s_a, 0.f});
    const bool resid = s.n < s.gb;
    bool use_q = resid;
    int resid0 = 0;
    F2 Rr{0.f, 0.f}, R{0.f, 0.f}, start{0.f, 0.f};
    for (int attempt = 0; attempt < 2; ++attempt) {
      Rr = Sr;
      if (use_q) {
        Rr = f2_add(Ar, f2_neg(f2_scale(ds, Qr)));
        if (Rr.hi < 0.f) Rr = F2{0.f, 0.f};
      }
      const F2 inc = warp_incl_scan_f2(Rr);
      R = F2{__shfl_sync(0xffffffffu, inc.hi, 31), __shfl_sync(0xffffffffu, inc.lo, 31)};
      start = f2_shfl_up(inc, 1);
      if (lane == 0) start = F2{0.f, 0.f};
      if (resid && use_q && !f2_pos(R)) {
        resid0 = 1;
        use_q = false;
        continue;
      }
      break;
    }
    const F2 t = f2_scale(R, __ldg(p.uniforms + b * G1 + s.gb));
    const bool cand = lane < S && f2_pos(Rr) && !f2_lt(t, start);
    const unsigned hit = __ballot_sync(0xffffffffu, cand);
    const int own = (s.mode == FD_SKIP || !f2_pos(R) || !hit) ? -1 : 31 - __clz(hit);
    if (own >= 0 && lane == own) {
      gv.on = 1;
      gv.use_q = use_q;
      gv.ds = ds;
      gv.t = f2_add(t, f2_neg(start));
    }
    if (lane == 0) {
      owner_s = own;
      resid0_s = resid0;
    }
  }
  __syncthreads();
  const int own = owner_s;
  int token = -1;
  if (own == p.rank) {
    int r0 = 0;
    token = p.v0 + fd_pick_block<T, false>(p, b, s, sm, sh_dyn, &r0, gv);
  } else {
    for (int k = tid; k < C; k += kFdThreads) {
      p.fd_part[(size_t)b * C + k] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.fd_q[(size_t)b * C + k] = 0.f;
    }
    if (own < 0 && p.rank == 0) token = 0;   // no mass anywhere: an in-range token from one shard
  }
  if (tid == 0) {
    p.out_tokens[b * G1 + s.n] = token;
    if (p.out_status) p.out_status[b] = s.status | (resid0_s ? SEQ_RESID0 : 0);
    SeqState zs;
    zs.n = 0; zs.status = 0; zs.M = 0.f; zs.qm = 0.f; zs.s = 0.0; zs.qinv = 0.f; zs.qbad = 0; zs.tpK = 0u; zs.tpIdx = 0;
    p.seq[b] = zs;
  }
}

// ---- truncated sampling over vocabulary shards (top-k, then top-p)
//
// Every token of a row's global top-k is in the top-k of the shard holding
// it, so the shards' candidate lists (stream_topk_kernel in shard mode 2:
// each list the shard's k best by (logit, lowest index), with q of the
// drafted row at each) hold the whole truncated distribution and the q it
// needs: one all-gather, then shard_topk_finish_kernel runs the rest of the
// round identically on every shard.
constexpr int kShCandMax = 2048;   // nshard * top_k entries merged per row

struct ShTopkSmem {
  unsigned long long key[kShCandMax];
  float q[kShCandMax];
  unsigned long long tkey[kMaxK];   // the row's top-k in rank order
  float tq[kMaxK];
  float w[kMaxK];                   // their weights, then the kept probabilities
  F2 rs[kMaxK];                     // final draw: residual weights in token order
  int sidx[kMaxK];
  float a[kMaxG1];
  LocateSmem loc;
  int N, J, nan, bad, hasd, n, status, token;
  float qd, WJ;
};

// Row i of sequence b: merge the shards' lists into the top-k (exact ranks
// over the union), softmax over them, the top-p cut; leaves the kept
// probabilities in w[0..J) (rank order) with tkey / tq, J, and the row's NaN
// flag and the draft's q (from the shard holding it) in sm.  Returns J.
__device__ int sh_topk_row(const Params& p, int b, int i, ShTopkSmem& sm) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int S = p.nshard, k = p.top_k, G1 = p.gamma + 1;
  const ShardCand* all = static_cast<const ShardCand*>(p.sh_in);
  const size_t rowrec = (size_t)(k + 1), shardrec = (size_t)p.B * G1 * rowrec;
  if (tid == 0) {
    sm.nan = 0;
    sm.hasd = 0;
    sm.qd = 0.f;
    sm.N = 0;
  }
  __syncthreads();
  for (int e = tid; e < S * k; e += nt) {
    const int r = e / k, j = e - r * k;
    const ShardCand c = all[r * shardrec + ((size_t)b * G1 + i) * rowrec + 1 + j];
    sm.key[e] = c.key;
    sm.q[e] = c.q;
  }
  if (tid < S) {
    const ShardCand h = all[tid * shardrec + ((size_t)b * G1 + i) * rowrec];
    if (h.aux & 2) atomicOr(&sm.nan, 1);
    if (h.aux & 1) {   // at most one shard holds the draft token
      sm.hasd = 1;
      sm.qd = h.q;
    }
  }
  __syncthreads();
  // exact ranks among the union (keys are distinct: the index is in them)
  int cnt = 0;
  for (int e = tid; e < S * k; e += nt) {
    const unsigned long long me = sm.key[e];
    if (me == 0ull) continue;
    ++cnt;
    int rank = 0;
    for (int j = 0; j < S * k; ++j) rank += sm.key[j] > me;
    if (rank < k) {
      sm.tkey[rank] = me;
      sm.tq[rank] = sm.q[e];
    }
  }
  if (cnt) atomicAdd(&sm.N, cnt);
  __syncthreads();
  const int kk = min(k, sm.N);
  // softmax(./T) over the top-k, then the top-p cut (the unsharded epilogue's rule)
  const float m0 = kk > 0 ? comp_val(sm.tkey[0]) : -INFINITY;
  const bool bad = sm.nan || !(m0 > -INFINITY && m0 < INFINITY);
  for (int e = tid; e < kk; e += nt) sm.w[e] = bad ? 0.f : exp2f((comp_val(sm.tkey[e]) - m0) * p.c);
  if (tid == 0) sm.bad = bad;
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    F2* pre = sm.rs;   // scratch for the prefixes
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
      J = kk > 0 ? 1 : 0;
      WJ = F2{1.f, 0.f};
      if (lane == 0 && J > 0) sm.w[0] = 1.f;
    } else if (p.top_p < 1.0f) {
      const F2 target = f2_scale(W, p.top_p);
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
    if (lane == 0) {
      sm.J = J;
      sm.WJ = WJ.hi + WJ.lo;
    }
  }
  __syncthreads();
  const int J = sm.J;
  const float WJ = sm.WJ;
  for (int e = tid; e < J; e += nt) sm.w[e] = sm.w[e] / WJ;
  __syncthreads();
  return J;
}

// One CTA per sequence: rows 0..gamma through sh_topk_row, a_i, n, then the
// final draw over row n's kept list in token order (residual max(p - q, 0)
// with q from the candidate entries, or p_gamma); every output.
__global__ void __launch_bounds__(kShThreads) shard_topk_finish_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char shk_dyn[];
  ShTopkSmem& sm = *reinterpret_cast<ShTopkSmem*>(shk_dyn);
  const int tid = threadIdx.x, nt = blockDim.x;
  const int b = blockIdx.x;
  const int G = p.gamma, G1 = G + 1, Vg = p.Vg;
  const int gb = G;
  if (tid == 0) sm.status = 0;
  for (int i = 0; i < gb; ++i) {
    const int J = sh_topk_row(p, b, i, sm);
    if (tid == 0) {
      int st = sm.bad ? SEQ_BADROW : 0;
      const int d = __ldg(p.draft + b * G + i);
      float a = 0.f;
      if (d < 0 || d >= Vg || !sm.hasd) {
        st |= SEQ_OOB;
      } else {
        float pd = 0.f;
        for (int e = 0; e < J; ++e)
          if (comp_idx(sm.tkey[e]) == d) pd = sm.w[e];
        if (sm.qd > 0.f) {
          a = fminf(1.f, pd / sm.qd);
        } else {
          a = pd > 0.f ? 1.f : 0.f;
          st |= SEQ_QBAD;
        }
      }
      sm.a[i] = a;
      sm.status |= st;
      if (p.out_a) p.out_a[b * G + i] = a;
    }
    __syncthreads();
  }
  if (tid == 0) {
    int n = gb;
    for (int i = 0; i < gb; ++i)
      if (!(__ldg(p.uniforms + b * G1 + i) < sm.a[i])) { n = i; break; }
    sm.n = n;
  }
  __syncthreads();
  const int n = sm.n;
  // the bonus row defines no distribution: the round is flagged as the
  // unsharded path flags it (every row 0..gamma counts)
  if (n < gb) {
    sh_topk_row(p, b, gb, sm);
    if (tid == 0 && sm.bad) sm.status |= SEQ_BADROW;
    __syncthreads();
  }
  const int J = sh_topk_row(p, b, n, sm);
  if (tid == 0 && sm.bad) sm.status |= SEQ_BADROW;
  const bool resid = n < gb;
  // kept entries in token order: r = max(p - q, 0) after a rejection, else p
  for (int e = tid; e < J; e += nt) {
    const int me = comp_idx(sm.tkey[e]);
    int rank = 0;
    for (int j = 0; j < J; ++j) rank += comp_idx(sm.tkey[j]) < me;
    const float pe = sm.w[e];
    const float qm = sm.tq[e];   // q_n at the token (one-hot at d_n for NULL q: set by the candidates step)
    sm.sidx[rank] = me;
    sm.rs[rank] = F2{resid ? fmaxf(__fsub_rn(pe, qm), 0.f) : pe, 0.f};
  }
  __syncthreads();
  const float u = __ldg(p.uniforms + b * G1 + gb);
  F2 R{0.f, 0.f}, base{0.f, 0.f}, tgt{0.f, 0.f};
  int pos = locate(sm.rs, J, u, &R, &base, &tgt, sm.loc, false);
  int status = sm.status;
  if (resid && !f2_pos(R)) {
    status |= SEQ_RESID0;   // zero residual mass (rounding only): draw from p_n
    for (int e = tid; e < J; e += nt) {
      const int me = comp_idx(sm.tkey[e]);
      int rank = 0;
      for (int j = 0; j < J; ++j) rank += comp_idx(sm.tkey[j]) < me;
      sm.rs[rank] = F2{sm.w[e], 0.f};
    }
    __syncthreads();
    pos = locate(sm.rs, J, u, &R, &base, &tgt, sm.loc, false);
  }
  if (tid == 0) {
    int tok = pos >= 0 ? sm.sidx[pos] : (J > 0 ? sm.sidx[0] : 0);
    if (tok < 0 || tok >= Vg) tok = 0;
    sm.token = tok;
    p.out_n[b] = n;
    if (p.out_status) p.out_status[b] = status;
  }
  __syncthreads();
  for (int j = tid; j < G1; j += nt)
    p.out_tokens[b * G1 + j] = j < n ? __ldg(p.draft + b * G + j) : (j == n ? sm.token : -1);
}

}  // namespace sv
