// Final draw of untruncated sampling: the one categorical draw per sequence,
// from the residual norm(max(p_n - q_n, 0)) after a rejection at n, or from
// p_gamma when every draft was accepted ("11.1 核心原理", section 11.1.2 and
// listing 10-1; the notes "Fast Inference from Transformers via Speculative
// Decoding", speculative-sampling paragraph).  The draw is the inverse CDF in
// token-index order: the smallest v with sum_{w <= v} r(w) > u * sum(r).
//
// One kernel follows the row statistics (streaming kernel, rows kernel, or
// the top-p rows kernel): final_draw_kernel, one CTA per sequence (persistent
// over sequences), 16 warps.
//   - Every warp takes sequence b's state: it merges the streaming kernel's
//     row partials, forms p_i(d_i) and a_i = min(1, p_i(d_i) / q_i(d_i)) and
//     scans for the first rejection n (the first sequence's drafts, their
//     logits and q values are gathered before the dependency wait); warp 0
//     writes every output but the drawn token.
//   - Sequence b's row n is cut into items of 2048 tokens and the items into
//     Z parts, one CTA each.  Warp w of a part sums its items w, w + 16, ...
//     chunk by chunk (512 tokens) through a lane-private cp.async ring: no
//     block barriers and no cross-warp waits.
//     Per item: the weights w = 2^((x - M) c) (S), and over the residual
//     support {w > s' q} the differences w - s' q (A) and q (Q), s' the float
//     normaliser; four items' warp totals at a time by a transposed
//     butterfly.
//   - The CTA that completes a sequence's last part (an acquire-release
//     ticket) searches: exact normaliser s = sum S, item masses, the item
//     holding u * R, then the token among its 2048 (re-read from L2, four
//     per thread).
//
// Precision (the draw is compared with a float64 reference over up to 10^5
// CDF steps).  Tokens whose exponent (x - M) c is above -8 carry most of the
// mass: their weights and residuals are two-float (Tang's table exp2; the
// residual formed exactly).  Every other token's weight is ex2.approx with a
// first-order correction for the exponent's low part, and a lane adds its 16
// such tokens of a chunk in float32: each is below 2^-8 of the largest
// weight, so the rounding of these short sums stays at the level of the
// weights' own error.  Chunk sums, lane sums and everything above them are
// two-float.
// The exact normaliser s = sum S is formed at the end; the residual mass of
// an item is A - (s - s') Q.
#pragma once

#include "sv_device.cuh"
#include "sv_topp.cuh"

namespace sv {

constexpr int kFdThreads = 512;            // 16 warps, one CTA per SM
constexpr int kFdWarps = kFdThreads / 32;
constexpr int kFdChunk = 512;              // tokens per ring stage: 4 groups x 32 lanes x 4 tokens
constexpr int kFdChunks = 4;               // chunks per item
constexpr int kFdTok = kFdChunk * kFdChunks;   // tokens per item (one stored sum)

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
  static constexpr int S = sizeof(T) == 4 ? 3 : 4;        // stages (items) per warp: 192 KB in all
  static constexpr size_t bytes = (size_t)kFdWarps * S * stage_bytes;
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
template <int S>
__device__ __forceinline__ void fd_wait_ring() {
  asm volatile("cp.async.wait_group %0;" ::"n"(S - 1) : "memory");
}

// Warp-wide two-float sum (every lane gets it), and lane l's value in every lane.
__device__ __forceinline__ F2 warp_sum_f2(F2 v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = f2_add(v, f2_shfl_xor(v, m));
  return v;
}
__device__ __forceinline__ F2 f2_bcast(F2 v, int l) {
  return F2{__shfl_sync(0xffffffffu, v.hi, l), __shfl_sync(0xffffffffu, v.lo, l)};
}

// What the final draw needs about one sequence: row n, how q is given, the
// row statistics and where the rows are.
template <typename T>
struct FdSeq {
  int n, gb, mode, status;
  float M, s_a;         // row n's maximum and normaliser (float32 of the merged two-float sum)
  int xq;               // deterministic draft: the rejected draft's token
  float u;              // the final draw's uniform
  QLrow qlr;            // q formed from the draft's logits: row n's statistics
  uint32_t K;           // top-p alone: row n's kept set (key > K, or key == K
  int idx;              // and index <= idx)
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
    s.xq = __ldg(p.draft + b * G + s.n) - p.v0;   // a token index of this row (of the shard's slice)
  }
}

// The state a previous kernel left for sequence b (the rows path's finisher,
// or final_draw_kernel's scanning warp, for the search).
template <typename T>
__device__ __forceinline__ void fd_load_state(const Params& p, int b, FdSeq<T>& s) {
  const SeqState* sp = p.seq + b;
  s.n = __ldcg(&sp->n);
  s.gb = seq_gamma(p, b);
  s.status = __ldcg(&sp->status);
  s.M = __ldcg(&sp->M);
  s.s_a = (float)__ldcg(&sp->s);
  s.qlr = QLrow{__ldcg(&sp->qm), __ldcg(&sp->qinv), __ldcg(&sp->qbad) != 0};
  s.K = __ldcg(&sp->tpK);
  s.idx = __ldcg(&sp->tpIdx);
  // (the shard totals step has no uniforms: it draws nothing)
  s.u = p.uniforms ? __ldg(p.uniforms + b * (p.gamma + 1) + s.gb) : 0.f;
  fd_bind(p, b, s);
}

// Inputs of sequence b's acceptance tests for draft rows i = lane and
// lane + 32 (gamma <= 64): d_i, u_i, the target logit at d_i and q_i(d_i) (or
// the draft's logit at d_i).  Inputs only: gathered before the dependency
// wait when the sequence is known then.
struct FdDrafts {
  int d[2];
  float u[2], l[2], q[2];
  float uf;   // the final draw's uniform
};
template <typename T>
__device__ __forceinline__ void fd_gather(const Params& p, int b, FdDrafts& g) {
  const int lane = threadIdx.x & 31;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);
  g.uf = __ldg(p.uniforms + b * G1 + gb);
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
// no positive sum defines no distribution; nrows <= 65: three entries).  One
// aligned lane segment merges one row.
__device__ __forceinline__ void fd_merge_rows(const Params& p, const float4* base, long long r0g, int nrows,
                                              float m[3], F2 s[3], int bad[3]) {
  const int lane = threadIdx.x & 31;
  const int NP = stream_np(p);
  const int per = 32 / NP;   // rows merged per pass
  const int E = nrows * NP;
  m[0] = m[1] = m[2] = -INFINITY;
  s[0] = s[1] = s[2] = F2{0.f, 0.f};
  bad[0] = bad[1] = bad[2] = 1;
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
    for (int h = 0; h < 3; ++h) {
      const int row = lane + 32 * h;
      const int j = row - r0;
      const bool mine = j >= 0 && j < per && row < nrows;
      const int src = mine ? j * NP : 0;
      const float Mr = __shfl_sync(0xffffffffu, M, src);
      const float th = __shfl_sync(0xffffffffu, t.hi, src), tl = __shfl_sync(0xffffffffu, t.lo, src);
      if (mine) {
        m[h] = Mr;
        s[h] = F2{th, tl};
        // (th, tl) is normalised: the sum is positive and finite exactly when th is
        bad[h] = !(Mr > -INFINITY && Mr < INFINITY) || !(th > 0.f && th < INFINITY);
      }
    }
  }
}

// The acceptance scan of sequence b by one warp (streaming path): row
// statistics merged from the partials, a_i for i < gamma_b, n = the first
// rejected position (gamma_b if none), the status bits, and row n's state
// in s.  `writer`: this warp writes the outputs (all but the drawn token).
template <typename T>
__device__ __forceinline__ void fd_scan(const Params& p, int b, const FdDrafts& g, bool writer, FdSeq<T>& s) {
  const int lane = threadIdx.x & 31;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);
  const int NP = stream_np(p);
  float rM[3], qM[3];
  F2 rS[3], qS[3];
  int rBad[3], qBad[3];
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
        if (p.ql) qd = qBad[h] ? 0.f : q_weight(qd, qM[h], p.c, p.c_lo) * f2_rcp(qS[h]);
        const float ssum = rS[h].hi + rS[h].lo;   // the float32 rounding of the two-float sum
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
  if (__any_sync(0xffffffffu, (lane <= gb && rBad[0]) || (lane + 32 <= gb && rBad[1]) || (lane + 64 <= gb && rBad[2])))
    bits |= SEQ_BADROW;
  // row n's statistics (and its draft row's, with q from draft logits) from lane n mod 32
  const int hn = n >> 5, ln = n & 31;
  const float Mn = __shfl_sync(0xffffffffu, hn == 0 ? rM[0] : (hn == 1 ? rM[1] : rM[2]), ln);
  const float Sh = __shfl_sync(0xffffffffu, hn == 0 ? rS[0].hi : (hn == 1 ? rS[1].hi : rS[2].hi), ln);
  const float Sl = __shfl_sync(0xffffffffu, hn == 0 ? rS[0].lo : (hn == 1 ? rS[1].lo : rS[2].lo), ln);
  s.n = n;
  s.gb = gb;
  s.status = bits;
  s.u = g.uf;
  s.M = Mn;
  s.s_a = Sh + Sl;
  s.qlr = QLrow{0.f, 0.f, true};
  s.K = 0u;
  s.idx = 0;
  if (p.ql) {
    // (draft rows: n < gb <= 64 when they are read, so entries 0 and 1)
    const float qm = __shfl_sync(0xffffffffu, hn ? qM[1] : qM[0], ln);
    const float qh = __shfl_sync(0xffffffffu, hn ? qS[1].hi : qS[0].hi, ln);
    const float ql = __shfl_sync(0xffffffffu, hn ? qS[1].lo : qS[0].lo, ln);
    const int qb = __shfl_sync(0xffffffffu, hn ? qBad[1] : qBad[0], ln);
    if (n < gb) s.qlr = QLrow{qm, f2_rcp(F2{qh, ql}), qb != 0};
  }
  fd_bind(p, b, s);
  if (writer) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      if (p.out_a && i < G) p.out_a[b * G + i] = i < gb ? a[h] : 0.f;
      if (i < G1 && i != n) p.out_tokens[b * G1 + i] = i < n ? g.d[h] : -1;
    }
    // position 64 (gamma = 64): after a rejection at n < 64 it is padding
    if (lane == 0 && G1 > 64 && n != 64) p.out_tokens[b * G1 + 64] = -1;
    if (lane == 0) p.out_n[b] = n;
  }
}

// The acceptance scan of sequence b by one warp for top-p alone: the rows'
// records from topp_row_kernel hold a_i and the status bits; n = the first
// rejected position; row n's kept set and mass give the state.  `writer` as
// in fd_scan.
template <typename T>
__device__ __forceinline__ void fd_scan_tp(const Params& p, int b, bool writer, FdSeq<T>& s) {
  const int lane = threadIdx.x & 31;
  const int G = p.gamma, G1 = G + 1;
  const int gb = seq_gamma(p, b);
  const TpRow* tr = p.tp + (size_t)b * G1;
  int bits = 0, d[2] = {-1, -1};
  float a[2] = {0.f, 0.f};
  unsigned rej[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    bool r = false;
    if (i <= gb) {
      const int st = __ldcg(&tr[i].status);
      bits |= st & SEQ_BADROW;
      if (i < gb) {
        bits |= st & (SEQ_OOB | SEQ_QBAD);
        a[h] = __ldcg(&tr[i].a);
        d[h] = __ldg(p.draft + b * G + i);
        r = !(__ldg(p.uniforms + b * G1 + i) < a[h]);
      }
    }
    rej[h] = __ballot_sync(0xffffffffu, r);
  }
  if (lane == 0 && gb >= 64) bits |= __ldcg(&tr[64].status) & SEQ_BADROW;   // the bonus row of gamma_b = 64
  const int n = rej[0] ? __ffs(rej[0]) - 1 : (rej[1] ? 32 + __ffs(rej[1]) - 1 : gb);
  bits = __reduce_or_sync(0xffffffffu, bits);
  s.n = n;
  s.gb = gb;
  s.status = bits;
  s.M = __ldcg(&tr[n].M);
  s.s_a = __ldcg(&tr[n].Wh) + __ldcg(&tr[n].Wl);
  s.qlr = QLrow{0.f, 0.f, true};
  s.K = __ldcg(&tr[n].K);
  s.idx = __ldcg(&tr[n].idx);
  s.u = __ldg(p.uniforms + b * G1 + gb);
  fd_bind(p, b, s);
  if (writer) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      if (p.out_a && i < G) p.out_a[b * G + i] = i < gb ? a[h] : 0.f;
      if (i < G1 && i != n) p.out_tokens[b * G1 + i] = i < n ? d[h] : -1;
    }
    // position 64 (gamma = 64): after a rejection at n < 64 it is padding
    if (lane == 0 && G1 > 64 && n != 64) p.out_tokens[b * G1 + 64] = -1;
    if (lane == 0) p.out_n[b] = n;
  }
}

// One 4-token group of an unaligned row (V % 4 != 0), token by token: the
// logits, and q or the draft's logits when given.  Tokens past the row's end
// are not read.
template <typename T>
__device__ __noinline__ void fd_scalar_group(const T* row, const float* qrow, const T* qlrow, int t0, int V,
                                             unsigned char* ld, unsigned char* qd) {
  const uint32_t pad = Tr<T>::kPadWord;   // -inf in the logits' type
  for (int t = 0; t < 4; ++t) {
    const bool in = t0 + t < V;
    if (sizeof(T) == 4) reinterpret_cast<uint32_t*>(ld)[t] = in ? Tr<T>::scalar_bits(row + t0 + t) : pad;
    else reinterpret_cast<unsigned short*>(ld)[t] = (unsigned short)(in ? Tr<T>::scalar_bits(row + t0 + t) : pad);
    if (qrow) {
      reinterpret_cast<float*>(qd)[t] = in ? __ldg(qrow + t0 + t) : 0.f;
    } else if (qlrow) {
      if (sizeof(T) == 4) reinterpret_cast<uint32_t*>(qd)[t] = in ? Tr<T>::scalar_bits(qlrow + t0 + t) : pad;
      else reinterpret_cast<unsigned short*>(qd)[t] = (unsigned short)(in ? Tr<T>::scalar_bits(qlrow + t0 + t) : pad);
    }
  }
}

// Issue this lane's copies of the chunk starting at token tc of sequence s
// into one ring stage: logits groups g = 0..3 (tokens tc + 128 g + 4 lane ..
// + 3) and, for a
// residual, the matching q (or draft logit) groups.  vec: 4-token groups are
// aligned (V % 4 == 0); otherwise the in-range tokens are loaded one by one.
// Tokens past the end of the row are not read: their slots are filled with
// -inf logits and zero q, which the sweep gives weight 0 with no test.
template <typename T>
__device__ __forceinline__ void fd_issue(const FdSeq<T>& s, int tc, int V, bool vec, unsigned char* st) {
  using R = FdRing<T>;
  if (s.mode == FD_SKIP) return;
  const int lane = threadIdx.x & 31;
  unsigned char* lg = st + lane * R::LB;
  unsigned char* qg = st + 4 * 32 * R::LB + lane * R::QB;
  const int tl = tc + 4 * lane;   // this lane's first token; group g adds 128 g
  if (vec && tc + kFdChunk <= V) {
    // the whole chunk is inside the row: base addresses plus constant offsets
    const T* lrow = s.row + tl;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (R::LB == 16) fd_cp16(lg + g * 32 * R::LB, lrow + 128 * g); else fd_cp8(lg + g * 32 * R::LB, lrow + 128 * g);
    }
    if (s.mode == FD_DENSE) {
      const float* qr = s.qrow + tl;
#pragma unroll
      for (int g = 0; g < 4; ++g) fd_cp16(qg + g * 32 * R::QB, qr + 128 * g);
    } else if (s.mode == FD_QL) {
      const T* qr = s.qlrow + tl;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        if (R::LB == 16) fd_cp16(qg + g * 32 * R::QB, qr + 128 * g); else fd_cp8(qg + g * 32 * R::QB, qr + 128 * g);
      }
    }
    return;
  }
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int t0 = tl + 128 * g;
    unsigned char* ld = lg + g * 32 * R::LB;
    unsigned char* qd = qg + g * 32 * R::QB;
    if (vec) {
      if (t0 < V) {
        if (R::LB == 16) fd_cp16(ld, s.row + t0); else fd_cp8(ld, s.row + t0);
        if (s.mode == FD_DENSE) {
          fd_cp16(qd, s.qrow + t0);
        } else if (s.mode == FD_QL) {
          if (R::LB == 16) fd_cp16(qd, s.qlrow + t0); else fd_cp8(qd, s.qlrow + t0);
        }
      } else {
        const uint32_t pad = Tr<T>::kPadWord;
        if (R::LB == 16) *reinterpret_cast<uint4*>(ld) = make_uint4(pad, pad, pad, pad);
        else *reinterpret_cast<uint2*>(ld) = make_uint2(pad, pad);
        if (s.mode == FD_DENSE) {
          *reinterpret_cast<uint4*>(qd) = make_uint4(0u, 0u, 0u, 0u);
        } else if (s.mode == FD_QL) {
          if (R::LB == 16) *reinterpret_cast<uint4*>(qd) = make_uint4(pad, pad, pad, pad);
          else *reinterpret_cast<uint2*>(qd) = make_uint2(pad, pad);
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

// One chunk's 16 tokens of this lane (tokens past the row's end arrive as
// -inf logits with zero q).  The per-token formulas are those of run_tail /
// run_top, so token_mass reproduces each token's share.
template <typename T, int MODE, bool MASK>
__device__ __forceinline__ void fd_sweep(const FdSeq<T>& s, const unsigned char* st, int tc, float cc, float c_lo,
                                         const float* tab, FdAcc& acc) {
  using R = FdRing<T>;
  constexpr bool EXACT = sizeof(T) == 2;
  const int lane = threadIdx.x & 31;
  const unsigned char* lg = st;
  const unsigned char* qg = st + 4 * 32 * R::LB;
  const float M = s.M, s_a = s.s_a;
  uint32_t near = 0u;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int t0 = tc + 128 * g + 4 * lane;
    float x[4], q[4], p[4], w[4];
    fd_unpack<T>(lg + (g * 32 + lane) * R::LB, x);
    fd_qgroup<T, MODE>(s, qg + (g * 32 + lane) * R::QB, t0, cc, c_lo, q);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      // top-p alone: a token outside the kept set has p~ = 0 (weight 0, and
      // max(0 - q, 0) = 0)
      if (MASK && !tp_kept<T>(x[t], t0 + t, s.K, s.idx)) x[t] = -INFINITY;
      float e;
      if (EXACT) {
        const float dh = fmaxf(x[t] - M, -1.0e4f);   // exact for 16-bit logits; -inf flushes to 0 below
        p[t] = dh * cc;
        e = fmaf(dh, c_lo, fmaf(dh, cc, -p[t]));
      } else {
        p[t] = tok_exponent<false>(x[t], M, cc, c_lo, &e);
      }
      const float y = ex2_approx(p[t]);
      w[t] = fmaf(y * 6.931471825e-01f, e, y);
      if (!EXACT) w[t] = p[t] > -1.0e30f ? w[t] : 0.f;   // -inf (float32 logits)
    }
    // a token near the maximum (exponent above -8) is rare: it leaves the
    // float32 sums and is added in two-float after the sweep
    if (fmaxf(fmaxf(p[0], p[1]), fmaxf(p[2], p[3])) > -8.f) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (p[t] > -8.f) {
          w[t] = 0.f;
          near |= 1u << (4 * g + t);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      acc.S[t & 1] += w[t];
      if (MODE != FD_NONE) {
        // the residual support {w > s' q}: the sign of w - s' q rounded once
        const float d = fmaf(-s_a, q[t], w[t]);
        acc.A[t & 1] += fmaxf(d, 0.f);
        acc.Q[t & 1] += d > 0.f ? q[t] : 0.f;
      }
    }
  }
  while (near) {
    const int o = __ffs(near) - 1;
    near &= near - 1;
    const int g = o >> 2, t = o & 3;
    const int t0 = tc + 128 * g + 4 * lane;
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

// Shared memory the search stages in: C item sums (float4 + float each),
// then the 2048 token masses of the chosen item (64-bit fixed point).
__host__ __device__ constexpr size_t fd_stash_bytes(int C) {
  return (((size_t)C * 20 + 15) & ~(size_t)15) + (size_t)kFdTok * sizeof(long long);
}

struct FdSmem {
  float tab[128];            // exp2_f2 table
  F2 wsum[kFdWarps];         // shard totals: warp sums
  long long wll[kFdWarps];   // token phase: warp totals, then their exclusive prefixes
  int wcand[kFdWarps];       // token phase: each warp's candidate
  int item, use_q, resid0, e;   // item phase results (warp 0); e: the fixed-point scale
  long long ibase, target;   // the item's start and the target, in units of 2^-e
  F2 ds;
  int is_last;               // this CTA completed the sequence (ticket)
};

// Fixed point for the search: a non-negative two-float v as round(v * 2^e)
// (hi and lo rounded apart; callers keep v * 2^e below 2^62), and the scale
// e that puts a positive float R in [2^60, 2^61).  Prefix sums of such
// integers are exact: every start and every comparison with the target is
// exact, whatever the order of the additions.
// round(x 2^e) for a float x with |x 2^e| < 2^62, from its bits on the
// integer pipes: the 24-bit significand shifted by the exponent, rounded to
// nearest (ties away from zero) when bits fall off.
__device__ __forceinline__ long long fx_float(float x, int e) {
  const uint32_t u = __float_as_uint(x);
  const int be = (int)((u >> 23) & 0xffu);
  if (be == 0) return 0;                                   // zero (and subnormals: far below 2^-e)
  const long long m = (long long)((u & 0x7fffffu) | 0x800000u);
  const int sh = be - 150 + e;                             // x 2^e = m 2^sh
  long long r;
  if (sh >= 0) r = m << sh;
  else if (sh > -25) r = (m + (1ll << (-sh - 1))) >> -sh;
  else r = 0;
  return (u >> 31) ? -r : r;
}
__device__ __forceinline__ long long fx_of(F2 v, int e) { return fx_float(v.hi, e) + fx_float(v.lo, e); }
__device__ __forceinline__ int fx_scale(float R) {
  int ex;
  frexpf(R, &ex);   // R = f 2^ex, f in [0.5, 1)
  return 61 - ex;
}
__device__ __forceinline__ long long warp_incl_scan_ll(long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const long long o = __shfl_up_sync(0xffffffffu, v, m);
    if (lane >= m) v += o;
  }
  return v;
}
__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// The inverse-CDF search of sequence s (b), by the CTA that completed it.
//   1. Every thread: the C item sums from global memory into `stash` (the
//      drained ring), zeroing them behind.
//   2. Warp 0 alone: the exact normaliser s = sum S, the item masses m_k
//      (A_k - (s - s') Q_k for a residual, clamped at 0; S_k for the bonus
//      draw, or for the fallback to p_n when the residual has no mass), their
//      total R, the target t = u R and the item.  Lane l holds items
//      [l P, l P + P): its sum, one warp scan of the lane sums, then each lane
//      walks its own items.
//   3. Every thread: four of the item's 2048 tokens (re-read from L2), their
//      masses, a block scan of the thread sums, and the token.
// The sums, scans and comparisons run in 64-bit fixed point (fx_of, with
// the scale of R: each mass rounded to 2^-61 R), so the prefixes are exact
// and t = floor(R u) is an exact product.  At both levels the pick is the
// last entry of positive mass whose start is <= t, which is the smallest
// entry whose cumulative mass exceeds t (the inverse CDF); a target past the
// item's token sum takes its last positive token.  Four block barriers.
// `given` (vocabulary shards): s - s', the kind of mass and the target are
// fixed by all shards' totals; the search runs over this shard's items only.
struct FdGiven {
  int on, use_q;
  F2 ds, t;
};
template <typename T, bool MASK>
__device__ __forceinline__ int fd_pick_block(const Params& p, int b, const FdSeq<T>& s, FdSmem& sm,
                                             unsigned char* stash, int* resid0_out, FdGiven given = FdGiven{}) {
  constexpr bool EXACT = sizeof(T) == 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, C = p.FC;
  float4* sSA = reinterpret_cast<float4*>(stash);
  float* sQ = reinterpret_cast<float*>(stash + (size_t)C * sizeof(float4));
  float4* gSA = p.fd_part + (size_t)b * C;
  float* gQ = p.fd_q + (size_t)b * C;
  asm volatile("cp.async.wait_group 0;" ::: "memory");   // the ring is drained (its last groups are empty)
  for (int k = tid; k < C; k += kFdThreads) {
    sSA[k] = __ldcg(gSA + k);
    sQ[k] = __ldcg(gQ + k);
    gSA[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    gQ[k] = 0.f;
  }
  *resid0_out = 0;
  if (tid == 0) sm.item = -1;
  __syncthreads();
  if (s.mode == FD_SKIP) return 0;
  const bool resid = s.n < s.gb;
  // ---- 2. the item (warp 0)
  if (warp == 0) {
    const int P = (C + 31) / 32;
    const int k0 = min(C, lane * P), k1 = min(C, k0 + P);
    F2 ds;
    bool use_q;
    if (given.on) {
      ds = given.ds;
      use_q = given.use_q != 0;
    } else {
      // s exactly, at the scale of s' (every S_k <= s ~ s')
      const int es = fx_scale(s.s_a > 0.f ? s.s_a : 1.f);
      long long sl = 0;
      for (int k = k0; k < k1; ++k) sl += fx_of(F2{sSA[k].x, sSA[k].y}, es);
      sl = warp_sum_ll(sl);
      ds = F2{ldexpf((float)(sl - fx_float(s.s_a, es)), -es), 0.f};   // s - s', tiny
      use_q = resid;
    }
    int resid0 = 0;
    auto mass = [&](int k) -> F2 {
      const float4 v = sSA[k];
      if (!use_q) return F2{v.x, v.y};
      F2 m = f2_add(F2{v.z, v.w}, f2_neg(f2_scale(ds, sQ[k])));
      if (m.hi < 0.f) m = F2{0.f, 0.f};
      return m;
    };
    float Rf = 0.f;
    for (int attempt = 0; attempt < 2; ++attempt) {
      Rf = 0.f;
      for (int k = k0; k < k1; ++k) Rf += mass(k).hi;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) Rf += __shfl_xor_sync(0xffffffffu, Rf, o);
      if (!given.on && resid && use_q && !(Rf > 0.f)) {   // (warp-uniform) zero residual mass, only through rounding
        resid0 = 1;
        use_q = false;
        continue;
      }
      break;
    }
    int best = -1;
    long long bstart = 0, t = 0;
    const int e = fx_scale(Rf > 0.f ? Rf : 1.f);
    if (Rf > 0.f) {
      long long lt = 0;
      for (int k = k0; k < k1; ++k) lt += fx_of(mass(k), e);
      const long long inc = warp_incl_scan_ll(lt);
      const long long R = __shfl_sync(0xffffffffu, inc, 31);
      if (given.on) {
        t = fx_of(given.t, e);
        if (t < 0) t = 0;
      } else {
        // u 2^64 (u in [0, 1); a u of 2^-40 or less rounds to a multiple of 2^-64)
        const unsigned long long ufx = s.u > 0.f ? (unsigned long long)fx_float(s.u, 62) << 2 : 0ull;
        t = (long long)__umul64hi((unsigned long long)R, ufx);             // floor(R u)
      }
      long long st = inc - lt;
      for (int k = k0; k < k1; ++k) {
        const long long m = fx_of(mass(k), e);
        if (m > 0 && st <= t) {
          best = k;
          bstart = st;
        }
        st += m;
      }
    }
    const int top = __reduce_max_sync(0xffffffffu, best);
    if (best >= 0 && best == top) {   // one lane: the lanes' items are disjoint
      sm.item = best;
      sm.ibase = bstart;
    }
    if (lane == 0) {
      sm.use_q = use_q;
      sm.resid0 = resid0;
      sm.target = t;
      sm.e = e;
      sm.ds = ds;
    }
  }
  __syncthreads();
  const int item = sm.item;
  if (item < 0) return 0;   // no positive mass (rounding)
  *resid0_out = sm.resid0;
  const bool use_q = sm.use_q != 0;
  const F2 ds = sm.ds;
  const int e = sm.e;
  // ---- 3. the token: thread t has the TPT consecutive tokens at item * kFdTok + TPT t.
  // Their logits and q are loaded first (one round trip: a vector load each
  // when the row allows), then the masses, kept in shared memory after the
  // item sums across the scan.
  constexpr int TPT = kFdTok / kFdThreads;
  static_assert(TPT == 4, "four tokens per thread: one 4-token group");
  const int mode = use_q ? s.mode : FD_NONE;
  const int v0 = item * kFdTok + TPT * tid;
  const bool full = ((V & 3) == 0) && v0 + TPT <= V;
  float x[TPT], qv[TPT];
  if (full) {
    if (sizeof(T) == 4) {
      const float4 w = __ldcg(reinterpret_cast<const float4*>(s.row + v0));
      fd_unpack<T>(reinterpret_cast<const unsigned char*>(&w), x);
    } else {
      const uint2 w = __ldcg(reinterpret_cast<const uint2*>(s.row + v0));
      fd_unpack<T>(reinterpret_cast<const unsigned char*>(&w), x);
    }
  } else {
#pragma unroll
    for (int j = 0; j < TPT; ++j)
      x[j] = v0 + j < V ? Tr<T>::get(load_slot<T>(s.row, v0 + j, 1, false), 0) : -INFINITY;
  }
#pragma unroll
  for (int j = 0; j < TPT; ++j) qv[j] = 0.f;
  if (mode == FD_DENSE) {
    if (full) {
      const float4 w = __ldcg(reinterpret_cast<const float4*>(s.qrow + v0));
      qv[0] = w.x; qv[1] = w.y; qv[2] = w.z; qv[3] = w.w;
    } else {
#pragma unroll
      for (int j = 0; j < TPT; ++j) qv[j] = v0 + j < V ? __ldcg(s.qrow + v0 + j) : 0.f;
    }
  } else if (mode == FD_QL) {
    float y[TPT];
    if (full) {
      if (sizeof(T) == 4) {
        const float4 w = __ldcg(reinterpret_cast<const float4*>(s.qlrow + v0));
        fd_unpack<T>(reinterpret_cast<const unsigned char*>(&w), y);
      } else {
        const uint2 w = __ldcg(reinterpret_cast<const uint2*>(s.qlrow + v0));
        fd_unpack<T>(reinterpret_cast<const unsigned char*>(&w), y);
      }
    } else {
#pragma unroll
      for (int j = 0; j < TPT; ++j)
        y[j] = v0 + j < V ? Tr<T>::get(load_slot<T>(s.qlrow, v0 + j, 1, false), 0) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < TPT; ++j) qv[j] = s.qlr.q(y[j], p.c, p.c_lo);
  } else if (mode == FD_DET) {
#pragma unroll
    for (int j = 0; j < TPT; ++j) qv[j] = v0 + j == s.xq ? INFINITY : 0.f;
  }
  long long* tmS = reinterpret_cast<long long*>(stash + fd_stash_bytes(C) - (size_t)kFdTok * sizeof(long long));
  long long m = 0;
#pragma unroll
  for (int j = 0; j < TPT; ++j) {
    const int v = v0 + j;
    long long tj = 0;
    if (v < V && (!MASK || tp_kept<T>(x[j], v, s.K, s.idx)))
      tj = fx_of(token_mass<EXACT>(x[j], qv[j], use_q, s.M, p.c, p.c_lo, s.s_a, ds, sm.tab), e);
    tmS[j * kFdThreads + tid] = tj;
    m += tj;
  }
  // block exclusive scan of the thread sums: warp scans, warp 0 scans the warp totals
  const long long inc = warp_incl_scan_ll(m);
  if (lane == 31) sm.wll[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const long long w = warp_incl_scan_ll(lane < kFdWarps ? sm.wll[lane] : 0ll);
    __syncwarp();
    if (lane < kFdWarps) sm.wll[lane] = w - sm.wll[lane];
  }
  __syncthreads();
  long long st = sm.ibase + sm.wll[warp] + (inc - m);   // this thread's first token's start
  const long long t = sm.target;
  int cand = -1;
#pragma unroll
  for (int j = 0; j < TPT; ++j) {
    const long long tj = tmS[j * kFdThreads + tid];
    if (tj > 0 && st <= t) cand = v0 + j;
    st += tj;
  }
  cand = __reduce_max_sync(0xffffffffu, cand);
  if (lane == 0) sm.wcand[warp] = cand;
  __syncthreads();
  int tok = -1;
#pragma unroll
  for (int w = 0; w < kFdWarps; ++w) tok = max(tok, sm.wcand[w]);
  return tok >= 0 ? tok : 0;
}

// One vocabulary shard's totals of sequence b's row-n items: sum S and sum A
// (two-float) and sum Q, written as 8 floats (S.hi, S.lo, A.hi, A.lo, Q, 0,
// 0, 0) to sh_out[b].  Items in thread order, warps in order: the same
// additions on every call.
__device__ __forceinline__ void fd_shard_totals(const Params& p, int b, FdSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = p.FC;
  F2 S{0.f, 0.f}, A{0.f, 0.f}, Q{0.f, 0.f};
  for (int k = tid; k < C; k += kFdThreads) {
    const float4 v = __ldcg(p.fd_part + (size_t)b * C + k);
    S = f2_add(S, F2{v.x, v.y});
    A = f2_add(A, F2{v.z, v.w});
    Q = f2_add(Q, F2{__ldcg(p.fd_q + (size_t)b * C + k), 0.f});
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    S = f2_add(S, f2_shfl_xor(S, o));
    A = f2_add(A, f2_shfl_xor(A, o));
    Q = f2_add(Q, f2_shfl_xor(Q, o));
  }
  // three two-float totals per warp through wsum (16 entries): S, then A and Q
  if (lane == 0) sm.wsum[warp] = S;
  __syncthreads();
  F2 tS{0.f, 0.f};
  if (tid == 0)
    for (int w = 0; w < kFdWarps; ++w) tS = f2_add(tS, sm.wsum[w]);
  __syncthreads();
  if (lane == 0) sm.wsum[warp] = A;
  __syncthreads();
  F2 tA{0.f, 0.f};
  if (tid == 0)
    for (int w = 0; w < kFdWarps; ++w) tA = f2_add(tA, sm.wsum[w]);
  __syncthreads();
  if (lane == 0) sm.wsum[warp] = Q;
  __syncthreads();
  if (tid == 0) {
    F2 tQ{0.f, 0.f};
    for (int w = 0; w < kFdWarps; ++w) tQ = f2_add(tQ, sm.wsum[w]);
    float* o = static_cast<float*>(p.sh_out) + (size_t)b * 8;
    *reinterpret_cast<float4*>(o) = make_float4(tS.hi, tS.lo, tA.hi, tA.lo);
    *reinterpret_cast<float4*>(o + 4) = make_float4(tQ.hi + tQ.lo, 0.f, 0.f, 0.f);
  }
}

// MASK: top-p alone (the rows' records come from topp_row_kernel).
// Work unit u = (sequence b = u / Z, part z = u % Z): part z sums items
// [z C / Z, (z + 1) C / Z) of row n; the CTA that completes a sequence's last
// part (an acquire-release ticket) runs its search.  Z = p.FZ parts per
// sequence, so that B * Z units fill the GPU's SMs once.
template <typename T, bool MASK>
__global__ void __launch_bounds__(kFdThreads, 1) final_draw_kernel(const Params p) {
  using R = FdRing<T>;
  constexpr int S = R::S;
  extern __shared__ __align__(16) unsigned char fd_dyn[];
  __shared__ FdSmem sm;
  load_exp2_table(sm.tab);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = fd_dyn + (size_t)warp * S * R::stage_bytes;
  const int G = p.gamma, G1 = G + 1, V = p.V, C = p.FC, Z = p.FZ;
  const int U = p.B * Z;
  const bool vec = (V & 3) == 0;
  const bool scan = !MASK && p.H > 0;   // streaming path: the row partials are merged here
  // the first unit's acceptance inputs, before the dependency wait
  FdDrafts dr;
  int dr_b = -1;
  if (scan && (int)blockIdx.x < U) {
    dr_b = blockIdx.x / Z;
    fd_gather<T>(p, dr_b, dr);
  }
  pdl_wait();   // the row statistics come from the previous kernel
  __syncthreads();
  for (int u = blockIdx.x; u < U; u += gridDim.x) {
    const int b = u / Z, z = u - b * Z;
    const int k0 = (int)((long long)z * C / Z), k1 = (int)((long long)(z + 1) * C / Z);
    // every warp: sequence b's state (part 0's warp 0 writes the outputs but the token)
    FdSeq<T> s;
    const bool writer = z == 0 && warp == 0;
    if (MASK) {
      fd_scan_tp<T>(p, b, writer, s);
    } else if (scan) {
      if (b != dr_b) {
        fd_gather<T>(p, b, dr);
        dr_b = b;
      }
      fd_scan<T>(p, b, dr, writer, s);
    } else {
      fd_load_state<T>(p, b, s);
    }
    // ---- warp w sums items k0 + w, k0 + w + 16, ... of the part, chunk by
    // chunk through its ring (the issuer S chunks ahead of the consumer)
    int ki = k0 + warp, kj = 0, stage = 0;
    auto issue_next = [&](unsigned char* dst) {
      if (ki < k1) {
        fd_issue(s, ki * kFdTok + kj * kFdChunk, V, vec, dst);
        if (++kj == kFdChunks) {
          kj = 0;
          ki += kFdWarps;
        }
      }
      fd_commit();
    };
#pragma unroll 1
    for (int st = 0; st < S; ++st) issue_next(ring + st * R::stage_bytes);
    for (int kb = k0 + warp; kb < k1; kb += 4 * kFdWarps) {
      const int nb = min(4, (k1 - kb + kFdWarps - 1) / kFdWarps);
      IT5 slot[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) slot[j] = IT5{};
#pragma unroll 1
      for (int j = 0; j < nb; ++j) {
        const int c = kb + j * kFdWarps;
        // the item's lane sums: the float32 sums of each chunk folded into two-float
        F2 iS{0.f, 0.f}, iA{0.f, 0.f};
        float iQ = 0.f;
        RunAcc top;
        top.zero();
#pragma unroll 1
        for (int h = 0; h < kFdChunks; ++h) {
          fd_wait_ring<S>();
          unsigned char* stp = ring + stage * R::stage_bytes;
          FdAcc acc;
          acc.S[0] = acc.S[1] = acc.A[0] = acc.A[1] = acc.Q[0] = acc.Q[1] = 0.f;
          acc.top = top;
          const int tc = c * kFdTok + h * kFdChunk;
          switch (s.mode) {
            case FD_NONE: fd_sweep<T, FD_NONE, MASK>(s, stp, tc, p.c, p.c_lo, sm.tab, acc); break;
            case FD_DENSE: fd_sweep<T, FD_DENSE, MASK>(s, stp, tc, p.c, p.c_lo, sm.tab, acc); break;
            case FD_DET: fd_sweep<T, FD_DET, MASK>(s, stp, tc, p.c, p.c_lo, sm.tab, acc); break;
            case FD_QL: fd_sweep<T, FD_QL, MASK>(s, stp, tc, p.c, p.c_lo, sm.tab, acc); break;
            default: break;   // a bad row: nothing was read
          }
          // this stage has been read: refill it S chunks ahead
          issue_next(stp);
          stage = stage + 1 == S ? 0 : stage + 1;
          top = acc.top;
          iS = f2_add(iS, F2{acc.S[0] + acc.S[1], 0.f});
          iA = f2_add(iA, F2{acc.A[0] + acc.A[1], 0.f});
          iQ += acc.Q[0] + acc.Q[1];
        }
        slot[3] = slot[2];
        slot[2] = slot[1];
        slot[1] = slot[0];
        slot[0] = IT5::of(f2_add(iS, top.S()), f2_add(iA, top.A()), iQ + top.q);
      }
      // slot j holds item kb + (nb - 1 - j) * 16; every lane of group
      // g = lane / 8 then holds slot g's warp total
      const IT5 tot = it5_reduce4(slot);
      const int g = lane >> 3;
      if ((lane & 7) == 0 && g < nb) {
        const int c = kb + (nb - 1 - g) * kFdWarps;
        p.fd_part[(size_t)b * C + c] = make_float4(tot.S.hi, tot.S.lo, tot.A.hi, tot.A.lo);
        p.fd_q[(size_t)b * C + c] = tot.Q;
      }
    }
    // ---- the part is summed: the last part of the sequence searches
    __syncthreads();
    if (tid == 0) {
      // release: this part's item sums; acquire: the other parts' (last arrival)
      const int prev = Z > 1 ? atomic_add_acq_rel_gpu(p.seq_ticket2 + b, 1) : Z - 1;
      sm.is_last = prev == Z - 1;
    }
    __syncthreads();
    if (sm.is_last && p.shard == 1) {
      // vocabulary shard: this shard's row-n totals; the items stay for the search
      fd_shard_totals(p, b, sm);
      if (tid == 0) p.seq_ticket2[b] = 0;
    } else if (sm.is_last) {
      int resid0 = 0;
      const int token = fd_pick_block<T, MASK>(p, b, s, sm, fd_dyn, &resid0);
      // the output; the row partials, the row records, the ticket and the
      // state zeroed behind it (the item sums were zeroed as they were read)
      if (scan) {
        const int E = G1 * stream_np(p);
        for (int e = tid; e < E; e += kFdThreads) p.part[(size_t)b * E + e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.ql) {
          const int Eq = G * stream_np(p);
          for (int e = tid; e < Eq; e += kFdThreads) p.qpart[(size_t)b * Eq + e] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (MASK) {
        for (int e = tid; e < G1 * (int)(sizeof(TpRow) / 4); e += kFdThreads)
          reinterpret_cast<int*>(p.tp + (size_t)b * G1)[e] = 0;
      }
      if (tid == 0) {
        p.out_tokens[b * G1 + s.n] = token;
        if (p.out_status) p.out_status[b] = s.status | (resid0 ? SEQ_RESID0 : 0);
        p.seq_ticket2[b] = 0;
        if (!scan && !MASK) {   // the rows kernel's state
          SeqState zs;
          zs.n = 0; zs.status = 0; zs.M = 0.f; zs.qm = 0.f; zs.s = 0.0; zs.qinv = 0.f; zs.qbad = 0; zs.tpK = 0u; zs.tpIdx = 0;
          p.seq[b] = zs;
        }
      }
    }
    __syncthreads();   // shared state reused by the next unit
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

}  // namespace sv
