// Streaming path of libspecverify for large batches: persistent CTAs, one
// row (or row part) at a time, each thread prefetching its own future 16-byte
// vectors with cp.async into a thread-private shared-memory ring S stages deep.
//
// Why this shape.  Every mode is bound by HBM bandwidth, which needs ~50 KB
// of reads in flight per SM at all times.  A CTA that loads, then reduces,
// then hands off, leaves HBM idle during the last two; here a thread's ring
// already holds (or is fetching) the next S chunks of its row sequence -
// including the first chunks of its NEXT row - while the current row is being
// finished.  The ring is private to the thread that filled it (the thread
// copies and later reads its own slots), so completion is tracked per thread
// with cp.async.wait_group: there are no cross-thread waits, no mbarriers and
// no spin loops.  The dense kernel gives every CTA the same number of
// vectors (the rows laid end to end and cut into equal ranges, so a row may
// be split between consecutive CTAs); the top-k kernel claims whole rows from
// a counter as its CTAs get through them.  With q formed from the draft's
// logits, the draft rows follow the target rows through both kernels.
//
//   greedy   argmax of each row segment (ties -> lowest index; NaN
//            flagged); stream_greedy_finish_kernel merges the segments,
//            scans the drafts and emits the tokens
//   softmax  online max / sum of 2^((L - m) c) with rescaling when the
//            running max grows; final_draw_kernel merges the segments,
//            computes p(d_i) and a_i, scans, sums the final draw's items and
//            locates the drawn token (sv_final.cuh)
//   top-k    pass 1 keeps per-thread maxima (and the two best vectors); the
//            k-th largest is a lower bound tau of the row's k-th value; only
//            threads with a third vector reaching tau are re-read (L2);
//            exact rank selection of the candidates >= tau; softmax(./T) +
//            top-p; a_i (with q from draft logits, in the finisher, from the
//            two rows' kept lists).  The last row of a sequence to finish
//            (atomic ticket, no waiting) runs the acceptance scan and the
//            final draw.
//
// The dense kernel ends a row segment with warp shuffles and one block
// barrier (a CTA ends at most H + 1 segments); chunks in between take none.
#pragma once

#include "sv_device.cuh"
#include "sv_topk.cuh"

namespace sv {

constexpr int kSt = 256;      // threads per CTA
constexpr int kStU = 4;       // vectors per thread per ring stage
constexpr int kStS = 4;       // ring stages (dense modes)
constexpr int kStSTopk = 3;   // ring stages (top-k; leaves room for its selection buffers)
constexpr int kStUTopk = 4;   // vectors per thread per ring stage (top-k)
static_assert(kSt == kThreads, "the block reductions assume kThreads threads");

__device__ __forceinline__ void cpa16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cpa_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The dense streaming kernel's block-wide state: the warps' partials at the
// end of a segment, double-buffered by segment parity (so that one barrier
// per segment suffices: warp 0 has read buffer k before it reaches segment
// k + 1's barrier, after which buffer k is written again at segment k + 2).
struct StreamSmem {
  float4 red[2][kWarps];
};

// Per-thread sequence of ring items: (j-th row of this CTA, pass, chunk c),
// PASSES passes over each row.  The issuer walks it S items ahead of the
// consumer with running counters (no divisions); each item copies this
// thread's U vectors of one chunk (U * kSt vectors) of a row.
struct RowWalk {
  int R, G1, NV, CH, NCH, nrows;
  int H = 1, NVP = 0;   // parts per row and vectors per part (NVP = NV when H = 1)
  // rows claimed at run time (H = 1): the CTA's j-th row is dyn[j & 3], and
  // the walk ends at the first claim >= R; otherwise rows are dealt statically
  const int* dyn = nullptr;
  // rows from Rt on are the draft's logits (q formed from them), row r - Rt of ql
  int Rt = 0x7fffffff;
  const void* ql = nullptr;
  __device__ __forceinline__ int row_of(int j) const { return dyn ? dyn[j & 3] : blockIdx.x + j * gridDim.x; }
  __device__ __forceinline__ bool live(int j) const { return dyn ? dyn[j & 3] < R : j < nrows; }
  // item j of this CTA: row r, vectors [vb, ve)
  __device__ __forceinline__ void item(int j, int* r, int* vb, int* ve) const {
    const int g = row_of(j);
    const int h = g % H;
    *r = g / H;
    *vb = h * NVP;
    *ve = min(*vb + NVP, NV);
  }
};

template <typename T, int S, int PASSES, int U = kStU>
struct Issuer {
  int j = 0, pass = 0, c = 0, stage = 0, vb = 0, ve = 0;
  const T* row = nullptr;
  __device__ __forceinline__ void at(const T* logits, size_t V, const RowWalk& w) {
    int r;
    w.item(j, &r, &vb, &ve);
    r = min(r, w.R - 1);
    row = r >= w.Rt ? static_cast<const T*>(w.ql) + (size_t)(r - w.Rt) * V : logits + (size_t)r * V;
  }
  __device__ __forceinline__ void start(const T* logits, size_t V, const RowWalk& w) { at(logits, V, w); }
  // issue the next item into its stage (an empty group past the end)
  __device__ __forceinline__ void issue(uint4* ring, const T* logits, size_t V, const RowWalk& w) {
    if (w.live(j)) {
      uint4* slot = ring + (size_t)stage * U * kSt + threadIdx.x;
      const int v0 = vb + c * w.CH + (int)threadIdx.x;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kSt;
        if (v < ve) cpa16(slot + u * kSt, row + (size_t)v * Tr<T>::VW);
      }
      if (++c == w.NCH) {
        c = 0;
        if (++pass == PASSES) {
          pass = 0;
          ++j;
          if (w.live(j)) at(logits, V, w);
        }
      }
    }
    cpa_commit();   // empty groups keep every thread's group count in step
    stage = (stage + 1 == S) ? 0 : stage + 1;
  }
};

// ---- greedy finish: one CTA per sequence after the streaming kernel
// Merges each row's per-warp (max, first index) partials into the target's
// argmax g_i, accepts drafts while d_i == g_i (stopping at the first
// mismatch n), emits d_0..d_{n-1}, g_n and -1 padding, and zeroes the
// partial slots it read.
__global__ void __launch_bounds__(kSt) stream_greedy_finish_kernel(const Params p) {
  __shared__ int sg[kMaxG1], sbad[kMaxG1], smis[kMaxG1];
  __shared__ int s_status, s_n;
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  const int G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);
  const int d = tid < gb ? __ldg(p.draft + b * G + tid) : -1;   // an input: before the wait
  pdl_wait();
  merge_row_parts<MODE_GREEDY>(p, b, G1, gb, nullptr, nullptr, sg, sbad);
  if (tid == 0) s_status = 0;
  __syncthreads();
  if (tid < gb) {
    const bool oob = d < 0 || d >= V;
    if (oob) atomicOr(&s_status, SEQ_OOB);
    smis[tid] = oob || d != sg[tid];
  }
  __syncthreads();
  if (tid < 32) {
    bool anybad = false;
    const int n0 = first_flag_w0(smis, gb, sbad, gb, &anybad);
    if (tid == 0) {
      s_n = n0;
      if (anybad) s_status |= SEQ_BADROW;
    }
  }
  __syncthreads();
  const int n = s_n;
  if (tid < G1) p.out_tokens[b * G1 + tid] = tid < n ? d : (tid == n ? sg[n] : -1);
  if (tid == 0) {
    p.out_n[b] = n;
    if (p.out_status) p.out_status[b] = s_status;
  }
  const int E = G1 * stream_np(p);
  for (int e = tid; e < E; e += kSt) p.part[(size_t)b * E + e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Maximum of the kStU vectors x (NaN-free: the softmax path treats NaN rows
// through the merged statistics), 16-bit types reduced as packed pairs.
template <typename T>
__device__ __forceinline__ float chunk_max(const uint4 (&x)[kStU]) {
  using TR = Tr<T>;
  if constexpr (TR::VW == 8) {
    using H2 = typename std::conditional<std::is_same<T, __half>::value, __half2, __nv_bfloat162>::type;
    H2 acc = *reinterpret_cast<const H2*>(&x[0].x);
#pragma unroll
    for (int u = 0; u < kStU; ++u) {
      const H2 a = *reinterpret_cast<const H2*>(&x[u].x), b = *reinterpret_cast<const H2*>(&x[u].y);
      const H2 c = *reinterpret_cast<const H2*>(&x[u].z), d = *reinterpret_cast<const H2*>(&x[u].w);
      acc = __hmax2(acc, __hmax2(__hmax2(a, b), __hmax2(c, d)));
    }
    return fmaxf(__low2float(acc), __high2float(acc));
  } else {
    float m = TR::template vmax<false>(x[0]);
#pragma unroll
    for (int u = 1; u < kStU; ++u) m = fmaxf(m, TR::template vmax<false>(x[u]));
    return m;
  }
}

// Greedy helpers over one ring stage (this thread's kStU vectors, element
// index (c0 + u*kSt + tid)*VW + t).  stage_max: the maximum, NaN if any element
// is NaN, -inf if the stage holds no real vector.  16-bit types reduce packed
// pairs first and convert once.
template <typename T, bool FULL>
__device__ __forceinline__ float stage_max(const uint4* slot, int c0, int NV) {
  using TR = Tr<T>;
  const int tid = threadIdx.x;
  if constexpr (TR::VW == 8) {
    using H2 = typename std::conditional<std::is_same<T, __half>::value, __half2, __nv_bfloat162>::type;
    uint32_t padw = TR::kPadWord;
    H2 acc = *reinterpret_cast<const H2*>(&padw);
#pragma unroll
    for (int u = 0; u < kStU; ++u) {
      if (FULL || c0 + u * kSt + tid < NV) {
        const uint4 x = slot[u * kSt + tid];
        const H2 a = *reinterpret_cast<const H2*>(&x.x), b = *reinterpret_cast<const H2*>(&x.y);
        const H2 cc = *reinterpret_cast<const H2*>(&x.z), d = *reinterpret_cast<const H2*>(&x.w);
        acc = __hmax2_nan(acc, __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(cc, d)));
      }
    }
    const float lo = __low2float(acc), hi = __high2float(acc);
    if (lo != lo || hi != hi) return __uint_as_float(0x7fffffffu);
    return fmaxf(lo, hi);
  } else {
    float m = -INFINITY;
    bool nan = false;
#pragma unroll
    for (int u = 0; u < kStU; ++u) {
      if (FULL || c0 + u * kSt + tid < NV) {
        const float vm = TR::template vmax<true>(slot[u * kSt + tid]);
        nan |= (vm != vm);
        m = fmaxf(m, vm);
      }
    }
    return nan ? __uint_as_float(0x7fffffffu) : m;
  }
}
// lowest element index of the stage holding the value m (m is not NaN)
template <typename T>
__device__ __noinline__ int stage_first_index(const uint4* slot, int c0, int NV, float m) {
  using TR = Tr<T>;
  const int tid = threadIdx.x;
  for (int u = 0; u < kStU; ++u) {
    const int v = c0 + u * kSt + tid;
    if (v < NV) {
      const uint4 x = slot[u * kSt + tid];
      for (int t = 0; t < TR::VW; ++t)
        if (TR::get(x, t) == m) return v * TR::VW + t;
    }
  }
  return 0x7fffffff;
}

// ---- greedy / softmax streaming kernel
//
// Every CTA streams the same number of 16-byte vectors: CTA j takes the range
// [start(j), start(j + 1)) of the flattened [rows][vectors] space, start(j) =
// floor(j * NVT / grid), whatever the row boundaries.  A row is thus split
// into at most H segments (consecutive CTAs), and each segment leaves one
// partial in slot row * H + segment, segment = j - seg_cta(row * NV) (its
// warps' partials combined by warp 0 after one block barrier; a CTA ends at
// most H + 1 segments).  Chunks of the ring never cross a row boundary.
//
// A walk over this CTA's range [v0, v1) of the flattened rows in chunks of
// at most CH vectors that end at a row boundary or the range's end: row r,
// vectors [v, ve) of it.  32-bit arithmetic inside a row.
struct SegWalk {
  int r, v, ve;         // current chunk: row r, vectors [v, min(v + CH, ve))
  int r1, e1;           // last row of the range and the range's end in it
  int NV, CH;
  __device__ __forceinline__ void init(long long v0, long long v1, int NV_, int CH_) {
    NV = NV_;
    CH = CH_;
    r = (int)(v0 / NV_);
    v = (int)(v0 - (long long)r * NV_);
    r1 = (int)((v1 - 1) / NV_);
    e1 = (int)(v1 - (long long)r1 * NV_);
    ve = r == r1 ? e1 : NV_;
    if (v0 >= v1) r = r1 + 1;   // an empty range
  }
  __device__ __forceinline__ bool live() const { return r <= r1; }
  // the current chunk (row, [vb, ce)); then advance
  __device__ __forceinline__ void take(int* row, int* vb, int* ce) {
    *row = r;
    *vb = v;
    *ce = min(v + CH, ve);
    v = *ce;
    if (v >= ve) {
      ++r;
      v = 0;
      ve = r == r1 ? e1 : NV;
    }
  }
};

template <typename T, int MODE>
__global__ void __launch_bounds__(kSt, 3)
stream_dense_kernel(const Params p) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  constexpr int S = kStS;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* ring = reinterpret_cast<uint4*>(smem_raw);
  StreamSmem& sred = *reinterpret_cast<StreamSmem*>(smem_raw + (size_t)S * kStU * kSt * sizeof(uint4));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G1 = p.gamma + 1, V = p.V;
  // the kernel that merges the partials may start its input-only prologue now
  pdl_launch_dependents();
  const int NV = V / VW;
  int par = 0;   // segment parity: the red buffer in use
  const int Rt = p.B * G1;          // target rows; draft rows (q formed from their logits) follow
  const T* logits = static_cast<const T*>(p.logits);
  const T* ql = static_cast<const T*>(p.ql);
  const long long NVT = p.NVT;
  const long long v0 = (long long)blockIdx.x * NVT / gridDim.x;
  const long long v1 = (long long)(blockIdx.x + 1) * NVT / gridDim.x;
  const int CH = kStU * kSt;
  auto rowptr = [&](int r) -> const T* {
    return r < Rt ? logits + (size_t)r * V : ql + (size_t)(r - Rt) * V;
  };
  // issuer: S chunks ahead of the consumer
  SegWalk iw;
  iw.init(v0, v1, NV, CH);
  int istage = 0;
  auto issue = [&]() {
    int r, vb, ve;
    if (iw.live()) {
      iw.take(&r, &vb, &ve);
      uint4* slot = ring + (size_t)istage * kStU * kSt + tid;
      const T* row = rowptr(r);
#pragma unroll
      for (int u = 0; u < kStU; ++u) {
        const int v = vb + u * kSt + tid;
        if (v < ve) cpa16(slot + u * kSt, row + (size_t)v * VW);
      }
    }
    cpa_commit();   // empty groups keep every thread's group count in step
    istage = istage + 1 == S ? 0 : istage + 1;
  };
#pragma unroll
  for (int s2 = 0; s2 < S; ++s2) issue();
  SegWalk cw;
  cw.init(v0, v1, NV, CH);
  int stage = 0;
  float best = -INFINITY;          // greedy: this thread's max, its first index, NaN seen
  int best_i = 0x7fffffff, nan_seen = 0;
  float m = -INFINITY, s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;   // softmax: running max and sums
  int r, vb, ve;
  while (cw.live()) {
    cw.take(&r, &vb, &ve);
    cpa_wait<S - 1>();
    const uint4* slot = ring + (size_t)stage * kStU * kSt;
    const bool fullc = ve - vb == CH;   // every thread has all kStU vectors of the chunk
    if (MODE == MODE_GREEDY) {
      // one max over the chunk's vectors of this thread; only a new best looks further
      const float cm = fullc ? stage_max<T, true>(slot, vb, ve) : stage_max<T, false>(slot, vb, ve);
      nan_seen |= (cm != cm);
      if (cm > best) {
        best = cm;
        best_i = stage_first_index<T>(slot, vb, ve, cm);
      }
    } else if (fullc) {
      // one maximum and at most one rescale per chunk, then the chunk's
      // elements into four independent sums
      uint4 x[kStU];
#pragma unroll
      for (int u = 0; u < kStU; ++u) x[u] = slot[u * kSt + tid];
      const float cm = chunk_max<T>(x);
      if (cm > m) {
        const float sc = (m == -INFINITY) ? 0.f : ex2_approx((m - cm) * p.c);
        s0 *= sc;
        s1 *= sc;
        s2 *= sc;
        s3 *= sc;
        m = cm;
      }
      if (m > -INFINITY) {
        const float mc = m * p.c;
#pragma unroll
        for (int u = 0; u < kStU; ++u) {
#pragma unroll
          for (int t = 0; t < VW; t += 4) {
            s0 += ex2_approx(fmaf(TR::get(x[u], t), p.c, -mc));
            s1 += ex2_approx(fmaf(TR::get(x[u], t + 1), p.c, -mc));
            s2 += ex2_approx(fmaf(TR::get(x[u], t + 2), p.c, -mc));
            s3 += ex2_approx(fmaf(TR::get(x[u], t + 3), p.c, -mc));
          }
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < kStU; ++u) {
        const int v = vb + u * kSt + tid;
        if (v < ve) {
          const uint4 x = slot[u * kSt + tid];
          const float vm = TR::template vmax<false>(x);
          if (vm > m) {
            const float sc = (m == -INFINITY) ? 0.f : ex2_approx((m - vm) * p.c);
            s0 *= sc;
            s1 *= sc;
            s2 *= sc;
            s3 *= sc;
            m = vm;
          }
          if (m > -INFINITY) {
            // four independent sums: short dependency chains
            const float mc = m * p.c;
#pragma unroll
            for (int t = 0; t < VW; t += 4) {
              s0 += ex2_approx(fmaf(TR::get(x, t), p.c, -mc));
              s1 += ex2_approx(fmaf(TR::get(x, t + 1), p.c, -mc));
              s2 += ex2_approx(fmaf(TR::get(x, t + 2), p.c, -mc));
              s3 += ex2_approx(fmaf(TR::get(x, t + 3), p.c, -mc));
            }
          }
        }
      }
    }
    issue();
    stage = stage + 1 == S ? 0 : stage + 1;
    if (ve == NV || !cw.live()) {
      // ---- the end of this CTA's segment of row r (the same chunk in every
      // thread): warp partials by shuffles, then warp 0 combines the 8 and
      // stores the segment's partial
      const int seg = (int)blockIdx.x - seg_cta((long long)r * NV, NVT, gridDim.x);
      float4* out = r < Rt ? p.part + (size_t)r * p.H + seg : p.qpart + (size_t)(r - Rt) * p.H + seg;
      if (MODE == MODE_GREEDY) {
        int bi = best_i;
        float bv = best;
        if (__any_sync(0xffffffffu, nan_seen)) bv = __int_as_float(0x7fffffff);   // a NaN flags the row
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) sred.red[par][warp] = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
        __syncthreads();
        if (warp == 0) {
          const float4 v = lane < kWarps ? sred.red[par][lane] : make_float4(-INFINITY, __int_as_float(0x7fffffff), 0.f, 0.f);
          bv = v.x;
          bi = __float_as_int(v.y);
#pragma unroll
          for (int o = kWarps >> 1; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
          }
          if (lane == 0) *out = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
        }
        best = -INFINITY;
        best_i = 0x7fffffff;
        nan_seen = 0;
      } else {
        float M = m;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        F2 acc{0.f, 0.f};
        if (m > -INFINITY && M < INFINITY) {
          const float sc = ex2_approx((m - M) * p.c);
          acc = f2_add(f2_add(F2{s0 * sc, 0.f}, F2{s1 * sc, 0.f}), f2_add(F2{s2 * sc, 0.f}, F2{s3 * sc, 0.f}));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc = f2_add(acc, f2_shfl_xor(acc, o));
        if (lane == 0) sred.red[par][warp] = make_float4(M, acc.hi, acc.lo, 0.f);
        __syncthreads();
        if (warp == 0) {
          const float4 v = lane < kWarps ? sred.red[par][lane] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
          float Mb = v.x;
#pragma unroll
          for (int o = kWarps >> 1; o >= 1; o >>= 1) Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, o));
          F2 t{0.f, 0.f};
          if (v.x > -INFINITY && Mb < INFINITY) {
            const float sc = ex2_approx((v.x - Mb) * p.c);
            t = f2_add(F2{v.y * sc, 0.f}, F2{v.z * sc, 0.f});
          }
#pragma unroll
          for (int o = kWarps >> 1; o >= 1; o >>= 1) t = f2_add(t, f2_shfl_xor(t, o));
          if (lane == 0) *out = make_float4(Mb, t.hi, t.lo, 0.f);
        }
        m = -INFINITY;
        s0 = s1 = s2 = s3 = 0.f;
      }
      par ^= 1;
    }
  }
  cpa_wait<0>();
}

// ---- top-k streaming kernel
//
// Pass 1 (the ring) keeps each thread's two best 16-byte vectors (maxima m1 >=
// m2) and m3, the largest maximum of its other vectors.  tau = the k-th
// largest thread maximum is a lower bound of the row's k-th largest value.
// Only threads with m1 >= tau hold elements >= tau; if m3 < tau they are all
// in the two kept vectors.  The rare threads with m3 >= tau too are re-read
// (pass 2, an L2 hit, spread over the whole CTA).  The candidates (all elements >=
// tau) are ranked exactly by (value desc, index asc).
// The largest K (bits below LOW zero) such that at least k of the block's
// 256 keys (one per thread; 0 = no key) are >= K: the k-th largest key with
// its bits below LOW cleared, 0 if fewer than k keys are positive.  Radix
// select from the top digit down: a shared-memory histogram of the digit
// among the keys that match the digits found so far, then warp 0 finds the
// digit holding the k-th largest by a scan from the top.
template <int LOW>
__device__ __forceinline__ uint32_t kth_largest_key(uint32_t key, int k, TopkSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t prefix = 0u;
  int rank = k;   // rank sought among the keys matching prefix
#pragma unroll
  for (int hi = 31; hi >= LOW; hi -= 8) {
    const int lo = hi - 7 > LOW ? hi - 7 : LOW;
    const int nb = hi - lo + 1;
    const uint32_t upper = hi == 31 ? 0u : ~((1u << (hi + 1)) - 1u);   // the digits already found
    sm.hist[tid] = 0;
    __syncthreads();
    if (key != 0u && (key & upper) == prefix) atomicAdd(&sm.hist[(key >> lo) & ((1u << nb) - 1u)], 1);
    __syncthreads();
    if (tid < 32) {
      // lane l holds digits 255 - 8l .. 248 - 8l (top first)
      int c[8];
      int lsum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c[e] = sm.hist[255 - 8 * lane - e];
        lsum += c[e];
      }
      int inc = lsum;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, m);
        if (lane >= m) inc += o;
      }
      const int excl = inc - lsum;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < rank && inc >= rank);
      if (hit) {
        const int l = __ffs(hit) - 1;
        if (lane == l) {
          int run = excl;
          int dg = 255 - 8 * lane;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (run + c[e] >= rank) {
              dg = 255 - 8 * lane - e;
              break;
            }
            run += c[e];
          }
          sm.pick_digit = dg;
          sm.pick_rank = rank - run;
        }
      } else if (lane == 0) {
        sm.pick_digit = -1;   // fewer than rank keys left: no key qualifies
        sm.pick_rank = rank;
      }
    }
    __syncthreads();
    const int dg = sm.pick_digit;
    if (dg < 0) return 0u;
    prefix |= (uint32_t)dg << lo;
    rank = sm.pick_rank;
  }
  return prefix;
}

template <typename T>
__global__ void __launch_bounds__(kSt, 3)
stream_topk_kernel(const Params p) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  constexpr int S = kStSTopk;
  constexpr int U = kStUTopk;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* ring = reinterpret_cast<uint4*>(smem_raw);
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw + (size_t)S * U * kSt * sizeof(uint4));
  const int tid = threadIdx.x;
  const int G = p.gamma, G1 = G + 1, V = p.V, k = p.top_k;
  RowWalk w;
  // target rows, then (q formed from the draft's logits) the draft rows,
  // whose kept lists the sequence finisher reads q from
  w.R = p.B * G1 + (p.ql ? p.B * G : 0);
  w.Rt = p.B * G1;
  w.ql = p.ql;
  w.G1 = G1;
  w.NV = V / VW;
  w.NVP = w.NV;
  w.CH = U * kSt;
  w.NCH = (w.NV + w.CH - 1) / w.CH;
  w.nrows = (w.R - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int MV = (w.NV + kSt - 1) / kSt;   // vectors of the thread with the most
  const T* logits = static_cast<const T*>(p.logits);
  // Rows are claimed as CTAs get through them (static dealing leaves the
  // CTAs that drew one row more, or share an SM with more CTAs, last): the
  // first row is blockIdx.x, the rest come from a counter.  Thread 0 claims
  // row j + 1 as row j starts and publishes it at a barrier before the issuer
  // looks up row j + 1 (with row j's last chunk, issued S chunks ahead of the
  // consumer, so at consumer chunk NCH - S - 1).  Needs rows of more than S
  // chunks, so that the ring never reaches past the next row.
  const bool dynamic = w.NCH > S;
  if (dynamic) {
    w.dyn = sm.rows;
    if (tid == 0) sm.rows[0] = blockIdx.x;
    __syncthreads();
  }

  Issuer<T, S, 1, U> iss;
  iss.start(logits, V, w);
#pragma unroll
  for (int s = 0; s < S; ++s) iss.issue(ring, logits, V, w);
  int stage = 0;
  for (int j = 0; w.live(j); ++j) {
    const int r = w.row_of(j);
    const bool draft_row = r >= w.Rt;
    const int rd = r - w.Rt;                                   // draft row index (draft rows)
    const int b = draft_row ? rd / G : r / G1;
    const int i = draft_row ? rd - b * G : r - b * G1;
    const int gb = seq_gamma(p, b);
    const T* row = draft_row ? static_cast<const T*>(p.ql) + (size_t)rd * V : logits + (size_t)r * V;
    __syncthreads();   // the previous row's shared state is no longer in use
    int claim = 0;
    if (tid == 0) {
      sm.count = 0;
      sm.nrel = 0;
      if (dynamic) claim = (int)gridDim.x + atomicAdd(p.ctr, 1);   // row j + 1
    }
    // the row's draft now, q(d) after pass 1 (its address needs the draft:
    // loading both here would hold warp 0 for two round trips)
    int d_row = -1;
    float q_row = 0.f;
    // (a vocabulary shard holds tokens from p.v0 on: the draft's index in its range)
    if (tid == 0 && i < gb && !p.ql) d_row = __ldg(p.draft + b * G + i) - p.v0;   // with ql: a_i in the finisher
    // ---- pass 1 through the ring: per thread its two best 16-byte vectors
    // (by maximum; the first such vector on ties) kept in registers with
    // their maxima m1 >= m2, and m3 = the largest maximum of its other vectors
    float m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
    uint4 bvec = make_uint4(0u, 0u, 0u, 0u), bvec2 = bvec;
    int bv = -1, bv2 = -1;
    int nan_seen = 0;
    for (int c = 0; c < w.NCH; ++c) {
      if (dynamic && c == w.NCH - S - 1) {
        // row j + 1's slot was row j - 3's: no longer read
        if (tid == 0) sm.rows[(j + 1) & 3] = claim;
        __syncthreads();
      }
      cpa_wait<S - 1>();
      const uint4* slot = ring + (size_t)stage * U * kSt;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = c * w.CH + u * kSt + tid;
        if (v < w.NV) {
          const uint4 x = slot[u * kSt + tid];
          const float vm = TR::template vmax<true>(x);
          nan_seen |= (vm != vm);
          m3 = fmaxf(m3, fminf(vm, m2));   // the vector that leaves the top two
          if (vm > m2) {
            if (vm > m1) {
              m2 = m1;
              bvec2 = bvec;
              bv2 = bv;
              m1 = vm;
              bvec = x;
              bv = v;
            } else {
              m2 = vm;
              bvec2 = x;
              bv2 = v;
            }
          }
        }
      }
      iss.issue(ring, logits, V, w);
      stage = (stage + 1 == S) ? 0 : stage + 1;
    }
    if (d_row >= 0 && d_row < V) q_row = p.q ? __ldg(p.q + ((size_t)b * G + i) * V + d_row) : 1.f;
    // ---- tau: the k-th largest finite thread maximum (its key bits from
    // bit 31 down to KEY_LOW_BIT, found by a radix select)
    const uint32_t tkey = m1 > -INFINITY ? okey(m1) : 0u;
    const uint32_t K = kth_largest_key<TR::KEY_LOW_BIT>(tkey, k, sm);
    const float tau = K == 0u ? -INFINITY : key_to_float(K);
    // ---- candidates.  A thread with m1 >= tau and m3 < tau has all its
    // elements >= tau in its two kept vectors; one with m3 >= tau too is
    // re-read (pass 2).
    if (m1 > -INFINITY && m1 >= tau) {
      if (m3 > -INFINITY && m3 >= tau) {
        sm.rel[atomicAdd(&sm.nrel, 1)] = tid;
      } else {
#pragma unroll
        for (int t = 0; t < VW; ++t) {
          const float xv = TR::get(bvec, t);
          if (xv > -INFINITY && xv >= tau) {
            const int pos = atomicAdd(&sm.count, 1);
            if (pos < kTkCap) sm.cand[pos] = comp_key(xv, bv * VW + t);
          }
        }
        if (m2 > -INFINITY && m2 >= tau) {
#pragma unroll
          for (int t = 0; t < VW; ++t) {
            const float xv = TR::get(bvec2, t);
            if (xv > -INFINITY && xv >= tau) {
              const int pos = atomicAdd(&sm.count, 1);
              if (pos < kTkCap) sm.cand[pos] = comp_key(xv, bv2 * VW + t);
            }
          }
        }
      }
    }
    const int bad_nan = __syncthreads_or(nan_seen);
    // ---- pass 2 (L2): the elements >= tau of the listed threads
    {
      const int nrel = sm.nrel;
      const int items = nrel * MV;
      for (int q0 = tid; q0 < items; q0 += kSt * 4) {
        uint4 x[4];
        int vv[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int q = q0 + h * kSt;
          vv[h] = -1;
          if (q < items) {
            const int l = q / MV, m = q - l * MV;
            const int v = sm.rel[l] + m * kSt;
            if (v < w.NV) {
              vv[h] = v;
              x[h] = ldg_v4(row + (size_t)v * VW);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          if (vv[h] >= 0 && !(TR::template vmax<false>(x[h]) < tau)) {
#pragma unroll
            for (int t = 0; t < VW; ++t) {
              const float xv = TR::get(x[h], t);
              if (xv > -INFINITY && xv >= tau) {   // NaN fails both
                const int pos = atomicAdd(&sm.count, 1);
                if (pos < kTkCap) sm.cand[pos] = comp_key(xv, vv[h] * VW + t);
              }
            }
          }
        }
      }
    }
    __syncthreads();
    int N = sm.count;
    if (N > kTkCap) {
      // more candidates than the buffer holds (heavy ties at tau): the exact
      // k-th largest (value, index) key by bisection over the row
      unsigned long long K64 = 0ull;
      for (int bit = 63; bit >= 0; --bit) {
        const unsigned long long Kt = K64 | (1ull << bit);
        int mine = 0;
        for (int vi = tid; vi < w.NV; vi += kSt) {
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
      for (int vi = tid; vi < w.NV; vi += kSt) {
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
    }
    // exact ranks among the candidates (keys are distinct: the index is in them)
    for (int e = tid; e < N; e += kSt) {
      const unsigned long long me = sm.cand[e];
      int rank = 0;
      for (int jj = 0; jj < N; ++jj) rank += sm.cand[jj] > me;
      if (rank < k) {
        sm.w[rank] = comp_val(me);
        sm.widx[rank] = comp_idx(me);
      }
    }
    __syncthreads();
    if (p.shard == 2) {
      // vocabulary shard: the row's local top-k and q there, merged across shards later
      topk_shard_candidates(p, r, b, i, min(k, N), bad_nan != 0, d_row, q_row, sm);
      continue;
    }
    topk_row_epilogue(p, b, i, gb,
                      draft_row ? p.qrowres + (size_t)rd * (k + 1) : p.rowres + (size_t)r * (k + 1),
                      min(k, N), bad_nan != 0, d_row, q_row, sm, draft_row);
    // the sequence is done when its target rows (and draft rows) all are
    if (arrive_last(p.seq_ticket + b, G1 + (p.ql ? G : 0), &sm.flag)) topk_finish_sequence(p, b, sm);
  }
  cpa_wait<0>();
  // every claim of this CTA has returned; the last CTA out resets the counter
  if (dynamic && tid == 0 && atomicAdd(p.ctr + 1, 1) == (int)gridDim.x - 1) {
    p.ctr[0] = 0;
    p.ctr[1] = 0;
  }
}

}  // namespace sv
