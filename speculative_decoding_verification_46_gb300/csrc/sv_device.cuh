// Device code of libspecverify: the batched verify/sample step of speculative
// decoding for sm_103a (GB300).
//
// The operation follows "11.1 核心原理: Draft + Verify 与 Rejection Sampling"
// (sections 11.1.1-11.1.3, code listing 10-1) and the notes "Fast Inference
// from Transformers via Speculative Decoding" (speculative-sampling paragraph):
// p_i = softmax(logits_i / T) (optionally top-k then top-p), accept d_i iff
// u_i < min(1, p_i(d_i) / q_i(d_i)), stop at the first rejection n, then draw
// from norm(max(p_n - q_n, 0)), or the bonus from p_gamma if all accepted.
// Greedy: accept while d_i == argmax p_i.
//
// Nothing here is a dense contraction: every kernel is bound by HBM bandwidth
// (the logits are streamed once; one row per sequence is touched again by the
// final draw).  Layout of the work:
//
//   rows_kernel      one CTA per (row, vocabulary slice); the slice is held in
//                    registers (U x 16-byte vectors per thread, 128-bit
//                    coalesced loads), reduced to a per-slice partial in
//                    workspace.  The last CTA to finish a sequence (an atomic
//                    ticket, no CTA ever waits) merges the partials and runs the
//                    acceptance scan.  In top-k mode a per-row ticket first
//                    merges the per-slice candidate lists of a row.
//   (untruncated sampling's final draw: sv_final.cuh)
//
// Data problems never trap: they set per-sequence status bits.  There are no
// spin-waits: cross-CTA hand-off is only "last arriving CTA continues".
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxU = 8;          // 16-byte vectors per thread per slice
constexpr int kCandCap = 2048;    // top-k candidate buffer (entries) per CTA
constexpr int kMaxK = 1024;       // largest top-k list
constexpr int kMaxG1 = 65;        // gamma + 1 <= 65

// per-sequence status bits (same values as the public header)
constexpr int SEQ_OOB = 1;
constexpr int SEQ_QBAD = 2;
constexpr int SEQ_BADROW = 4;
constexpr int SEQ_RESID0 = 8;

struct SeqState {
  int n;          // accepted count
  int status;     // SEQ_* bits gathered so far
  float M;        // max logit of the row the final draw uses
  float qm;       // q formed from the draft's logits: that row's maximum,
  double s;       // sum_v 2^((L_v - M) c) of the row the final draw uses
  float qinv;     // 1 / its sum of 2^((x - qm) c),
  int qbad;       // and whether it defines no distribution
  uint32_t tpK;   // top-p alone: the kept set of the row (key > tpK, or
  int tpIdx;      // key == tpK and index <= tpIdx)
};

struct Params {
  int B, gamma, V;
  int S, U, SL;          // rows kernel: slices per row, vectors per thread, slice length
  int FC;                // final draw: 512-token items per row
  int FZ;                // final draw: parts (CTAs) per sequence
  int top_k;             // top-k list length (top-k mode)
  int H;                 // streaming kernel: partial slots (segments) per row, 1, 2 or 4
  int SG;                // streaming kernel: its grid (CTA j streams vectors [j NVT / SG, (j+1) NVT / SG))
  int VWs;               // streaming kernel: elements per 16-byte vector
  long long NVT;         // streaming kernel: vectors of all its rows
  float top_p;
  float c;               // log2(e) / temperature (rounded to float)
  float c_lo;            // log2(e) / temperature - c
  const void* logits;
  const float* q;
  const int32_t* draft;
  const float* uniforms;
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_a;
  int32_t* out_status;
  int* seq_ticket;
  int* seq_ticket2;
  int* row_ticket;
  int* ctr;                       // [4] streaming top-k: next unclaimed row, CTAs done
  SeqState* seq;
  double* acc;                    // [B][gamma] acceptance probabilities (top-k mode)
  float4* part;                   // [R][S] per-slice partials
  unsigned long long* lists;      // [R][S][top_k] per-slice top-k candidates
  int2* rowres;                   // [R][top_k + 1] kept (index, probability) lists
  float4* fd_part;                // [B][FC] final-draw item sums (S, A as two-float pairs)
  float* fd_q;                    // [B][FC] final-draw item sums of q over the residual support
  const int* gamma_b;             // [B] drafts per sequence (ragged rounds), or nullptr: gamma
  const void* ql;                 // [B][gamma][V] draft logits (same dtype as logits) when q is formed
                                  // from them in the streaming path, else nullptr
  float4* qpart;                  // [B * gamma][H][kWarps] the draft rows' streaming partials (with ql)
  int2* qrowres;                  // [B * gamma][top_k + 1] the draft rows' kept lists (with ql and top-k / top-p)
  struct TpRow* tp;               // [B][gamma + 1] top-p alone: each row's kept set, mass and a_i
  // vocabulary-sharded verify (this process holds tokens [v0, v0 + V) of Vg)
  int v0, Vg;
  int nshard, rank;               // shards and this one's index (shards in token order)
  int shard;                      // final draw: 0 = whole row; 1 = write this shard's row-n totals, no search
  const void* sh_in;              // all shards' records (gathered by the caller)
  void* sh_out;                   // this shard's records
};

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// q(v) of a draft row from its logit x, the row's maximum qm and sum qs of
// 2^((x - qm) c): the weight is formed as every tail weight of the final draw
// (16-bit x - qm exact; -inf clamped to an exponent that flushes to 0;
// ex2.approx with a first-order correction), then divided by the sum.
__device__ __forceinline__ float q_weight(float x, float qm, float c, float c_lo) {
  const float dh = fmaxf(x - qm, -1.0e4f);
  const float p = dh * c;
  const float e = fmaf(dh, c_lo, fmaf(dh, c, -p));
  const float y = ex2_approx(p);
  return fmaf(y * 6.931471825e-01f, e, y);
}

// q of the final-draw row when it is formed from the draft's logits: the
// row's maximum, 1 / its sum, and whether the row defines no distribution
// (then q = 0).
struct QLrow {
  float m, inv;
  bool bad;
  __device__ __forceinline__ float q(float x, float c, float c_lo) const {
    return bad ? 0.f : q_weight(x, m, c, c_lo) * inv;
  }
};

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue early / wait until this grid's memory is visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}
__device__ __forceinline__ void set_word(uint4& v, int w, uint32_t x) {
  if (w == 0) v.x = x; else if (w == 1) v.y = x; else if (w == 2) v.z = x; else v.w = x;
}

// Order-preserving 32-bit key of a float; -0.0 is first made +0.0 so that equal
// values get equal keys.
__device__ __forceinline__ uint32_t okey(float x) {
  uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Composite ranking key: larger value first, then lower index first.
__device__ __forceinline__ unsigned long long comp_key(float x, int idx) {
  return ((unsigned long long)okey(x) << 32) | (unsigned long long)(~(uint32_t)idx);
}
__device__ __forceinline__ int comp_idx(unsigned long long c) {
  return (int)(~(uint32_t)(c & 0xffffffffull));
}
__device__ __forceinline__ float comp_val(unsigned long long c) {
  return key_to_float((uint32_t)(c >> 32));
}

// ------------------------------------------------------------------ dtype traits

template <typename T> struct Tr;

template <> struct Tr<float> {
  static constexpr int VW = 4;                // elements per 16-byte vector
  static constexpr int KEY_LOW_BIT = 0;       // lowest key bit that can differ
  static constexpr uint32_t kPadWord = 0xff800000u;   // -inf
  __device__ static __forceinline__ float get(const uint4& v, int t) {
    return __uint_as_float(word_of(v, t));
  }
  __device__ static __forceinline__ uint32_t scalar_bits(const float* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
  }
  __device__ static __forceinline__ void put(uint4& v, int t, uint32_t bits) { set_word(v, t, bits); }
  // max of the 4 values; NANPROP: a NaN anywhere gives NaN
  template <bool NANPROP>
  __device__ static __forceinline__ float vmax(const uint4& v) {
    float a = __uint_as_float(v.x), b = __uint_as_float(v.y);
    float c = __uint_as_float(v.z), d = __uint_as_float(v.w);
    float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
    if (NANPROP && (a != a || b != b || c != c || d != d)) m = __uint_as_float(0x7fffffffu);
    return m;
  }
};

template <> struct Tr<__nv_bfloat16> {
  static constexpr int VW = 8;
  static constexpr int KEY_LOW_BIT = 16;
  static constexpr uint32_t kPadWord = 0xff80ff80u;
  __device__ static __forceinline__ float get(const uint4& v, int t) {
    uint32_t w = word_of(v, t >> 1);
    uint32_t bits = (t & 1) ? (w & 0xffff0000u) : (w << 16);
    return __uint_as_float(bits);
  }
  __device__ static __forceinline__ uint32_t scalar_bits(const __nv_bfloat16* p) {
    return (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p));
  }
  __device__ static __forceinline__ void put(uint4& v, int t, uint32_t bits) {
    uint32_t w = word_of(v, t >> 1);
    w = (t & 1) ? ((w & 0x0000ffffu) | (bits << 16)) : ((w & 0xffff0000u) | bits);
    set_word(v, t >> 1, w);
  }
  template <bool NANPROP>
  __device__ static __forceinline__ float vmax(const uint4& v) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    __nv_bfloat162 m = NANPROP ? __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d))
                               : __hmax2(__hmax2(a, b), __hmax2(c, d));
    float lo = __low2float(m), hi = __high2float(m);
    if (NANPROP && (lo != lo || hi != hi)) return __uint_as_float(0x7fffffffu);
    return fmaxf(lo, hi);
  }
};

template <> struct Tr<__half> {
  static constexpr int VW = 8;
  static constexpr int KEY_LOW_BIT = 13;
  static constexpr uint32_t kPadWord = 0xfc00fc00u;
  __device__ static __forceinline__ float get(const uint4& v, int t) {
    uint32_t w = word_of(v, t >> 1);
    unsigned short bits = (unsigned short)((t & 1) ? (w >> 16) : (w & 0xffffu));
    return __half2float(__ushort_as_half(bits));
  }
  __device__ static __forceinline__ uint32_t scalar_bits(const __half* p) {
    return (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p));
  }
  __device__ static __forceinline__ void put(uint4& v, int t, uint32_t bits) {
    uint32_t w = word_of(v, t >> 1);
    w = (t & 1) ? ((w & 0x0000ffffu) | (bits << 16)) : ((w & 0xffff0000u) | bits);
    set_word(v, t >> 1, w);
  }
  template <bool NANPROP>
  __device__ static __forceinline__ float vmax(const uint4& v) {
    __half2 a = *reinterpret_cast<const __half2*>(&v.x);
    __half2 b = *reinterpret_cast<const __half2*>(&v.y);
    __half2 c = *reinterpret_cast<const __half2*>(&v.z);
    __half2 d = *reinterpret_cast<const __half2*>(&v.w);
    __half2 m = NANPROP ? __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d))
                        : __hmax2(__hmax2(a, b), __hmax2(c, d));
    float lo = __low2float(m), hi = __high2float(m);
    if (NANPROP && (lo != lo || hi != hi)) return __uint_as_float(0x7fffffffu);
    return fmaxf(lo, hi);
  }
};

// One 16-byte slot of VW elements starting at element e0 of `row`; the first
// nv (1..VW) are real, the rest are -inf.  Vector load when the slot is full and
// 16-byte aligned.
template <typename T>
__device__ __forceinline__ uint4 load_slot(const T* row, int e0, int nv, bool vec_ok) {
  using TR = Tr<T>;
  if (nv == TR::VW && vec_ok) return ldg_v4(row + e0);
  uint4 v = make_uint4(TR::kPadWord, TR::kPadWord, TR::kPadWord, TR::kPadWord);
#pragma unroll
  for (int t = 0; t < TR::VW; ++t)
    if (t < nv) TR::put(v, t, TR::scalar_bits(row + e0 + t));
  return v;
}

// ------------------------------------------------------------------ reductions

// Two-float (hi + lo) sums: error-free transformation per addition, so block
// totals keep about 44 bits while every operation stays on the float32 pipes.
struct F2 {
  float hi, lo;
};
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  float s = a.hi + b.hi;
  float bb = s - a.hi;
  float e = (a.hi - (s - bb)) + (b.hi - bb);
  e += a.lo + b.lo;
  float h = s + e;
  return F2{h, e - (h - s)};
}
// Two-float (Dekker) products and a two-float exp2, for the one row per
// sequence whose inverse CDF must agree with a float64 reference to ~1e-10.
__device__ __forceinline__ F2 f2_norm(float s, float e) {
  const float h = s + e;
  return F2{h, e - (h - s)};
}
// a * b, both two-float
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return f2_norm(p, e);
}
__device__ __forceinline__ F2 f2_neg(F2 a) { return F2{-a.hi, -a.lo}; }

// 2^(j/64), j = 0..63, as float pairs (hi + lo) rounded from the exact values.
__device__ const float kExp2Hi[64] = {
    1.000000000e+00f, 1.010889292e+00f, 1.021897197e+00f, 1.033024907e+00f,
    1.044273734e+00f, 1.055645227e+00f, 1.067140460e+00f, 1.078760743e+00f,
    1.090507746e+00f, 1.102382541e+00f, 1.114386797e+00f, 1.126521587e+00f,
    1.138788581e+00f, 1.151189208e+00f, 1.163724899e+00f, 1.176396966e+00f,
    1.189207077e+00f, 1.202156782e+00f, 1.215247393e+00f, 1.228480577e+00f,
    1.241857767e+00f, 1.255380750e+00f, 1.269050956e+00f, 1.282870054e+00f,
    1.296839595e+00f, 1.310961246e+00f, 1.325236678e+00f, 1.339667559e+00f,
    1.354255557e+00f, 1.369002461e+00f, 1.383909941e+00f, 1.398979664e+00f,
    1.414213538e+00f, 1.429613352e+00f, 1.445180774e+00f, 1.460917830e+00f,
    1.476826191e+00f, 1.492907763e+00f, 1.509164453e+00f, 1.525598168e+00f,
    1.542210817e+00f, 1.559004426e+00f, 1.575980902e+00f, 1.593142152e+00f,
    1.610490322e+00f, 1.628027439e+00f, 1.645755529e+00f, 1.663676620e+00f,
    1.681792855e+00f, 1.700106382e+00f, 1.718619347e+00f, 1.737333894e+00f,
    1.756252170e+00f, 1.775376439e+00f, 1.794709086e+00f, 1.814252138e+00f,
    1.834008098e+00f, 1.853979111e+00f, 1.874167681e+00f, 1.894575953e+00f,
    1.915206552e+00f, 1.936061740e+00f, 1.957144141e+00f, 1.978456020e+00f,
};
__device__ const float kExp2Lo[64] = {
    0.000000000e+00f, -5.711605411e-09f, -4.811559862e-08f, -2.809089317e-08f,
    4.833470157e-08f, -4.907169426e-08f, -5.933751979e-08f, 5.461594554e-08f,
    -1.307753994e-08f, 4.260501996e-08f, -5.435540018e-08f, 3.123641434e-08f,
    5.386222313e-08f, 2.192228266e-08f, -4.051441493e-08f, 2.566975077e-08f,
    3.797635273e-08f, -5.069756526e-08f, -3.267394888e-08f, -4.136200360e-08f,
    4.496838102e-08f, 7.322237483e-09f, 1.419333318e-09f, -3.816621685e-08f,
    -4.018999533e-08f, -3.496571566e-08f, -3.496373324e-08f, -3.461673970e-08f,
    -1.012334927e-08f, -3.845881835e-08f, -5.875577358e-08f, 8.689434061e-09f,
    2.420323497e-08f, -1.342992917e-08f, 3.324199938e-08f, -3.628657552e-08f,
    -4.500898854e-08f, -3.423620143e-08f, -2.495937323e-08f, -1.762856883e-08f,
    8.070904833e-09f, -2.576466507e-08f, -5.661025426e-08f, -4.903136785e-10f,
    9.836217174e-09f, -1.726008314e-08f, -5.124972091e-08f, -3.920298752e-08f,
    -2.475532668e-08f, -2.865147231e-08f, -4.849617596e-08f, -5.850223417e-08f,
    -9.235770371e-09f, 5.343197884e-08f, -1.141504491e-08f, 3.736258236e-08f,
    -1.123927795e-08f, 1.436561181e-08f, -4.663005626e-08f, 2.810338451e-08f,
    9.845328108e-09f, 5.357072297e-08f, -1.702180441e-08f, 6.032726318e-09f,
};

// 2^a for a two-float a with a.hi <= ~127, to ~2e-12 relative (Tang's
// table-driven method): k = round(64 a), 2^a = 2^(k>>6) * 2^((k&63)/64) * e^g
// with g = (a - k/64) ln 2, |g| <= ln 2 / 128.  The 64 values 2^(j/64) are
// float pairs from their exact values; e^g = 1 + g + (g^2/2 + g^3/6 + g^4/24),
// the bracket (< 2e-5) in float32.  a.hi < -125 gives 0.  tab: the 64 high
// then the 64 low parts, staged in shared memory by load_exp2_table.
__device__ __forceinline__ F2 exp2_f2(F2 a, const float* tab) {
  const F2 kLn2{6.931471825e-01f, -1.904654212e-09f};
  if (a.hi < -125.f) return F2{0.f, 0.f};
  const float k = rintf(a.hi * 64.f);
  const F2 r = f2_norm(a.hi - k * 0.015625f, a.lo);   // the subtraction is exact
  const float gh = r.hi * kLn2.hi;
  const float gl = fmaf(r.hi, kLn2.hi, -gh) + fmaf(r.hi, kLn2.lo, r.lo * kLn2.hi);
  const float small = gh * gh * fmaf(gh, fmaf(gh, 1.0f / 24.0f, 1.0f / 6.0f), 0.5f);
  const float eh = 1.f + gh;                          // |gh| < 1: Fast2Sum
  const float el = ((1.f - eh) + gh) + (gl + small);
  const int ki = (int)k;
  const int j = ki & 63;
  const float th = tab[j], tl = tab[64 + j];
  const float yh = th * eh;
  const float yl = fmaf(th, eh, -yh) + fmaf(th, el, tl * eh);
  const float scale = __int_as_float((127 + (ki >> 6)) << 23);   // 2^(k>>6), k>>6 in [-125, 127]
  return F2{yh * scale, yl * scale};
}

// Stage the exp2_f2 table (128 floats) in shared memory; visible to the
// block after its next barrier.
__device__ __forceinline__ void load_exp2_table(float* tab) {
  for (int i = threadIdx.x; i < 128; i += blockDim.x) tab[i] = i < 64 ? __ldg(kExp2Hi + i) : __ldg(kExp2Lo + i - 64);
}

// Ordering of normalised two-float numbers (|lo| <= ulp(hi) / 2, as f2_add
// returns them).
__device__ __forceinline__ bool f2_lt(F2 a, F2 b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ bool f2_pos(F2 a) { return a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f); }
// u * a with the product's rounding error kept (FMA two-product).
__device__ __forceinline__ F2 f2_scale(F2 a, float u) {
  const float p = u * a.hi;
  float e = fmaf(u, a.hi, -p);
  e = fmaf(u, a.lo, e);
  const float h = p + e;
  return F2{h, e - (h - p)};
}
// 1 / (a.hi + a.lo) in float32: the reciprocal of hi refined by one Newton
// step against the two-float value (within an ulp of the exact reciprocal).
// hi = 0 gives +inf, an infinite hi 0.
__device__ __forceinline__ float f2_rcp(F2 a) {
  const float r = 1.f / a.hi;
  float e = fmaf(-r, a.hi, 1.f);
  e = fmaf(-r, a.lo, e);
  return e == e ? fmaf(r, e, r) : r;
}
__device__ __forceinline__ F2 f2_shfl_xor(F2 a, int m) {
  return F2{__shfl_xor_sync(0xffffffffu, a.hi, m), __shfl_xor_sync(0xffffffffu, a.lo, m)};
}
__device__ __forceinline__ F2 f2_shfl_up(F2 a, int m) {
  return F2{__shfl_up_sync(0xffffffffu, a.hi, m), __shfl_up_sync(0xffffffffu, a.lo, m)};
}

// Block-wide F2 sum; every thread gets the total.  Uses `sm` (kWarps entries).
__device__ __forceinline__ F2 block_sum_f2(F2 v, F2* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = f2_add(v, f2_shfl_xor(v, m));
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  F2 t = sm[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) t = f2_add(t, sm[w]);
  return t;
}

// Block-wide exclusive prefix of F2 values in thread order, plus the total.
__device__ __forceinline__ F2 block_exclusive_f2(F2 v, F2* sm, F2* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  F2 inc = v;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    F2 o = f2_shfl_up(inc, m);
    if (lane >= m) inc = f2_add(o, inc);
  }
  __syncthreads();
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  F2 base{0.f, 0.f}, tot{0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) base = f2_add(base, sm[w]);
    tot = f2_add(tot, sm[w]);
  }
  *total = tot;
  // exclusive prefix = warp base + inclusive prefix of the lane below
  F2 below = f2_shfl_up(inc, 1);
  if (lane == 0) below = F2{0.f, 0.f};
  return f2_add(base, below);
}

__device__ __forceinline__ float block_max(float v, float* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  float t = sm[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) t = fmaxf(t, sm[w]);
  return t;
}

__device__ __forceinline__ int block_sum_int(int v, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += sm[w];
  return t;
}

__device__ __forceinline__ double warp_incl_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, m);
    if (lane >= m) v += o;
  }
  return v;
}

__device__ __forceinline__ F2 warp_incl_scan_f2(F2 v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const F2 o = f2_shfl_up(v, m);
    if (lane >= m) v = f2_add(o, v);
  }
  return v;
}

struct LocateSmem {
  F2 wsum[32];
  F2 carry;
  F2 base;
  F2 lastbase;
  int found;
  int last;
};

// Block-wide inverse-CDF search over NT two-float masses in index order
// (global or shared memory): total R, then the first k whose running interval
// [prefix_k, prefix_k + m_k) holds t = u * R.  Both passes add in the same
// order, so t < R lands inside unless rounding pushes it to the very end, in
// which case the last positive mass is taken.  Returns k (-1 if R <= 0), its
// exclusive prefix in *base_out and t in *t_out; every thread gets them.
// Float32 pipes only (two-float sums): this part's float64 rate is low.
__device__ int block_locate(const F2* masses, int NT, float u, F2* R_out, F2* base_out, F2* t_out,
                            LocateSmem& ls, bool from_global) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = blockDim.x >> 5, nt = blockDim.x;
  F2 R{0.f, 0.f};
  F2 t{0.f, 0.f};
  for (int pass = 0; pass < 2; ++pass) {
    t = f2_scale(R, u);
    __syncthreads();   // every thread has read ls (the previous pass's total) before it is reset
    if (tid == 0) {
      ls.carry = F2{0.f, 0.f};
      ls.found = 0x7fffffff;
      ls.last = -1;
      ls.lastbase = F2{0.f, 0.f};
    }
    __syncthreads();
    for (int c0 = 0; c0 < NT; c0 += nt) {
      const int k = c0 + tid;
      F2 m{0.f, 0.f};
      if (k < NT) {
        if (from_global) {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(masses) + k);
          m = F2{v.x, v.y};
        } else {
          m = masses[k];
        }
      }
      const F2 inc = warp_incl_scan_f2(m);
      if (lane == 31) ls.wsum[warp] = inc;
      __syncthreads();
      F2 off = ls.carry, tot = ls.carry;
      for (int w = 0; w < nw; ++w) {
        if (w < warp) off = f2_add(off, ls.wsum[w]);
        tot = f2_add(tot, ls.wsum[w]);
      }
      F2 below = f2_shfl_up(inc, 1);
      if (lane == 0) below = F2{0.f, 0.f};
      const F2 excl = f2_add(off, below);
      if (pass == 1 && k < NT && f2_pos(m)) {
        if (!f2_lt(t, excl) && f2_lt(t, f2_add(excl, m))) atomicMin(&ls.found, k);   // at most one k
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
  if (ls.found != 0x7fffffff) { *base_out = ls.base; return ls.found; }
  *base_out = ls.lastbase;
  return ls.last;
}

// The same search done by warp 0 alone (no block barriers during the scan;
// one __syncthreads publishes the result).  Same summation order for the
// total and the prefixes: 32-wide chunks, two-float inclusive scans, carry.
__device__ int warp_locate(const F2* masses, int NT, float u, F2* R_out, F2* base_out, F2* t_out,
                           LocateSmem& ls, bool from_global) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    const int lane = tid;
    auto load = [&](int k) -> F2 {
      if (k >= NT) return F2{0.f, 0.f};
      if (from_global) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(masses) + k);
        return F2{v.x, v.y};
      }
      return masses[k];
    };
    F2 carry{0.f, 0.f};
    for (int c0 = 0; c0 < NT; c0 += 32) {
      const F2 inc = f2_add(carry, warp_incl_scan_f2(load(c0 + lane)));
      carry = F2{__shfl_sync(0xffffffffu, inc.hi, 31), __shfl_sync(0xffffffffu, inc.lo, 31)};
    }
    const F2 R = carry;
    const F2 t = f2_scale(R, u);
    int found = -1, last = -1;
    F2 fbase{0.f, 0.f}, lbase{0.f, 0.f};
    carry = F2{0.f, 0.f};
    for (int c0 = 0; c0 < NT && found < 0; c0 += 32) {
      const F2 m = load(c0 + lane);
      const F2 inc = f2_add(carry, warp_incl_scan_f2(m));
      F2 excl = F2{__shfl_up_sync(0xffffffffu, inc.hi, 1), __shfl_up_sync(0xffffffffu, inc.lo, 1)};
      if (lane == 0) excl = carry;
      const bool live = c0 + lane < NT && f2_pos(m);
      const unsigned hit = __ballot_sync(0xffffffffu, live && !f2_lt(t, excl) && f2_lt(t, f2_add(excl, m)));
      const unsigned pos = __ballot_sync(0xffffffffu, live);
      if (hit) {
        const int l = __ffs(hit) - 1;
        found = c0 + l;
        fbase = F2{__shfl_sync(0xffffffffu, excl.hi, l), __shfl_sync(0xffffffffu, excl.lo, l)};
      }
      if (pos) {
        const int l = 31 - __clz(pos);
        last = c0 + l;
        lbase = F2{__shfl_sync(0xffffffffu, excl.hi, l), __shfl_sync(0xffffffffu, excl.lo, l)};
      }
      carry = F2{__shfl_sync(0xffffffffu, inc.hi, 31), __shfl_sync(0xffffffffu, inc.lo, 31)};
    }
    if (lane == 0) {
      ls.carry = R;
      ls.wsum[0] = t;
      ls.found = found >= 0 ? found : last;
      ls.base = found >= 0 ? fbase : lbase;
    }
  }
  __syncthreads();
  *R_out = ls.carry;
  *t_out = ls.wsum[0];
  *base_out = ls.base;
  const int k = f2_pos(ls.carry) ? ls.found : -1;
  __syncthreads();   // ls may be reused right after
  return k;
}

__device__ __forceinline__ int locate(const F2* masses, int NT, float u, F2* R_out, F2* base_out, F2* t_out,
                                      LocateSmem& ls, bool from_global) {
  return NT <= 1024 ? warp_locate(masses, NT, u, R_out, base_out, t_out, ls, from_global)
                    : block_locate(masses, NT, u, R_out, base_out, t_out, ls, from_global);
}

// "Does (va, ia) beat (vb, ib)?" for the greedy argmax: a larger value wins,
// equal values (-0.0 == +0.0) go to the lower index; NaN wins (it is flagged).
__device__ __forceinline__ bool argmax_better(float va, int ia, float vb, int ib) {
  const bool na = va != va, nb = vb != vb;
  if (na || nb) return (na && nb) ? (ia < ib) : na;
  if (va > vb) return true;
  if (va < vb) return false;
  return ia < ib;
}

// Drafts of sequence b in this round: gamma_b[b] clamped to [0, gamma] for a
// ragged round, else gamma.  Its rows beyond gamma_b are not part of the round.
__device__ __forceinline__ int seq_gamma(const Params& p, int b) {
  if (!p.gamma_b) return p.gamma;
  return min(max(__ldg(p.gamma_b + b), 0), p.gamma);
}

// Last-arriving-CTA hand-off.  Every thread's writes are collected by the
// barrier; thread 0 then takes a ticket with one acquire-release atomic (the
// release publishes what the CTA wrote, the acquire makes the other CTAs'
// writes visible to the last one; the closing barrier extends both to the
// whole CTA).  The CTA that takes ticket count-1 resets the counter and
// returns true; its later reads of other CTAs' data use ld.global.cg.
// single_writer is kept for the call sites that document that only thread 0
// wrote: the ordering is the same either way.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ bool arrive_last(int* ticket, int count, int* s_flag, bool single_writer = false) {
  (void)single_writer;
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomic_add_acq_rel_gpu(ticket, 1);
    const int last = (prev == count - 1);
    if (last) *ticket = 0;
    *s_flag = last;
  }
  __syncthreads();
  return *s_flag != 0;
}

// ------------------------------------------------------------------ rows kernel

enum { MODE_GREEDY = 0, MODE_SOFTMAX = 1, MODE_TOPK = 2, MODE_TOPP = 3 };

struct RowsSmem {
  float fred[kWarps];
  int ired[kWarps];
  F2 f2red[kWarps];
  float2 pair[kWarps];
  int flag;
  int count;
  int n;
  int token;
  float M[kMaxG1];
  double s[kMaxG1];
  float a[kMaxG1];
  int g[kMaxG1];
  int bad[kMaxG1];
  int status;
  double dred[kWarps];
  int dr[kMaxG1];          // this sequence's drafts, loaded at kernel start
  float ur[kMaxG1];        // and its uniforms
  unsigned long long cand[kCandCap];   // top-k candidates; reused by the row merge
  unsigned long long mout[kMaxK];
  double w[kMaxK];
  int widx[kMaxK];
};

// Greedy / softmax sequence finisher: one warp per row merges that row's S
// slice partials (lanes load them in parallel), then the acceptance scan.
template <typename T, int MODE>
__device__ void finish_sequence_dense(const Params& p, int b, RowsSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.gamma, G1 = G + 1, V = p.V, S = p.S;
  const int gb = seq_gamma(p, b);
  for (int i = warp; i < G1; i += kWarps) {
    const int rr = b * G1 + i;
    const float4* pp = p.part + (size_t)rr * S;
    if (MODE == MODE_GREEDY) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll 4
      for (int s2 = lane; s2 < S; s2 += 32) {
        const float4 v = __ldcg(pp + s2);
        const int vi = __float_as_int(v.y);
        if (argmax_better(v.x, vi, bv, bi)) { bv = v.x; bi = vi; }
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, m);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, m);
        if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        const bool nan = bv != bv;
        sm.g[i] = (nan || bi == 0x7fffffff) ? 0 : bi;
        sm.bad[i] = (nan && i <= gb) ? 1 : 0;
      }
    } else {
      float M = -INFINITY;
#pragma unroll 4
      for (int s2 = lane; s2 < S; s2 += 32) M = fmaxf(M, __ldcg(pp + s2).x);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
      F2 acc{0.f, 0.f};
      if (M > -INFINITY && M < INFINITY) {
#pragma unroll 4
        for (int s2 = lane; s2 < S; s2 += 32) {
          const float4 v = __ldcg(pp + s2);
          if (v.x > -INFINITY) {
            const float sc = exp2f((v.x - M) * p.c);
            acc = f2_add(acc, f2_add(F2{v.y * sc, 0.f}, F2{v.z * sc, 0.f}));
          }
        }
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) acc = f2_add(acc, f2_shfl_xor(acc, m));
      if (lane == 0) {
        const double s = (double)acc.hi + (double)acc.lo;
        const bool bad = !(M > -INFINITY && M < INFINITY) || !(s > 0.0 && s < 1e300);
        sm.M[i] = M;
        sm.s[i] = s;
        sm.bad[i] = (bad && i <= gb) ? 1 : 0;
        if (i < gb) {
          const int d = sm.dr[i];
          float a = 0.f;
          int st = 0;
          if (d < 0 || d >= V) {
            st |= SEQ_OOB;
          } else {
            const T* row = static_cast<const T*>(p.logits) + (size_t)rr * V;
            const float l = Tr<T>::get(load_slot<T>(row, d, 1, false), 0);
            const float qd = p.q ? __ldg(p.q + ((size_t)b * G + i) * V + d) : 1.f;   // NULL: one-hot
            const float pd = bad ? 0.f : exp2f((l - M) * p.c) / (float)s;
            if (qd > 0.0f) {
              a = fminf(1.f, pd / qd);
            } else {
              a = pd > 0.f ? 1.f : 0.f;
              st |= SEQ_QBAD;
            }
          }
          sm.a[i] = a;
          sm.g[i] = st;
          if (p.out_a) p.out_a[b * G + i] = a;
        } else if (i < G && p.out_a) {
          p.out_a[b * G + i] = 0.f;   // beyond this sequence's drafts
        }
      }
    }
  }
  __syncthreads();
  // every partial of this sequence has been read: leave the workspace zeroed
  for (int e = tid; e < G1 * S; e += kThreads)
    p.part[(size_t)b * G1 * S + e] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid == 0) {
    int status = 0, n = gb;
    for (int i = 0; i <= gb; ++i)
      if (sm.bad[i]) status |= SEQ_BADROW;
    if (MODE == MODE_GREEDY) {
      for (int i = 0; i < gb; ++i) {
        const int d = sm.dr[i];
        if (d < 0 || d >= V) status |= SEQ_OOB;
      }
      for (int i = 0; i < gb; ++i)
        if (sm.dr[i] != sm.g[i]) { n = i; break; }
      sm.token = sm.g[n];
    } else {
      for (int i = 0; i < gb; ++i) status |= sm.g[i];
      for (int i = 0; i < gb; ++i)
        if (!(sm.ur[i] < (float)sm.a[i])) { n = i; break; }
      SeqState st;
      st.n = n;
      st.status = status;
      st.M = sm.M[n];
      st.qm = 0.f;
      st.s = sm.s[n];
      st.qinv = 0.f;
      st.qbad = 0;
      st.tpK = 0u;
      st.tpIdx = 0;
      p.seq[b] = st;
    }
    sm.n = n;
    sm.status = status;
    p.out_n[b] = n;
    if (MODE == MODE_GREEDY && p.out_status) p.out_status[b] = status;
  }
  __syncthreads();
  const int n = sm.n;
  for (int j = tid; j < G1; j += kThreads) {
    if (j < n) p.out_tokens[b * G1 + j] = sm.dr[j];
    else if (j > n) p.out_tokens[b * G1 + j] = -1;
    else if (MODE == MODE_GREEDY) p.out_tokens[b * G1 + j] = sm.token;
  }
}

// Number of entries of the descending list X[0..n) that beat key v.
__device__ __forceinline__ int count_greater(const unsigned long long* X, int n, unsigned long long v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (X[mid] > v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Top-k row finisher: merge the S per-slice lists of row rr into the row's
// top-k, apply softmax(./T) over it, cut by top-p, renormalise, store the kept
// (index, probability) list and the acceptance probability of the row's draft.
__device__ void finish_row_topk(const Params& p, int b, int i, int rr, RowsSmem& sm) {
  const int tid = threadIdx.x;
  const int k = p.top_k, G = p.gamma, V = p.V;
  const int gb = seq_gamma(p, b);
  unsigned long long* A = sm.cand;            // running merged list
  unsigned long long* Bl = sm.cand + kMaxK;   // next slice list
  unsigned long long* O = sm.mout;
  const unsigned long long* L0 = p.lists + (size_t)rr * p.S * k;
  int na = 0;
  {
    int c = 0;
    for (int e = tid; e < k; e += kThreads) {
      const unsigned long long v = __ldcg(L0 + e);
      A[e] = v;
      c += v != 0ull;
    }
    na = block_sum_int(c, sm.ired);
  }
  for (int s2 = 1; s2 < p.S; ++s2) {
    const unsigned long long* Ls = L0 + (size_t)s2 * k;
    int c = 0;
    for (int e = tid; e < k; e += kThreads) {
      const unsigned long long v = __ldcg(Ls + e);
      Bl[e] = v;
      c += v != 0ull;
    }
    const int nb = block_sum_int(c, sm.ired);   // includes a __syncthreads
    for (int e = tid; e < na; e += kThreads) {
      const int rank = e + count_greater(Bl, nb, A[e]);
      if (rank < k) O[rank] = A[e];
    }
    for (int e = tid; e < nb; e += kThreads) {
      const int rank = e + count_greater(A, na, Bl[e]);
      if (rank < k) O[rank] = Bl[e];
    }
    na = min(k, na + nb);
    __syncthreads();
    for (int e = tid; e < na; e += kThreads) A[e] = O[e];
    __syncthreads();
  }
  // the slice lists have been consumed: leave the workspace zeroed
  for (int e = tid; e < p.S * k; e += kThreads) p.lists[(size_t)rr * p.S * k + e] = 0ull;
  // softmax over the merged top-k (descending), then the top-p cut
  const float m = na > 0 ? comp_val(A[0]) : -INFINITY;
  const bool bad = !(m > -INFINITY && m < INFINITY);
  for (int e = tid; e < na; e += kThreads) {
    sm.w[e] = bad ? 0.0 : (double)exp2f((comp_val(A[e]) - m) * p.c);
    sm.widx[e] = comp_idx(A[e]);
  }
  __syncthreads();
  int2* out = p.rowres + (size_t)rr * (k + 1);
  if (tid == 0) {
    int J = na;
    double W = 0.0;
    for (int e = 0; e < na; ++e) W += sm.w[e];
    if (bad || na == 0) {
      J = na > 0 ? 1 : 0;
      if (na > 0) sm.w[0] = 1.0;
      W = 1.0;
      if (bad && i <= gb) atomicOr(&p.seq[b].status, SEQ_BADROW);
    } else if (p.top_p < 1.0f) {
      const double tp = (double)p.top_p;
      double cum = 0.0;
      for (int e = 0; e < na; ++e) {
        cum += sm.w[e];
        if (cum / W >= tp) { J = e + 1; break; }
      }
    }
    double WJ = 0.0;
    for (int e = 0; e < J; ++e) WJ += sm.w[e];
    sm.count = J;
    sm.s[0] = WJ;
    out[0] = make_int2(J, 0);
  }
  __syncthreads();
  const int J = sm.count;
  const double WJ = sm.s[0];
  for (int e = tid; e < J; e += kThreads)
    out[1 + e] = make_int2(sm.widx[e], __float_as_int((float)(sm.w[e] / WJ)));
  // acceptance probability of this row's draft
  if (i < gb) {
    const int d = p.draft[b * G + i];
    if (tid == 0) sm.dred[0] = 0.0;
    __syncthreads();
    if (d >= 0 && d < V)
      for (int e = tid; e < J; e += kThreads)
        if (sm.widx[e] == d) sm.dred[0] = sm.w[e] / WJ;
    __syncthreads();
    if (tid == 0) {
      double a = 0.0;
      int st = 0;
      if (d < 0 || d >= V) {
        st |= SEQ_OOB;
      } else {
        const double pd = sm.dred[0];
        const float qd = p.q ? __ldg(p.q + ((size_t)b * G + i) * V + d) : 1.f;   // NULL: one-hot
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
}

// Top-k sequence finisher: scan, then the final draw from the kept list of
// row n (residual against q gathered at the kept indices) or row gamma.
__device__ void finish_sequence_topk(const Params& p, int b, RowsSmem& sm) {
  const int tid = threadIdx.x;
  const int k = p.top_k, G = p.gamma, G1 = G + 1, V = p.V;
  const int gb = seq_gamma(p, b);
  if (tid == 0) {
    int n = gb;
    for (int i = 0; i < gb; ++i) {
      const double u = (double)p.uniforms[b * G1 + i];
      if (!(u < __ldcg(p.acc + b * G + i))) { n = i; break; }
    }
    sm.n = n;
    sm.status = __ldcg(&p.seq[b].status);
  }
  __syncthreads();
  const int n = sm.n;
  const int rr = b * G1 + n;
  const int2* kept = p.rowres + (size_t)rr * (k + 1);
  const int J = __ldcg(kept).x;
  const bool resid = n < gb;
  const float* qrow = (resid && p.q) ? p.q + ((size_t)b * G + n) * V : nullptr;
  const int dn = (resid && !p.q) ? __ldg(p.draft + b * G + n) : -1;   // deterministic draft: q_n one-hot
  // r_j in index order: rank each kept entry by its index
  for (int e = tid; e < J; e += kThreads) {
    const int2 en = __ldcg(kept + 1 + e);
    sm.widx[e] = en.x;
    sm.w[e] = (double)__int_as_float(en.y);
  }
  __syncthreads();
  for (int e = tid; e < J; e += kThreads) {
    const int me = sm.widx[e];
    int rank = 0;
    for (int j = 0; j < J; ++j) rank += sm.widx[j] < me;
    double r = sm.w[e];
    if (resid) r = fmax(r - (qrow ? (double)__ldg(qrow + me) : (me == dn ? 1.0 : 0.0)), 0.0);
    sm.mout[rank] = (unsigned long long)me;
    reinterpret_cast<double*>(sm.cand)[rank] = r;
  }
  __syncthreads();
  if (tid == 0) {
    double* rs = reinterpret_cast<double*>(sm.cand);
    int status = sm.status;
    double R = 0.0;
    for (int e = 0; e < J; ++e) R += rs[e];
    if (resid && !(R > 0.0)) {
      // zero residual mass (only through rounding): draw from p_n instead
      status |= SEQ_RESID0;
      for (int e = 0; e < J; ++e) {
        double pe = 0.0;
        for (int j = 0; j < J; ++j)
          if (sm.widx[j] == (int)sm.mout[e]) pe = sm.w[j];
        rs[e] = pe;
      }
      R = 0.0;
      for (int e = 0; e < J; ++e) R += rs[e];
    }
    const double t = (double)p.uniforms[b * G1 + gb] * R;
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
  for (int j = tid; j < G1; j += kThreads)
    p.out_tokens[b * G1 + j] = j < n ? p.draft[b * G + j] : (j == n ? sm.token : -1);
  if (p.out_a)
    for (int j = gb + tid; j < G; j += kThreads) p.out_a[b * G + j] = 0.f;   // beyond this sequence's drafts
  // kept lists and acceptance probabilities have been consumed: zero them
  for (int e = tid; e < G1 * (k + 1); e += kThreads) p.rowres[(size_t)b * G1 * (k + 1) + e] = make_int2(0, 0);
  for (int e = tid; e < G; e += kThreads) p.acc[b * G + e] = 0.0;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads)
rows_kernel(const Params p) {
  using TR = Tr<T>;
  constexpr int VW = TR::VW;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RowsSmem& sm = *reinterpret_cast<RowsSmem*>(smem_raw);

  const int tid = threadIdx.x;
  const int G1 = p.gamma + 1;
  const int s = blockIdx.x % p.S;
  const int r = blockIdx.x / p.S;
  const int b = r / G1;
  const int i = r - b * G1;

  pdl_launch_dependents();
  if (MODE != MODE_TOPK) {
    // the sequence finisher needs the drafts and uniforms; fetch them with the data
    if (tid < p.gamma) sm.dr[tid] = p.draft[b * p.gamma + tid];
    if (MODE == MODE_SOFTMAX && tid < G1) sm.ur[tid] = p.uniforms[b * G1 + tid];
  }

  const T* row = static_cast<const T*>(p.logits) + (size_t)r * p.V;
  const int s0 = s * p.SL;
  const int s1 = min(s0 + p.SL, p.V);
  const bool vec_ok = (p.V % VW) == 0;

  // the whole slice goes to registers first: U 16-byte loads in flight per thread
  uint4 buf[kMaxU];
#pragma unroll
  for (int j = 0; j < kMaxU; ++j) {
    buf[j] = make_uint4(TR::kPadWord, TR::kPadWord, TR::kPadWord, TR::kPadWord);
    if (j < p.U) {
      const int e0 = s0 + (j * kThreads + tid) * VW;
      const int nv = min(max(s1 - e0, 0), VW);
      if (nv > 0) buf[j] = load_slot<T>(row, e0, nv, vec_ok);
    }
  }

  if (MODE == MODE_GREEDY) {
    // thread max (NaN propagates), the first slot holding it, its first element
    float tmax = -INFINITY;
    int tslot = -1;
#pragma unroll
    for (int j = 0; j < kMaxU; ++j) {
      if (j < p.U && s0 + (j * kThreads + tid) * VW < s1) {
        const float m = TR::template vmax<true>(buf[j]);
        if (tslot < 0 || argmax_better(m, 1, tmax, 0)) { tmax = m; tslot = j; }  // equal: keep the earlier slot
      }
    }
    int tidx = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kMaxU; ++j) {
      if (j == tslot) {
        const int e0 = s0 + (j * kThreads + tid) * VW;
        const int nv = min(s1 - e0, VW);
#pragma unroll
        for (int t = VW - 1; t >= 0; --t) {
          const float x = TR::get(buf[j], t);
          const bool hit = (tmax != tmax) ? (x != x) : (x == tmax);
          if (t < nv && hit) tidx = e0 + t;
        }
      }
    }
    if (tslot < 0) tmax = -INFINITY;
    // block argmax
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, tmax, m);
      const int oi = __shfl_xor_sync(0xffffffffu, tidx, m);
      if (argmax_better(ov, oi, tmax, tidx)) { tmax = ov; tidx = oi; }
    }
    if (lane == 0) sm.pair[warp] = make_float2(tmax, __int_as_float(tidx));
    __syncthreads();
    if (tid == 0) {
      float bv = sm.pair[0].x;
      int bi = __float_as_int(sm.pair[0].y);
      for (int w = 1; w < kWarps; ++w) {
        const float ov = sm.pair[w].x;
        const int oi = __float_as_int(sm.pair[w].y);
        if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      p.part[(size_t)r * p.S + s] = make_float4(bv, __int_as_float(bi), 0.f, 0.f);
    }
    if (arrive_last(p.seq_ticket + b, p.S * G1, &sm.flag, true)) finish_sequence_dense<T, MODE>(p, b, sm);
    return;
  }

  if (MODE == MODE_SOFTMAX) {
    // slice max, then sum of 2^((x - M) c) over the registers
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxU; ++j)
      if (j < p.U) tmax = fmaxf(tmax, TR::template vmax<false>(buf[j]));
    const float M = block_max(tmax, sm.fred);
    float a0 = 0.f, a1 = 0.f;
    if (M > -INFINITY) {
      const float Mc = M * p.c;
#pragma unroll
      for (int j = 0; j < kMaxU; ++j) {
        if (j < p.U) {
#pragma unroll
          for (int t = 0; t < VW; t += 2) {
            a0 += ex2_approx(fmaf(TR::get(buf[j], t), p.c, -Mc));
            a1 += ex2_approx(fmaf(TR::get(buf[j], t + 1), p.c, -Mc));
          }
        }
      }
    }
    F2 tot = block_sum_f2(F2{a0 + a1, 0.f}, sm.f2red);
    if (tid == 0) p.part[(size_t)r * p.S + s] = make_float4(M, tot.hi, tot.lo, 0.f);
    if (arrive_last(p.seq_ticket + b, p.S * G1, &sm.flag, true)) finish_sequence_dense<T, MODE>(p, b, sm);
    return;
  }

  // ---------------------------------------------------------------- top-k mode
  const int k = p.top_k;
  float tmax = -INFINITY;
  int has_nan = 0, nreal = 0;
#pragma unroll
  for (int j = 0; j < kMaxU; ++j) {
    if (j < p.U) {
      const int e0 = s0 + (j * kThreads + tid) * VW;
      const int nv = min(max(s1 - e0, 0), VW);
#pragma unroll
      for (int t = 0; t < VW; ++t) {
        if (t < nv) {
          const float x = TR::get(buf[j], t);
          if (x != x) has_nan = 1;
          else { tmax = fmaxf(tmax, x); ++nreal; }
        }
      }
    }
  }
  if (tid == 0) sm.count = 0;
  if (__syncthreads_or(has_nan) && tid == 0 && i <= seq_gamma(p, b)) atomicOr(&p.seq[b].status, SEQ_BADROW);
  const int total_real = block_sum_int(nreal, sm.ired);
  // threshold key K: the k-th largest of the per-thread maxima (a lower bound
  // of the slice's k-th largest value: those k threads each hold one element >= it)
  const uint32_t tkey = nreal > 0 ? okey(tmax) : 0u;
  uint32_t K = 0u;
  if (total_real > k) {
    for (int bit = 31; bit >= TR::KEY_LOW_BIT; --bit) {
      const uint32_t Kt = K | (1u << bit);
      if (__syncthreads_count(tkey >= Kt) >= k) K = Kt;
    }
  }
  // collect the candidates (value key >= K) into shared memory
  auto collect = [&](auto pred) {
    int mine = 0;
#pragma unroll
    for (int j = 0; j < kMaxU; ++j) {
      if (j < p.U) {
        const int e0 = s0 + (j * kThreads + tid) * VW;
        const int nv = min(max(s1 - e0, 0), VW);
#pragma unroll
        for (int t = 0; t < VW; ++t) {
          const float x = TR::get(buf[j], t);
          if (t < nv && x == x && pred(x, e0 + t)) ++mine;
        }
      }
    }
    const int lane = tid & 31;
    int inc = mine;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, m);
      if (lane >= m) inc += o;
    }
    int base = 0;
    if (lane == 31) base = atomicAdd(&sm.count, inc);
    base = __shfl_sync(0xffffffffu, base, 31);
    int pos = base + inc - mine;
#pragma unroll
    for (int j = 0; j < kMaxU; ++j) {
      if (j < p.U) {
        const int e0 = s0 + (j * kThreads + tid) * VW;
        const int nv = min(max(s1 - e0, 0), VW);
#pragma unroll
        for (int t = 0; t < VW; ++t) {
          const float x = TR::get(buf[j], t);
          if (t < nv && x == x && pred(x, e0 + t)) {
            if (pos < kCandCap) sm.cand[pos] = comp_key(x, e0 + t);
            ++pos;
          }
        }
      }
    }
    __syncthreads();
    return sm.count;
  };
  int N = collect([&](float x, int) { return okey(x) >= K; });
  if (N > kCandCap) {
    // too many ties / too large k: find the exact k-th largest composite key by
    // bisection over the slice held in registers, then collect exactly k
    unsigned long long K64 = 0ull;
    for (int bit = 63; bit >= 0; --bit) {
      const unsigned long long Kt = K64 | (1ull << bit);
      int mine = 0;
#pragma unroll
      for (int j = 0; j < kMaxU; ++j) {
        if (j < p.U) {
          const int e0 = s0 + (j * kThreads + tid) * VW;
          const int nv = min(max(s1 - e0, 0), VW);
#pragma unroll
          for (int t = 0; t < VW; ++t) {
            const float x = TR::get(buf[j], t);
            if (t < nv && x == x && comp_key(x, e0 + t) >= Kt) ++mine;
          }
        }
      }
      if (block_sum_int(mine, sm.ired) >= k) K64 = Kt;
    }
    __syncthreads();
    if (tid == 0) sm.count = 0;
    __syncthreads();
    N = collect([&](float x, int e) { return comp_key(x, e) >= K64; });
  }
  // rank-select the slice's top-k, written in descending order
  const int kk = min(k, N);
  unsigned long long* list = p.lists + ((size_t)r * p.S + s) * k;
  for (int e = tid; e < N; e += kThreads) {
    const unsigned long long me = sm.cand[e];
    int rank = 0;
    for (int j = 0; j < N; ++j) rank += sm.cand[j] > me;
    if (rank < kk) list[rank] = me;
  }
  for (int e = kk + tid; e < k; e += kThreads) list[e] = 0ull;
  if (!arrive_last(p.row_ticket + r, p.S, &sm.flag)) return;
  finish_row_topk(p, b, i, r, sm);
  if (!arrive_last(p.seq_ticket + b, G1, &sm.flag)) return;
  finish_sequence_topk(p, b, sm);
}

// Three two-float sums reduced together.
struct F2x3 {
  F2 a, b, c;
};

// Block-wide F2x3 sum (one pair of barriers), valid in the lanes of warp 0
// only (the callers need the total in one thread or in warp 0): the per-warp
// totals are combined by warp 0 in a shuffle tree instead of by every thread.
__device__ __forceinline__ F2x3 block_sum_f2x3_w0(F2x3 v, F2x3* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    v.a = f2_add(v.a, f2_shfl_xor(v.a, m));
    v.b = f2_add(v.b, f2_shfl_xor(v.b, m));
    v.c = f2_add(v.c, f2_shfl_xor(v.c, m));
  }
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  F2x3 t{F2{0.f, 0.f}, F2{0.f, 0.f}, F2{0.f, 0.f}};
  if (warp == 0) {
    if (lane < nw) t = sm[lane];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      if (m < nw) {   // block-uniform: a tree over the first (power of two >= nw) lanes
        t.a = f2_add(t.a, f2_shfl_xor(t.a, m));
        t.b = f2_add(t.b, f2_shfl_xor(t.b, m));
        t.c = f2_add(t.c, f2_shfl_xor(t.c, m));
      }
    }
    // lanes 0 .. (power of two >= nw) - 1 hold the total: give it to all 32
    t.a = F2{__shfl_sync(0xffffffffu, t.a.hi, 0), __shfl_sync(0xffffffffu, t.a.lo, 0)};
    t.b = F2{__shfl_sync(0xffffffffu, t.b.hi, 0), __shfl_sync(0xffffffffu, t.b.lo, 0)};
    t.c = F2{__shfl_sync(0xffffffffu, t.c.hi, 0), __shfl_sync(0xffffffffu, t.c.lo, 0)};
  }
  return t;
}

// ------------------------------------------------------------------ final draw
//
// The cluster kernel's final draw gives each thread a run of consecutive
// tokens, so its inverse-CDF search goes CTA slice -> thread -> token, every
// level contiguous in token order (the grid path's, in sv_final.cuh, goes
// item -> 4-token group -> token).
//
// Precision.  This is the one row per sequence whose inverse CDF is compared
// step by step with a float64 reference over up to ~10^5 steps.  A token's
// weight 2^((x - M) c) takes its exponent in two-float; the tokens within
// 2^-8 of the row maximum (they carry most of the mass, so their rounding
// would shift every later CDF step) get the two-float exp2, the rest
// ex2.approx with a first-order correction for the exponent's low part; all
// running sums are two-float (RunAcc).  The residual max(p - q, 0) = max(w - s q, 0) / s is kept
// unnormalised (the inverse CDF does not change under scaling).  Each
// sub-range reports (S, A, Q) - the sum of its weights, and over its residual
// support {w > s' q} (s' the row-statistics kernel's float normaliser) the sum
// of w - s' q and of q.  The finisher forms the exact normaliser s = sum S and
// the masses A - (s - s') Q: no second pass, and no cancellation, since
// s - s' is tiny.  Tokens whose support membership s' and s would decide
// differently have |w - s q| < 1e-6 w and contribute nothing measurable.

// (S, A, Q) of one thread's run (see "Precision" above), two-float with the
// error of every addition collected in the low words.
struct RunAcc {
  float sh, sl, ah, al, q;
  __device__ __forceinline__ void zero() { sh = sl = ah = al = q = 0.f; }
  __device__ static __forceinline__ void acc2(float& h, float& l, float x, float xl) {
    const float s = h + x;
    const float bb = s - h;
    l += ((h - (s - bb)) + (x - bb)) + xl;
    h = s;
  }
  // a weight near the maximum (two-float), its residual formed exactly
  __device__ __forceinline__ void add(F2 w, float qv, bool use_q, float s_a) {
    acc2(sh, sl, w.hi, w.lo);
    if (use_q) {
      const float pr = s_a * qv;
      if (w.hi > pr) {
        const float pe = fmaf(s_a, qv, -pr);
        const float dh = w.hi - pr;
        const float bb = dh - w.hi;
        const float de = (w.hi - (dh - bb)) + (-pr - bb);
        acc2(ah, al, dh, de + (w.lo - pe));
        q += qv;
      }
    }
  }
  __device__ __forceinline__ F2 S() const { return f2_norm(sh, sl); }
  __device__ __forceinline__ F2 A() const { return f2_norm(ah, al); }
  __device__ __forceinline__ F2 mass(bool resid, F2 ds) const {
    return resid ? f2_add(A(), f2_neg(f2_scale(ds, q))) : S();
  }
};

// The exponent (x - M) c of one token as p + e: x - M is exact for 16-bit
// logits (EXACT_DIFF); for float32 its rounding error is kept (two-diff).  A
// weight whose p is not above -1e30 (x = -inf, or an exponent that overflows)
// is 0.
template <bool EXACT_DIFF>
__device__ __forceinline__ float tok_exponent(float x, float M, float c, float c_lo, float* e_out) {
  const float dh = x - M;
  const float p = dh * c;
  float e = fmaf(dh, c, -p);
  e = fmaf(dh, c_lo, e);
  if (!EXACT_DIFF) {
    const float bb = dh - x;
    const float dl = (x - (dh - bb)) + (-M - bb);   // x - M = dh + dl exactly
    e = fmaf(dl, c, e);
  }
  *e_out = e;
  return p;
}

// One token of the final-draw row: a tail token (p <= -8) is added here
// (weight ex2.approx(p) with a first-order correction for e - on this range
// ex2.approx.ftz.f32 and exp2f agree - and its residual w - s' q with one
// rounding) and run_tail returns false; a token near the maximum is left to
// run_top (two-float exp2, exact residual) and run_tail returns true.
template <bool EXACT_DIFF, bool USE_Q>
__device__ __forceinline__ bool run_tail_t(RunAcc& acc, float x, float qv, float M, float c, float c_lo, float s_a) {
  float e;
  const float p = tok_exponent<EXACT_DIFF>(x, M, c, c_lo, &e);
  const bool top = p > -8.f;
  const float y = ex2_approx(p);   // results below 2^-126 flush to 0
  const float w = (top || !(p > -1e30f)) ? 0.f : fmaf(y * 6.931471825e-01f, e, y);
  RunAcc::acc2(acc.sh, acc.sl, w, 0.f);
  if (USE_Q) {
    // on the residual support {w > s' q}: w - s' q, rounded once (its sign
    // is the exact difference's sign), and q
    const float d = fmaf(-s_a, qv, w);
    if (d > 0.f) {
      RunAcc::acc2(acc.ah, acc.al, d, 0.f);
      acc.q += qv;
    }
  }
  return top;
}
template <bool EXACT_DIFF>
__device__ __forceinline__ bool run_tail(RunAcc& acc, float x, float qv, bool use_q, float M, float c, float c_lo,
                                         float s_a) {
  return use_q ? run_tail_t<EXACT_DIFF, true>(acc, x, qv, M, c, c_lo, s_a)
               : run_tail_t<EXACT_DIFF, false>(acc, x, qv, M, c, c_lo, s_a);
}
template <bool EXACT_DIFF>
__device__ __forceinline__ void run_top(RunAcc& acc, float x, float qv, bool use_q, float M, float c, float c_lo,
                                        float s_a, const float* tab) {
  float e;
  const float p = tok_exponent<EXACT_DIFF>(x, M, c, c_lo, &e);
  acc.add(exp2_f2(f2_norm(p, e), tab), qv, use_q, s_a);
}

// One token's increment of the walked mass, with the run's arithmetic: the
// weight w (bonus / fallback to p) or, on the residual support {w > s' q},
// w - s' q - (s - s') q.
template <bool EXACT_DIFF>
__device__ __forceinline__ F2 token_mass(float x, float qv, bool use_q, float M, float c, float c_lo, float s_a,
                                         F2 ds, const float* tab) {
  RunAcc one;
  one.zero();
  if (run_tail<EXACT_DIFF>(one, x, qv, use_q, M, c, c_lo, s_a))
    run_top<EXACT_DIFF>(one, x, qv, use_q, M, c, c_lo, s_a, tab);
  F2 m = one.mass(use_q, ds);
  if (m.hi < 0.f) m = F2{0.f, 0.f};
  return m;
}

// ---- streaming-path row statistics
// The streaming kernel leaves one partial per row segment (the part of a row
// one CTA streamed): slot row * H + h holds (max, first index) of the
// segment (greedy) or (max M_h, sum of 2^((L - M_h) c) as two floats)
// (sampling); slots past the row's last segment stay empty (seg_valid).  A
// row's NP = H slots are contiguous, so sequence b's G1 rows occupy slots
// [b * G1 * NP, (b + 1) * G1 * NP).  NP (1, 2 or 4) divides 32: one aligned
// lane segment merges one row.
__device__ __forceinline__ int stream_np(const Params& p) { return p.H; }

// The CTA holding vector x of the flattened space: the largest j with
// start(j) <= x.
__device__ __forceinline__ int seg_cta(long long x, long long NVT, int grid) {
  return (int)(((x + 1) * (long long)grid - 1) / NVT);
}
// Valid partial slot `seg` of row r (segments past the row's last CTA stay
// empty): the merges skip the others.
__device__ __forceinline__ bool seg_valid(const Params& p, long long r, int seg) {
  const long long NV = p.V / p.VWs;
  const long long NVT = p.NVT;
  return seg < seg_cta((r + 1) * NV - 1, NVT, p.SG) - seg_cta(r * NV, NVT, p.SG) + 1;
}


// base: the first of the nrow rows' partial slots (sequence b's rows are
// contiguous).  sBad[i] = the row defines no distribution (greedy: a NaN), for
// i <= gb only when mask_gb.
template <int MODE>
__device__ __forceinline__ void merge_row_parts_at(const Params& p, const float4* base, long long r0, int G1, int gb,
                                                   bool mask_gb, float* sM, double* sS, int* sG, int* sBad) {
  const int NP = stream_np(p);
  const int E = G1 * NP;
  for (int e0 = 0; e0 < E; e0 += kThreads) {        // uniform over the block: every lane shuffles
    const int e = e0 + (int)threadIdx.x;
    const bool ok = e < E && seg_valid(p, r0 + e / NP, e % NP);
    const float4 v = ok ? __ldcg(base + e) : make_float4(-INFINITY, __int_as_float(0x7fffffff), 0.f, 0.f);
    const bool head = ok && (e % NP) == 0;
    const int i = e / NP;
    if (MODE == MODE_GREEDY) {
      float bv = v.x;
      int bi = __float_as_int(v.y);
      for (int o = NP >> 1; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (argmax_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (head) {
        const bool nan = bv != bv;
        sG[i] = (nan || bi == 0x7fffffff) ? 0 : bi;
        sBad[i] = nan && (!mask_gb || i <= gb);
      }
    } else {
      float M = v.x;
      for (int o = NP >> 1; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      F2 t{0.f, 0.f};
      if (ok && v.x > -INFINITY && M < INFINITY) {
        const float sc = ex2_approx((v.x - M) * p.c);
        t = f2_add(F2{v.y * sc, 0.f}, F2{v.z * sc, 0.f});
      }
      for (int o = NP >> 1; o >= 1; o >>= 1) t = f2_add(t, f2_shfl_xor(t, o));
      if (head) {
        const double sum = (double)t.hi + (double)t.lo;
        sM[i] = M;
        sS[i] = sum;
        sBad[i] = (!(M > -INFINITY && M < INFINITY) || !(sum > 0.0 && sum < 1e300)) && (!mask_gb || i <= gb);
      }
    }
  }
}
template <int MODE>
__device__ __forceinline__ void merge_row_parts(const Params& p, int b, int G1, int gb, float* sM, double* sS,
                                                int* sG, int* sBad) {
  merge_row_parts_at<MODE>(p, p.part + (size_t)b * G1 * stream_np(p), (long long)b * G1, G1, gb, true, sM, sS, sG,
                           sBad);
}


// Warp 0: the first i < count with flags[i] != 0 (count if none), and
// whether any flag2[i] is set for i <= last.
__device__ __forceinline__ int first_flag_w0(const int* flags, int count, const int* flag2, int last, bool* any2) {
  const int lane = threadIdx.x & 31;
  int first = count;
  bool a2 = false;
  for (int k = 0; k <= last; k += 32) {
    const int i = k + lane;
    const unsigned hit = __ballot_sync(0xffffffffu, i < count && flags[i] != 0);
    if (hit && first == count) first = k + __ffs(hit) - 1;
    a2 |= __any_sync(0xffffffffu, i <= last && flag2[i] != 0);
  }
  *any2 = a2;
  return first;
}

}  // namespace sv
