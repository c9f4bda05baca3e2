// Host side of libspecverify: argument validation, workspace layout and kernel
// dispatch for the C ABI declared in include/specverify.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdint>

#include <cstdlib>
#include <cstring>
#include <string>

#include "specverify.h"
#include "sv_cluster.cuh"
#include "sv_device.cuh"
#include "sv_final.cuh"
#include "sv_qsoftmax.cuh"
#include "sv_topp.cuh"
#include "sv_stream.cuh"
#include "sv_truncate.cuh"
#include "sv_topk.cuh"
#include "sv_shard.cuh"

namespace {

// sv_set_timing_events registration (benchmark hook)
cudaEvent_t g_timing[3] = {nullptr, nullptr, nullptr};
bool g_timing_on = false;

void timing_record(int which, cudaStream_t stream) {
  if (g_timing_on) cudaEventRecord(g_timing[which], stream);
}

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Length of the top-k candidate lists the workspace reserves for (top_k, V):
// top_k itself, or the whole vocabulary when top-p alone is allowed (V <= 1024).
int list_len(int V, int top_k) {
  if (top_k > 0) return top_k < V ? top_k : V;
  return V <= SV_MAX_TOP_K ? V : 0;
}

struct Layout {
  size_t seq_ticket, seq_ticket2, row_ticket, ctr, seq, acc, part, lists, rowres, fd_part, fd_q, tp, total;
  int S_part, S_list, FC, klist;
};

// One layout for any dtype and launch shape: slices are sized for the
// smallest slice the dispatcher may pick (float32, one vector per thread) and
// chunks for the smallest chunk (8 elements per thread).
Layout make_layout(int B, int gamma, int V, int top_k) {
  Layout L{};
  const long long R = (long long)B * (gamma + 1);
  L.klist = list_len(V, top_k);
  L.S_part = (int)ceil_div(V, sv::kThreads * 1 * 4);
  L.S_list = L.klist > 0 ? (int)ceil_div(V, sv::kThreads * sv::kMaxU * 4) : 0;
  // final draw: 512-token items per row
  L.FC = (int)ceil_div(V, sv::kFdTok);
  size_t o = 0;
  L.seq_ticket = o;  o += up(sizeof(int) * (size_t)B);
  L.seq_ticket2 = o; o += up(sizeof(int) * (size_t)B);
  L.row_ticket = o;  o += up(sizeof(int) * (size_t)R);
  L.ctr = o;         o += up(sizeof(int) * 4);
  L.seq = o;         o += up(sizeof(sv::SeqState) * (size_t)B);
  L.acc = o;         o += up(sizeof(double) * (size_t)B * gamma);
  // rows path: S_part slice partials per row; streaming path: up to 4 parts x
  // 8 warps per row
  L.part = o;        o += up(sizeof(float4) * (size_t)R * std::max(L.S_part, 4 * sv::kWarps));
  L.lists = o;       o += up(sizeof(unsigned long long) * (size_t)R * L.S_list * L.klist);
  L.rowres = o;      o += up(L.klist > 0 ? sizeof(int2) * (size_t)R * (L.klist + 1) : 0);
  L.fd_part = o;     o += up(sizeof(float4) * (size_t)B * L.FC);
  L.fd_q = o;        o += up(sizeof(float) * (size_t)B * L.FC);
  L.tp = o;          o += up(sizeof(sv::TpRow) * (size_t)R);
  L.total = o;
  return L;
}

bool sizes_ok(int B, int gamma, int V) {
  return B >= 0 && gamma >= 0 && gamma <= SV_MAX_GAMMA && V >= 1 && V <= SV_MAX_VOCAB &&
         (long long)B * (gamma + 1) <= (1ll << 24);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

int vec_width(sv_dtype dt) { return dt == SV_DTYPE_F32 ? 4 : 8; }

// Carve the workspace and fill the pointer fields of p.
void bind_workspace(sv::Params& p, const Layout& L, void* ws) {
  unsigned char* w = static_cast<unsigned char*>(ws);
  p.seq_ticket = reinterpret_cast<int*>(w + L.seq_ticket);
  p.seq_ticket2 = reinterpret_cast<int*>(w + L.seq_ticket2);
  p.row_ticket = reinterpret_cast<int*>(w + L.row_ticket);
  p.ctr = reinterpret_cast<int*>(w + L.ctr);
  p.seq = reinterpret_cast<sv::SeqState*>(w + L.seq);
  p.acc = reinterpret_cast<double*>(w + L.acc);
  p.part = reinterpret_cast<float4*>(w + L.part);
  p.lists = reinterpret_cast<unsigned long long*>(w + L.lists);
  p.rowres = reinterpret_cast<int2*>(w + L.rowres);
  p.fd_part = reinterpret_cast<float4*>(w + L.fd_part);
  p.fd_q = reinterpret_cast<float*>(w + L.fd_q);
  p.FC = L.FC;
  p.tp = reinterpret_cast<sv::TpRow*>(w + L.tp);
}

// Rows-kernel slicing: 8 vectors per thread unless that leaves fewer than two
// CTAs per SM, in which case the slices shrink (latency-bound small batches).
void choose_slices(sv::Params& p, sv_dtype dt, bool topk) {
  const int VW = vec_width(dt);
  const long long R = (long long)p.B * (p.gamma + 1);
  int U = sv::kMaxU;
  if (!topk) {
    const long long want = 2ll * sm_count();
    while (U > 1 && R * ceil_div(p.V, (long long)sv::kThreads * U * VW) < want) U >>= 1;
  }
  p.U = U;
  p.SL = sv::kThreads * U * VW;
  p.S = (int)ceil_div(p.V, p.SL);
}

template <typename T, int MODE>
sv_status launch_rows(const sv::Params& p, cudaStream_t stream) {
  const size_t smem = MODE == sv::MODE_TOPK ? sizeof(sv::RowsSmem) : offsetof(sv::RowsSmem, cand);
  auto kern = sv::rows_kernel<T, MODE>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return SV_ERR_CUDA;
  const long long grid = (long long)p.B * (p.gamma + 1) * p.S;
  kern<<<(unsigned)grid, sv::kThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Programmatic dependent launch of `kern` after the previous kernel on the stream.
template <typename K>
sv_status launch_pdl(K kern, dim3 grid, dim3 block, size_t smem, const sv::Params& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// The final draw: Z CTAs per sequence (one part of row n each; persistent
// when the units exceed the CTAs that fit), the last part's CTA searches.
template <typename T, bool MASK = false>
sv_status launch_final_draw(const sv::Params& p, cudaStream_t stream) {
  auto kern = sv::final_draw_kernel<T, MASK>;
  // the ring; the search stages a sequence's item sums (float4 + float each) in it
  const size_t smem = std::max(sv::FdRing<T>::bytes, sv::fd_stash_bytes(p.FC));
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, sv::kFdThreads, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  // parts per sequence: the B * Z units fill the CTA slots once (at most one
  // part per 4 items)
  const long long slots = (long long)per_sm * sm_count();
  sv::Params q = p;
  q.FZ = (int)std::max(1ll, std::min(slots / std::max(1, p.B), ceil_div(p.FC, 4)));
  const long long grid = std::max(1ll, std::min(slots, (long long)p.B * q.FZ));
  return launch_pdl(kern, dim3((unsigned)grid), dim3(sv::kFdThreads), smem, q, stream);
}

// ---------------------------------------------------------------- cluster path
// Small problems run as one kernel with one thread-block cluster per sequence
// (sv_cluster.cuh).  SPECVERIFY_PATH=grid / =cluster overrides the choice
// (tests use it to cover both paths).
constexpr size_t kClusterMaxBytes = 8u << 20;      // logits of the whole batch
constexpr size_t kClusterBytesPerCta = 16u << 10;  // slice bytes a CTA aims for
constexpr size_t kClusterMaxSmem = 200u << 10;

int path_override() {
  const char* e = std::getenv("SPECVERIFY_PATH");
  if (!e) return 0;
  if (!std::strcmp(e, "grid")) return 1;
  if (!std::strcmp(e, "cluster")) return 2;
  if (!std::strcmp(e, "slices")) return 3;   // top-k: the per-slice kernel instead of the per-row one
  if (!std::strcmp(e, "topp")) return 4;     // top-p alone: the per-row threshold path at any V
  if (!std::strcmp(e, "topprow")) return 5;  // top-p alone, threshold path, and one CTA per row (no cluster)
  return 0;
}

bool plan_cluster(const sv::Params& p, sv_dtype dt, int mode, sv::ClusterParams* cp, size_t* smem) {
  if (mode == sv::MODE_TOPK || mode == sv::MODE_TOPP || p.ql) return false;   // q from draft logits: the streaming path
  const int ov = path_override();
  if (ov == 1) return false;
  const int VW = vec_width(dt);
  const size_t sl = dt == SV_DTYPE_F32 ? 4 : 2;
  if (p.V % VW != 0) return false;
  const size_t G1 = (size_t)p.gamma + 1;
  const bool qrows = mode == sv::MODE_SOFTMAX && p.q != nullptr;   // q rows staged in shared memory
  const size_t per_seq = G1 * p.V * sl + (qrows ? (size_t)p.gamma * p.V * 4 : 0);
  if (ov != 2 && (size_t)p.B * G1 * p.V * sl > kClusterMaxBytes) return false;
  int CN = (int)std::min<size_t>(sv::kClusterMax, std::max<size_t>(1, (per_seq + kClusterBytesPerCta - 1) / kClusterBytesPerCta));
  int W = (int)ceil_div(p.V, CN);
  W = (W + 7) / 8 * 8;
  CN = (int)ceil_div(p.V, W);
  const int NS = (int)ceil_div(W / VW, sv::kThreads);
  if (NS > sv::kClusterMaxNS) return false;
  const size_t sm = ((sizeof(sv::ClusterSmem) + 15) & ~size_t(15)) + G1 * W * sl +
                    (qrows ? (size_t)p.gamma * W * 4 : 0);
  if (sm > kClusterMaxSmem) return false;
  cp->p = p;
  cp->CN = CN;
  cp->W = W;
  cp->NS = NS;
  cp->EPT = NS * VW;
  *smem = sm;
  return true;
}

template <typename T, int MODE>
sv_status launch_cluster(const sv::ClusterParams& cp, size_t smem, cudaStream_t stream, bool* launched) {
  auto kern = sv::cluster_kernel<T, MODE>;
  *launched = false;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      (cp.CN > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    cudaGetLastError();
    return SV_OK;   // not available: the caller takes the grid path
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(cp.p.B * cp.CN));
  cfg.blockDim = dim3(sv::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cp.CN;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess || nclusters < 1) {
    cudaGetLastError();
    return SV_OK;
  }
  if (cudaLaunchKernelEx(&cfg, kern, cp) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  *launched = true;
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Streaming kernels (sv_stream.cuh): persistent CTAs, balanced row counts.
template <typename K>
long long stream_grid(K kern, size_t smem, long long R) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, sv::kSt, smem) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const long long slots = (long long)per_sm * sm_count();
  const long long per = ceil_div(R, std::min(R, slots));
  return ceil_div(R, per);
}

template <typename T>
sv_status launch_stream_topk(const sv::Params& p, cudaStream_t stream) {
  auto kern = sv::stream_topk_kernel<T>;
  const size_t smem = (size_t)sv::kStSTopk * sv::kStUTopk * sv::kSt * sizeof(uint4) + sizeof(sv::TopkSmem);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  // target rows, then (q formed from the draft's logits) the draft rows
  const long long R = (long long)p.B * (p.gamma + 1) + (p.ql ? (long long)p.B * p.gamma : 0);
  // rows of more than kStSTopk ring chunks are claimed at run time (the
  // kernel makes the same test): then one CTA per slot; else equal static shares
  const long long nch = ceil_div((long long)(p.V / (sizeof(T) == 4 ? 4 : 8)), (long long)sv::kStUTopk * sv::kSt);
  long long grid;
  if (nch > sv::kStSTopk) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, sv::kSt, smem) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    grid = std::min(R, (long long)per_sm * sm_count());
  } else {
    grid = stream_grid(kern, smem, R);
  }
  kern<<<(unsigned)grid, sv::kSt, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Dense streaming kernel: every CTA streams the same number of vectors (the
// flattened rows split evenly, sv_stream.cuh).  Sets p.SG (the grid), p.NVT,
// p.VWs and p.H (partial slots per row: a power of two at least the number of
// CTAs that can share a row), which the kernels that merge the partials read.
template <typename T, int MODE>
sv_status launch_stream_dense(sv::Params& p, cudaStream_t stream) {
  auto kern = sv::stream_dense_kernel<T, MODE>;
  const size_t smem = (size_t)sv::kStS * sv::kStU * sv::kSt * sizeof(uint4) + sizeof(sv::StreamSmem);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  // rows streamed: the target's, then (q formed from the draft's logits) the draft's
  const long long R = (long long)p.B * (p.gamma + 1) + (p.ql ? (long long)p.B * p.gamma : 0);
  const int VW = sizeof(T) == 4 ? 4 : 8;
  const long long NV = p.V / VW;
  const long long NVT = R * NV;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, sv::kSt, smem) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const long long chunk = (long long)sv::kStU * sv::kSt;
  long long grid = std::min((long long)per_sm * sm_count(), ceil_div(NVT, chunk));
  // at most 4 CTAs share a row: every range at least ceil(NV / 3) vectors long
  grid = std::max(1ll, std::min(grid, NVT / ceil_div(NV, 3)));
  const long long L = NVT / grid;                       // shortest range
  const long long segs = ceil_div(NV, std::max(L, 1ll)) + 1;
  p.H = segs <= 1 ? 1 : (segs <= 2 ? 2 : 4);
  p.SG = (int)grid;
  p.NVT = NVT;
  p.VWs = VW;
  kern<<<(unsigned)grid, sv::kSt, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Greedy streaming path, second kernel: one CTA per sequence, launched as a
// programmatic dependent of the streaming kernel.
sv_status launch_greedy_finish(const sv::Params& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.B);
  cfg.blockDim = dim3(sv::kSt);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, sv::stream_greedy_finish_kernel, p) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return SV_OK;
}

// Kernels launched by the last call on this host thread (sv_last_kernels).
thread_local const char* g_last_kernels = "";

// Top-p alone with each row resident in a cluster's shared memory
// (topp_cluster_kernel): rows of whole 16-byte vectors, at most kTcMaxC
// slices of kTcSliceBytes.  *launched = false: not applicable here (the
// per-row kernel runs instead).
template <typename T>
sv_status launch_topp_cluster(const sv::Params& p, cudaStream_t stream, bool* launched) {
  *launched = false;
  const int VW = (int)(16 / sizeof(T));
  if (path_override() == 5 || p.V % VW != 0 || !aligned16(p.logits)) return SV_OK;
  const long long C = ceil_div((long long)p.V * (long long)sizeof(T), (long long)sv::kTcSliceBytes);
  if (C > sv::kTcMaxC) return SV_OK;
  const long long Vc = ceil_div(ceil_div((long long)p.V, C), (long long)VW) * VW;
  const size_t smem = sv::tc_head_bytes() + (size_t)Vc * sizeof(T);
  auto kern = sv::topp_cluster_kernel<T>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return SV_OK;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)p.B * (p.gamma + 1) * C));
  cfg.blockDim = dim3(sv::kTpThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess || nclusters < 1) {
    cudaGetLastError();
    return SV_OK;
  }
  if (cudaLaunchKernelEx(&cfg, kern, p, p.tp, (int)Vc) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  *launched = true;
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

template <typename T>
sv_status dispatch(sv::Params& p, int mode, cudaStream_t stream, sv_dtype dt) {
  sv::ClusterParams cp;
  size_t smem = 0;
  g_last_kernels = "";
  if (plan_cluster(p, dt, mode, &cp, &smem)) {
    bool launched = false;
    timing_record(0, stream);
    const sv_status st = mode == sv::MODE_GREEDY ? launch_cluster<T, sv::MODE_GREEDY>(cp, smem, stream, &launched)
                                                 : launch_cluster<T, sv::MODE_SOFTMAX>(cp, smem, stream, &launched);
    if (st != SV_OK) return st;
    if (launched) {
      g_last_kernels = "cluster_kernel";
      timing_record(1, stream);
      timing_record(2, stream);
      return SV_OK;
    }
  }
  timing_record(0, stream);
  sv_status st = SV_OK;
  if (mode == sv::MODE_TOPP) {
    // top-p alone: the rows' kept sets, then the final draw under the mask
    bool in_cluster = false;
    st = launch_topp_cluster<T>(p, stream, &in_cluster);
    if (st != SV_OK) return st;
    if (!in_cluster) {
      const size_t smem = sizeof(sv::TpSmem);
      auto tk = sv::topp_row_kernel<T>;
      if (cudaFuncSetAttribute(tk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
      }
      tk<<<(unsigned)((long long)p.B * (p.gamma + 1)), sv::kTpThreads, smem, stream>>>(p, p.tp);
      if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    }
    timing_record(1, stream);
    p.H = 0;
    st = launch_final_draw<T, true>(p, stream);
    timing_record(2, stream);
    g_last_kernels = st != SV_OK ? "" : (in_cluster ? "topp_cluster_kernel,final_draw_kernel"
                                                     : "topp_row_kernel,final_draw_kernel");
    return st;
  }
  const bool streamable = p.V % vec_width(dt) == 0 && path_override() != 3;
  if (mode == sv::MODE_GREEDY) {
    st = streamable ? launch_stream_dense<T, sv::MODE_GREEDY>(p, stream) : launch_rows<T, sv::MODE_GREEDY>(p, stream);
    g_last_kernels = streamable ? "stream_dense_kernel,stream_greedy_finish_kernel" : "rows_kernel";
  } else if (mode == sv::MODE_TOPK) {
    st = streamable ? launch_stream_topk<T>(p, stream) : launch_rows<T, sv::MODE_TOPK>(p, stream);
    g_last_kernels = streamable ? "stream_topk_kernel" : "rows_kernel";
  } else {
    st = streamable ? launch_stream_dense<T, sv::MODE_SOFTMAX>(p, stream) : launch_rows<T, sv::MODE_SOFTMAX>(p, stream);
    g_last_kernels = streamable ? "stream_dense_kernel,final_draw_kernel" : "rows_kernel,final_draw_kernel";
  }
  if (st != SV_OK) {
    g_last_kernels = "";
    return st;
  }
  timing_record(1, stream);
  if (mode == sv::MODE_SOFTMAX) {
    if (!streamable) p.H = 0;   // the rows kernel leaves merged statistics
    st = launch_final_draw<T>(p, stream);
  } else if (mode == sv::MODE_GREEDY && streamable) {
    st = launch_greedy_finish(p, stream);
  }
  timing_record(2, stream);
  return st;
}

sv_status run(sv::Params& p, sv_dtype dt, int mode, void* workspace, size_t workspace_bytes, int top_k_layout,
              cudaStream_t stream) {
  const Layout L = make_layout(p.B, p.gamma, p.V, top_k_layout);
  if (workspace == nullptr || workspace_bytes < L.total || !aligned16(workspace)) return SV_ERR_WORKSPACE;
  bind_workspace(p, L, workspace);
  choose_slices(p, dt, mode == sv::MODE_TOPK);
  switch (dt) {
    case SV_DTYPE_F32: return dispatch<float>(p, mode, stream, dt);
    case SV_DTYPE_BF16: return dispatch<__nv_bfloat16>(p, mode, stream, dt);
    case SV_DTYPE_F16: return dispatch<__half>(p, mode, stream, dt);
  }
  return SV_ERR_INVALID_ARG;
}

}  // namespace

extern "C" size_t sv_workspace_bytes(int B, int gamma, int V, int top_k) {
  if (!sizes_ok(B, gamma, V) || top_k < 0 || top_k > SV_MAX_TOP_K) return 0;
  return make_layout(B, gamma, V, top_k).total;
}

// sv_verify_sample_qlogits: the usual layout first (so a later call of any
// other entry point on the same workspace finds its part zero-filled), then
// the float32 q the transform kernel writes.
// + the kept-index lists of truncated draft rows ([B * gamma][klist] int).
size_t qlogits_list_bytes(int B, int gamma, int V, int top_k) {
  return up(sizeof(int) * (size_t)B * gamma * std::max(list_len(V, top_k), 1));
}
extern "C" size_t sv_qlogits_workspace_bytes(int B, int gamma, int V, int top_k) {
  if (!sizes_ok(B, gamma, V) || top_k < 0 || top_k > SV_MAX_TOP_K) return 0;
  return up(make_layout(B, gamma, V, top_k).total) + up(sizeof(float) * (size_t)B * gamma * V) +
         qlogits_list_bytes(B, gamma, V, top_k);
}

namespace {

sv_status verify_sample_impl(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype, const float* q,
                             const int32_t* draft_tokens, const float* uniforms, const int32_t* gamma_b,
                             float temperature, int top_k, float top_p, int32_t* out_tokens,
                             int32_t* out_num_accepted, float* out_accept_prob, int32_t* out_status, void* workspace,
                             size_t workspace_bytes, sv_stream_t stream, const void* ql = nullptr,
                             float4* qpart = nullptr, int2* qrowres = nullptr) {
  g_last_kernels = "";
  if (!sizes_ok(B, gamma, V)) return SV_ERR_INVALID_ARG;
  if (logits_dtype != SV_DTYPE_F32 && logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F16)
    return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (top_k < 0 || top_k > SV_MAX_TOP_K) return SV_ERR_INVALID_ARG;
  if (!(top_p > 0.0f && top_p <= 1.0f)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !uniforms || !out_tokens || !out_num_accepted) return SV_ERR_INVALID_ARG;
  if (gamma > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;   // q == NULL: deterministic drafts
  if (!aligned16(logits) || (q && !aligned16(q))) return SV_ERR_INVALID_ARG;

  // top-k below V (then top-p on its list): the candidate-list path.  top-p
  // without an effective top-k: the list path for V <= SV_MAX_TOP_K, else the
  // per-row threshold path (any V; q from draft logits excepted).
  const bool truncate = (top_k > 0 && top_k < V) || top_p < 1.0f;
  const bool topp_only = truncate && !(top_k > 0 && top_k < V);
  const bool topp_rows = topp_only && !ql && (V > SV_MAX_TOP_K || path_override() == 4);
  int klist = 0;
  if (truncate && !topp_rows) {
    klist = (top_k > 0 && top_k < V) ? top_k : V;
    if (klist > SV_MAX_TOP_K) return SV_ERR_UNSUPPORTED;
  }

  sv::Params p{};
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.top_k = klist;
  p.top_p = top_p;
  {
    const double c = 1.4426950408889634 / (double)temperature;
    p.c = (float)c;
    p.c_lo = (float)(c - (double)p.c);
  }
  p.logits = logits;
  p.q = q;
  p.draft = draft_tokens;
  p.uniforms = uniforms;
  p.gamma_b = gamma_b;
  p.ql = ql;
  p.qpart = qpart;
  p.qrowres = qrowres;
  p.out_tokens = out_tokens;
  p.out_n = out_num_accepted;
  p.out_a = out_accept_prob;
  p.out_status = out_status;
  // list_len(V, top_k) == klist whenever the list path runs
  const int mode = topp_rows ? sv::MODE_TOPP : (truncate ? sv::MODE_TOPK : sv::MODE_SOFTMAX);
  return run(p, logits_dtype, mode, workspace, workspace_bytes, top_k, reinterpret_cast<cudaStream_t>(stream));
}

sv_status verify_greedy_impl(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype,
                             const int32_t* draft_tokens, const int32_t* gamma_b, int32_t* out_tokens,
                             int32_t* out_num_accepted, int32_t* out_status, void* workspace, size_t workspace_bytes,
                             sv_stream_t stream) {
  g_last_kernels = "";
  if (!sizes_ok(B, gamma, V)) return SV_ERR_INVALID_ARG;
  if (logits_dtype != SV_DTYPE_F32 && logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F16)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !out_tokens || !out_num_accepted) return SV_ERR_INVALID_ARG;
  if (gamma > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;
  if (!aligned16(logits)) return SV_ERR_INVALID_ARG;
  sv::Params p{};
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.top_k = 0;
  p.top_p = 1.0f;
  p.c = 1.0f;
  p.logits = logits;
  p.draft = draft_tokens;
  p.gamma_b = gamma_b;
  p.out_tokens = out_tokens;
  p.out_n = out_num_accepted;
  p.out_status = out_status;
  return run(p, logits_dtype, sv::MODE_GREEDY, workspace, workspace_bytes, 0, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" sv_status sv_verify_sample(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype,
                                      const float* q, const int32_t* draft_tokens, const float* uniforms,
                                      float temperature, int top_k, float top_p, int32_t* out_tokens,
                                      int32_t* out_num_accepted, float* out_accept_prob, int32_t* out_status,
                                      void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  return verify_sample_impl(B, gamma, V, logits, logits_dtype, q, draft_tokens, uniforms, nullptr, temperature, top_k,
                            top_p, out_tokens, out_num_accepted, out_accept_prob, out_status, workspace,
                            workspace_bytes, stream);
}

extern "C" sv_status sv_verify_sample_ragged(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype,
                                             const float* q, const int32_t* draft_tokens, const float* uniforms,
                                             const int32_t* gamma_b, float temperature, int top_k, float top_p,
                                             int32_t* out_tokens, int32_t* out_num_accepted, float* out_accept_prob,
                                             int32_t* out_status, void* workspace, size_t workspace_bytes,
                                             sv_stream_t stream) {
  if (!gamma_b && B > 0) {
    g_last_kernels = "";
    return SV_ERR_INVALID_ARG;
  }
  return verify_sample_impl(B, gamma, V, logits, logits_dtype, q, draft_tokens, uniforms, gamma_b, temperature, top_k,
                            top_p, out_tokens, out_num_accepted, out_accept_prob, out_status, workspace,
                            workspace_bytes, stream);
}

namespace {
thread_local std::string g_qlogits_kernels;

template <typename TQ>
sv_status launch_q_softmax(const void* q_logits, float* q, int rows, int V, float c, float c_lo, int klist,
                           float top_p, int* kept_list, cudaStream_t st) {
  const TQ* src = static_cast<const TQ*>(q_logits);
  if (klist > 0) {   // truncation: top-k then top-p, the target's transform
    const bool vec = V % vec_width(std::is_same<TQ, float>::value ? SV_DTYPE_F32 : SV_DTYPE_BF16) == 0;
    auto kern = vec ? sv::q_truncate_kernel<TQ, true> : sv::q_truncate_kernel<TQ, false>;
    const int smem = (int)sizeof(sv::QtSmem);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return SV_ERR_CUDA;
    }
    kern<<<(unsigned)rows, sv::kQsThreads, smem, st>>>(src, q, V, klist, top_p, c, c_lo, kept_list);
  } else if (V % vec_width(std::is_same<TQ, float>::value ? SV_DTYPE_F32 : SV_DTYPE_BF16) == 0)
    sv::q_softmax_kernel<TQ, true><<<(unsigned)rows, sv::kQsThreads, 0, st>>>(src, q, V, c, c_lo);
  else
    sv::q_softmax_kernel<TQ, false><<<(unsigned)rows, sv::kQsThreads, 0, st>>>(src, q, V, c, c_lo);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
}  // namespace

extern "C" sv_status sv_verify_sample_qlogits(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype,
                                              const void* q_logits, sv_dtype q_logits_dtype,
                                              const int32_t* draft_tokens, const float* uniforms, float temperature,
                                              int top_k, float top_p, int32_t* out_tokens, int32_t* out_num_accepted,
                                              float* out_accept_prob, int32_t* out_status, void* workspace,
                                              size_t workspace_bytes, sv_stream_t stream) {
  g_last_kernels = "";
  if (!sizes_ok(B, gamma, V)) return SV_ERR_INVALID_ARG;
  auto dtype_ok = [](sv_dtype d) { return d == SV_DTYPE_F32 || d == SV_DTYPE_BF16 || d == SV_DTYPE_F16; };
  if (!dtype_ok(logits_dtype) || !dtype_ok(q_logits_dtype)) return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (top_k < 0 || top_k > SV_MAX_TOP_K) return SV_ERR_INVALID_ARG;
  if (!(top_p > 0.0f && top_p <= 1.0f)) return SV_ERR_INVALID_ARG;
  // truncation as in sv_verify_sample: k candidates at most SV_MAX_TOP_K
  const bool truncate = (top_k > 0 && top_k < V) || top_p < 1.0f;
  const int klist = truncate ? ((top_k > 0 && top_k < V) ? top_k : V) : 0;
  if (klist > SV_MAX_TOP_K) return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  if (!logits || !uniforms || !out_tokens || !out_num_accepted) return SV_ERR_INVALID_ARG;
  if (gamma > 0 && (!draft_tokens || !q_logits)) return SV_ERR_INVALID_ARG;
  if (!aligned16(logits) || (q_logits && !aligned16(q_logits))) return SV_ERR_INVALID_ARG;
  const size_t q_off = up(make_layout(B, gamma, V, top_k).total);
  const size_t q_bytes = up(sizeof(float) * (size_t)B * gamma * V);
  const size_t need = q_off + q_bytes + qlogits_list_bytes(B, gamma, V, top_k);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return SV_ERR_WORKSPACE;
  float* qbuf = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + q_off);
  int* klist_buf = reinterpret_cast<int*>(static_cast<unsigned char*>(workspace) + q_off + q_bytes);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // Fused: the streaming kernel also streams the draft rows (their maximum and
  // sum) and the final-draw kernel forms q from the draft's logits where it
  // needs it, so q is never written out.  Needs the streaming path (16-byte
  // vectors of one dtype on both sides); its draft-row partials (at most 4
  // parts x 8 warps per row) use the q scratch.
  const bool fused = gamma > 0 && !truncate && q_logits_dtype == logits_dtype && V % vec_width(logits_dtype) == 0 &&
                     path_override() != 3 && (size_t)V * sizeof(float) >= 4 * sv::kWarps * sizeof(float4);
  if (fused) {
    const sv_status s = verify_sample_impl(B, gamma, V, logits, logits_dtype, nullptr, draft_tokens, uniforms,
                                           nullptr, temperature, top_k, top_p, out_tokens, out_num_accepted,
                                           out_accept_prob, out_status, workspace, q_off, stream, q_logits,
                                           reinterpret_cast<float4*>(qbuf));
    return s;
  }
  // Truncated, fused: the streaming top-k kernel selects the draft rows like
  // the target rows and keeps their lists (in the q scratch), and the
  // sequence finisher reads q_i(d_i) and q(v) from them.  Needs the streaming
  // top-k path (16-byte vectors of one dtype) and room for the lists.
  const bool fused_topk = gamma > 0 && truncate && q_logits_dtype == logits_dtype &&
                          V % vec_width(logits_dtype) == 0 && path_override() != 3 &&
                          (size_t)V * sizeof(float) >= (size_t)(klist + 1) * sizeof(int2);
  if (fused_topk)
    return verify_sample_impl(B, gamma, V, logits, logits_dtype, nullptr, draft_tokens, uniforms, nullptr,
                              temperature, top_k, top_p, out_tokens, out_num_accepted, out_accept_prob, out_status,
                              workspace, q_off, stream, q_logits, nullptr, reinterpret_cast<int2*>(qbuf));
  if (gamma > 0) {
    const double cd = 1.4426950408889634 / (double)temperature;
    const float c = (float)cd, c_lo = (float)(cd - (double)c);
    const int rows = B * gamma;
    sv_status s = SV_OK;
    switch (q_logits_dtype) {
      case SV_DTYPE_F32: s = launch_q_softmax<float>(q_logits, qbuf, rows, V, c, c_lo, klist, top_p, klist_buf, st); break;
      case SV_DTYPE_BF16: s = launch_q_softmax<__nv_bfloat16>(q_logits, qbuf, rows, V, c, c_lo, klist, top_p, klist_buf, st); break;
      case SV_DTYPE_F16: s = launch_q_softmax<__half>(q_logits, qbuf, rows, V, c, c_lo, klist, top_p, klist_buf, st); break;
    }
    if (s != SV_OK) return s;
  }
  const sv_status s = verify_sample_impl(B, gamma, V, logits, logits_dtype, gamma > 0 ? qbuf : nullptr,
                                         draft_tokens, uniforms, nullptr, temperature, top_k, top_p, out_tokens,
                                         out_num_accepted, out_accept_prob, out_status, workspace, q_off, stream);
  if (s != SV_OK || gamma == 0) return s;
  // leave the q scratch zero-filled: the kept entries (truncated q) or all of it
  const char* first = klist > 0 ? "q_truncate_kernel," : "q_softmax_kernel,";
  const char* last = klist > 0 ? ",q_clear_kernel" : "";
  if (klist > 0) {
    sv::q_clear_kernel<<<(unsigned)(B * gamma), 256, 0, st>>>(qbuf, klist_buf, V, klist);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  } else if (cudaMemsetAsync(qbuf, 0, sizeof(float) * (size_t)B * gamma * V, st) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  g_qlogits_kernels = std::string(first) + g_last_kernels + last;
  g_last_kernels = g_qlogits_kernels.c_str();
  return s;
}

extern "C" sv_status sv_verify_greedy(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype,
                                      const int32_t* draft_tokens, int32_t* out_tokens, int32_t* out_num_accepted,
                                      int32_t* out_status, void* workspace, size_t workspace_bytes,
                                      sv_stream_t stream) {
  return verify_greedy_impl(B, gamma, V, logits, logits_dtype, draft_tokens, nullptr, out_tokens, out_num_accepted,
                            out_status, workspace, workspace_bytes, stream);
}

extern "C" sv_status sv_verify_greedy_ragged(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype,
                                             const int32_t* draft_tokens, const int32_t* gamma_b,
                                             int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_status,
                                             void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  if (!gamma_b && B > 0) {
    g_last_kernels = "";
    return SV_ERR_INVALID_ARG;
  }
  return verify_greedy_impl(B, gamma, V, logits, logits_dtype, draft_tokens, gamma_b, out_tokens, out_num_accepted,
                            out_status, workspace, workspace_bytes, stream);
}

extern "C" sv_status sv_truncate_emitted(int B, int gamma, int32_t* tokens, const int32_t* num_accepted,
                                         const int32_t* stop_tokens, int n_stop, const int32_t* max_new,
                                         int32_t* out_num_emitted, sv_stream_t stream) {
  if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || n_stop < 0 || n_stop > SV_MAX_STOP_TOKENS) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!tokens || !num_accepted || !out_num_emitted || (n_stop > 0 && !stop_tokens)) return SV_ERR_INVALID_ARG;
  const int threads = 128;
  sv::truncate_kernel<<<(unsigned)((B + threads - 1) / threads), threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      B, gamma, tokens, num_accepted, stop_tokens, n_stop, max_new, out_num_emitted);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: a size, pointer, alignment or parameter is invalid";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: valid arguments this library does not implement";
    case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA launch or runtime call failed";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded device wait gave up";
  }
  return "unknown sv_status";
}

extern "C" const char* sv_last_kernels(void) { return g_last_kernels; }

extern "C" int sv_pointer_device_readable(const void* p) {
  if (p == nullptr) return 0;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return 1;
  return at.type == cudaMemoryTypeHost && at.devicePointer == p ? 1 : 0;
}

extern "C" sv_status sv_set_timing_events(void* const* events, int n) {
  if (n == 0) {
    g_timing_on = false;
    g_timing[0] = g_timing[1] = g_timing[2] = nullptr;
    return SV_OK;
  }
  if (n != 3 || events == nullptr || !events[0] || !events[1] || !events[2]) return SV_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i) g_timing[i] = reinterpret_cast<cudaEvent_t>(events[i]);
  g_timing_on = true;
  return SV_OK;
}

// ------------------------------------------------------- vocabulary shards
// The steps of sv_shard.cuh behind the C entry points of include/specverify.h.
namespace {

bool shard_args_ok(int B, int gamma, int V, int v0, int Vg) {
  return sizes_ok(B, gamma, Vg) && V >= 1 && v0 >= 0 && (long long)v0 + V <= Vg;
}

// Parameters of this shard's slice: the layout of a call on V tokens.
sv_status shard_params(sv::Params& p, int B, int gamma, int V, int v0, int Vg, float temperature, void* workspace,
                       size_t workspace_bytes) {
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.v0 = v0;
  p.Vg = Vg;
  p.top_p = 1.0f;
  const double c = 1.4426950408889634 / (double)temperature;
  p.c = (float)c;
  p.c_lo = (float)(c - (double)p.c);
  if (workspace) {
    const Layout L = make_layout(B, gamma, V, 0);
    if (workspace_bytes < L.total || !aligned16(workspace)) return SV_ERR_WORKSPACE;
    bind_workspace(p, L, workspace);
  }
  return SV_OK;
}

template <typename T>
sv_status launch_shard_stats(const sv::Params& p, bool greedy, cudaStream_t st) {
  const unsigned grid = (unsigned)((long long)p.B * (p.gamma + 1));
  if (greedy) sv::shard_stats_kernel<T, true><<<grid, sv::kShThreads, 0, st>>>(p);
  else sv::shard_stats_kernel<T, false><<<grid, sv::kShThreads, 0, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

template <typename T>
sv_status launch_shard_pick(const sv::Params& p, cudaStream_t st) {
  auto kern = sv::shard_pick_kernel<T>;
  const size_t smem = sv::fd_stash_bytes(p.FC);   // the staged item sums and token masses
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  kern<<<(unsigned)p.B, sv::kFdThreads, smem, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace

extern "C" size_t sv_shard_workspace_bytes(int B, int gamma, int V) {
  if (!sizes_ok(B, gamma, V)) return 0;
  return make_layout(B, gamma, V, 0).total;
}

extern "C" sv_status sv_shard_row_stats(int B, int gamma, int V, int v0, int Vg, const void* logits,
                                        sv_dtype logits_dtype, const float* q, const int32_t* draft_tokens,
                                        float temperature, int greedy, void* stats_out, sv_stream_t stream) {
  g_last_kernels = "";
  if (!shard_args_ok(B, gamma, V, v0, Vg)) return SV_ERR_INVALID_ARG;
  if (logits_dtype != SV_DTYPE_F32 && logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F16)
    return SV_ERR_INVALID_ARG;
  if (!greedy && (!(temperature > 0.0f) || !std::isfinite(temperature))) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !stats_out || (gamma > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
  if (!aligned16(logits) || (q && !aligned16(q))) return SV_ERR_INVALID_ARG;
  sv::Params p{};
  shard_params(p, B, gamma, V, v0, Vg, greedy ? 1.0f : temperature, nullptr, 0);
  p.logits = logits;
  p.q = greedy ? nullptr : q;
  p.draft = draft_tokens;
  p.sh_out = stats_out;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  sv_status r = SV_ERR_INVALID_ARG;
  switch (logits_dtype) {
    case SV_DTYPE_F32: r = launch_shard_stats<float>(p, greedy != 0, st); break;
    case SV_DTYPE_BF16: r = launch_shard_stats<__nv_bfloat16>(p, greedy != 0, st); break;
    case SV_DTYPE_F16: r = launch_shard_stats<__half>(p, greedy != 0, st); break;
  }
  if (r == SV_OK) g_last_kernels = "shard_stats_kernel";
  return r;
}

extern "C" sv_status sv_shard_scan(int nshard, int B, int gamma, int V, int Vg, const void* stats_all,
                                   const int32_t* draft_tokens, const float* uniforms, float temperature, int greedy,
                                   int32_t* out_tokens, int32_t* out_num_accepted, float* out_accept_prob,
                                   int32_t* out_status, void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  g_last_kernels = "";
  if (nshard < 1 || nshard > sv::kMaxShards || !shard_args_ok(B, gamma, V, 0, Vg)) return SV_ERR_INVALID_ARG;
  if (!greedy && (!(temperature > 0.0f) || !std::isfinite(temperature))) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!stats_all || !out_tokens || !out_num_accepted || (gamma > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
  if (!greedy && !uniforms) return SV_ERR_INVALID_ARG;
  sv::Params p{};
  const sv_status ws = shard_params(p, B, gamma, V, 0, Vg, greedy ? 1.0f : temperature, greedy ? nullptr : workspace,
                                    workspace_bytes);
  if (ws != SV_OK) return ws;
  if (!greedy && !workspace) return SV_ERR_WORKSPACE;
  p.nshard = nshard;
  p.sh_in = stats_all;
  p.draft = draft_tokens;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_n = out_num_accepted;
  p.out_a = greedy ? nullptr : out_accept_prob;
  p.out_status = out_status;
  const unsigned grid = (unsigned)((B + sv::kShWarps - 1) / sv::kShWarps);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (greedy) sv::shard_scan_kernel<true><<<grid, sv::kShThreads, 0, st>>>(p);
  else sv::shard_scan_kernel<false><<<grid, sv::kShThreads, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  g_last_kernels = "shard_scan_kernel";
  return SV_OK;
}

extern "C" sv_status sv_shard_draw_sums(int B, int gamma, int V, int v0, int Vg, const void* logits,
                                        sv_dtype logits_dtype, const float* q, const int32_t* draft_tokens,
                                        float temperature, void* totals_out, void* workspace, size_t workspace_bytes,
                                        sv_stream_t stream) {
  g_last_kernels = "";
  if (!shard_args_ok(B, gamma, V, v0, Vg)) return SV_ERR_INVALID_ARG;
  if (logits_dtype != SV_DTYPE_F32 && logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F16)
    return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !totals_out || !workspace || (gamma > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
  if (!aligned16(logits) || (q && !aligned16(q)) || !aligned16(totals_out)) return SV_ERR_INVALID_ARG;
  sv::Params p{};
  const sv_status ws = shard_params(p, B, gamma, V, v0, Vg, temperature, workspace, workspace_bytes);
  if (ws != SV_OK) return ws;
  p.logits = logits;
  p.q = q;
  p.draft = draft_tokens;
  p.H = 0;          // the state comes from sv_shard_scan
  p.shard = 1;      // totals, no search
  p.sh_out = totals_out;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  sv_status r = SV_ERR_INVALID_ARG;
  switch (logits_dtype) {
    case SV_DTYPE_F32: r = launch_final_draw<float, false>(p, st); break;
    case SV_DTYPE_BF16: r = launch_final_draw<__nv_bfloat16, false>(p, st); break;
    case SV_DTYPE_F16: r = launch_final_draw<__half, false>(p, st); break;
  }
  if (r == SV_OK) g_last_kernels = "final_draw_kernel";
  return r;
}

extern "C" sv_status sv_shard_draw_pick(int nshard, int rank, int B, int gamma, int V, int v0, int Vg,
                                        const void* logits, sv_dtype logits_dtype, const float* q,
                                        const int32_t* draft_tokens, const float* uniforms, float temperature,
                                        const void* totals_all, int32_t* out_tokens, int32_t* out_status,
                                        void* workspace, size_t workspace_bytes, sv_stream_t stream) {
  g_last_kernels = "";
  if (nshard < 1 || nshard > sv::kMaxShards || rank < 0 || rank >= nshard) return SV_ERR_INVALID_ARG;
  if (!shard_args_ok(B, gamma, V, v0, Vg)) return SV_ERR_INVALID_ARG;
  if (logits_dtype != SV_DTYPE_F32 && logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F16)
    return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !uniforms || !totals_all || !out_tokens || !workspace || (gamma > 0 && !draft_tokens))
    return SV_ERR_INVALID_ARG;
  if (!aligned16(logits) || (q && !aligned16(q)) || !aligned16(totals_all)) return SV_ERR_INVALID_ARG;
  sv::Params p{};
  const sv_status ws = shard_params(p, B, gamma, V, v0, Vg, temperature, workspace, workspace_bytes);
  if (ws != SV_OK) return ws;
  p.nshard = nshard;
  p.rank = rank;
  p.logits = logits;
  p.q = q;
  p.draft = draft_tokens;
  p.uniforms = uniforms;
  p.sh_in = totals_all;
  p.out_tokens = out_tokens;
  p.out_status = out_status;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  sv_status r = SV_ERR_INVALID_ARG;
  switch (logits_dtype) {
    case SV_DTYPE_F32: r = launch_shard_pick<float>(p, st); break;
    case SV_DTYPE_BF16: r = launch_shard_pick<__nv_bfloat16>(p, st); break;
    case SV_DTYPE_F16: r = launch_shard_pick<__half>(p, st); break;
  }
  if (r == SV_OK) g_last_kernels = "shard_pick_kernel";
  return r;
}

// ------------------------------------------- vocabulary shards, truncated sampling
extern "C" sv_status sv_shard_topk_candidates(int B, int gamma, int V, int v0, int Vg, const void* logits,
                                              sv_dtype logits_dtype, const float* q, const int32_t* draft_tokens,
                                              float temperature, int top_k, void* cand_local, void* workspace,
                                              size_t workspace_bytes, sv_stream_t stream) {
  g_last_kernels = "";
  if (!shard_args_ok(B, gamma, V, v0, Vg)) return SV_ERR_INVALID_ARG;
  if (logits_dtype != SV_DTYPE_F32 && logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F16)
    return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > SV_MAX_TOP_K) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !cand_local || !workspace || (gamma > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
  if (!aligned16(logits) || (q && !aligned16(q)) || !aligned16(cand_local)) return SV_ERR_INVALID_ARG;
  if (V % vec_width(logits_dtype) != 0) return SV_ERR_UNSUPPORTED;   // the streaming top-k kernel's rows
  sv::Params p{};
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.v0 = v0;
  p.Vg = Vg;
  p.top_k = top_k;
  p.top_p = 1.0f;
  const double c = 1.4426950408889634 / (double)temperature;
  p.c = (float)c;
  p.c_lo = (float)(c - (double)p.c);
  const Layout L = make_layout(B, gamma, V, top_k);
  if (workspace_bytes < L.total || !aligned16(workspace)) return SV_ERR_WORKSPACE;
  bind_workspace(p, L, workspace);
  p.logits = logits;
  p.q = q;
  p.draft = draft_tokens;
  p.shard = 2;
  p.sh_out = cand_local;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  sv_status r = SV_ERR_INVALID_ARG;
  switch (logits_dtype) {
    case SV_DTYPE_F32: r = launch_stream_topk<float>(p, st); break;
    case SV_DTYPE_BF16: r = launch_stream_topk<__nv_bfloat16>(p, st); break;
    case SV_DTYPE_F16: r = launch_stream_topk<__half>(p, st); break;
  }
  if (r == SV_OK) g_last_kernels = "stream_topk_kernel";
  return r;
}

extern "C" sv_status sv_shard_topk_finish(int nshard, int B, int gamma, int Vg, const void* cand_all,
                                          const int32_t* draft_tokens, const float* uniforms, float temperature,
                                          int top_k, float top_p, int32_t* out_tokens, int32_t* out_num_accepted,
                                          float* out_accept_prob, int32_t* out_status, sv_stream_t stream) {
  g_last_kernels = "";
  if (nshard < 1 || nshard > sv::kMaxShards || !sizes_ok(B, gamma, Vg)) return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > SV_MAX_TOP_K || !(top_p > 0.0f && top_p <= 1.0f)) return SV_ERR_INVALID_ARG;
  if ((long long)nshard * top_k > sv::kShCandMax) return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  if (!cand_all || !uniforms || !out_tokens || !out_num_accepted || (gamma > 0 && !draft_tokens))
    return SV_ERR_INVALID_ARG;
  sv::Params p{};
  p.B = B;
  p.gamma = gamma;
  p.Vg = Vg;
  p.top_k = top_k;
  p.top_p = top_p;
  const double c = 1.4426950408889634 / (double)temperature;
  p.c = (float)c;
  p.c_lo = (float)(c - (double)p.c);
  p.nshard = nshard;
  p.sh_in = cand_all;
  p.draft = draft_tokens;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_n = out_num_accepted;
  p.out_a = out_accept_prob;
  p.out_status = out_status;
  const size_t smem = sizeof(sv::ShTopkSmem);
  if (cudaFuncSetAttribute(sv::shard_topk_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  sv::shard_topk_finish_kernel<<<(unsigned)B, sv::kShThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  g_last_kernels = "shard_topk_finish_kernel";
  return SV_OK;
}
