// sv_verify_greedy_noalloc: greedy verify that needs no workspace from the
// caller.  Its scratch is one array of SV_NOALLOC_SCRATCH_BYTES defined below;
// every GPU that loads this library holds a copy until the process exits.
//
// Some callers cannot allocate device memory: plugins whose host framework
// owns every device allocation and passes none down, runtimes that plan a
// fixed memory budget before serving starts, or loops that must not call
// cudaMalloc because it can synchronise the device and stall other streams.
// They call this entry point instead of sv_verify_greedy.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "specverify.h"

// The scratch shared by all calls on a device.  It keeps whatever the last
// call left in it; each call clears the bytes it uses before its kernel runs.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
// One cached address per device.  Atomic: host threads making their first
// call on the same device at the same time may both look the address up;
// they store the same value and neither reads a torn one.
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device.  Looked up once per
// device (with that device current) and cached; the array's name in host code
// is only a host-side stand-in, never a device address.
sv_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SV_ERR_CUDA;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return SV_OK;
}

}  // namespace

extern "C" sv_status sv_verify_greedy_noalloc(int B, int gamma, int V, const void* logits, sv_dtype logits_dtype,
                                              const int32_t* draft_tokens, int32_t* out_tokens,
                                              int32_t* out_num_accepted, int32_t* out_status, sv_stream_t stream) {
  const size_t need = sv_workspace_bytes(B, gamma, V, 0);
  if (need == 0) return SV_ERR_INVALID_ARG;
  if (need > (size_t)SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;   // problem too large for the scratch
  if (logits_dtype != SV_DTYPE_F32 && logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F16)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !out_tokens || !out_num_accepted || (gamma > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) != 0) return SV_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const sv_status st = scratch_on_current_device(&scratch);
  if (st != SV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  return sv_verify_greedy(B, gamma, V, logits, logits_dtype, draft_tokens, out_tokens, out_num_accepted, out_status,
                          scratch, need, stream);
}
