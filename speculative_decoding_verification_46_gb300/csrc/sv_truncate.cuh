// Ending a round early: stop tokens and max_new_tokens ("11.1 核心原理",
// listing 10-1's comment: EOS / stop / max_new_tokens may end the round, and
// no bonus token is forced).  The round emitted tokens[b][0 .. n_b]; keep them
// up to and including the first stop token and at most max_new[b] of them;
// the rest become -1.  One thread per sequence (at most gamma + 1 tokens and
// SV_MAX_STOP_TOKENS stop ids each): the work is tiny, launch latency rules.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

__global__ void truncate_kernel(int B, int G, int32_t* tokens, const int32_t* n_acc, const int32_t* stops, int n_stop,
                                const int32_t* max_new, int32_t* out_emitted) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int G1 = G + 1;
  int32_t* row = tokens + (size_t)b * G1;
  const int n = min(max(n_acc[b], 0), G);   // as the verify calls write it; clamped
  int k = n + 1;
  for (int j = 0; j <= n; ++j) {
    const int32_t t = row[j];
    bool hit = false;
    for (int s = 0; s < n_stop; ++s) hit |= (t == __ldg(stops + s));
    if (hit) {
      k = j + 1;
      break;
    }
  }
  if (max_new) k = min(k, max(max_new[b], 0));
  for (int j = k; j < G1; ++j) row[j] = -1;
  out_emitted[b] = k;
}

}  // namespace sv
