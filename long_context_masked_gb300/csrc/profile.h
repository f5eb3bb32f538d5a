// Optional per-kernel CUDA-event timing of the library's launches (lca_profile_*).
#pragma once

#include <cuda_runtime.h>

namespace lca {

enum KernelId {
  K_CLASSIFY = 0, K_SCAN, K_COLLEN, K_FILL, K_LPT, K_FWD, K_BWD_PRE, K_BWD,
  K_BLOCK_SCORES, K_BLOCK_TOPK,
  K_COUNT
};

bool profiling_on();
long profile_begin(int id, int launches, cudaStream_t st);
void profile_end(long token, cudaStream_t st);

// Records events around the launches in its scope when profiling is enabled.
struct ProfScope {
  long tok = 0;
  cudaStream_t st;
  ProfScope(int id, cudaStream_t s, int launches = 1) : st(s) {
    if (profiling_on()) tok = profile_begin(id, launches, s);
  }
  ~ProfScope() {
    if (tok) profile_end(tok, st);
  }
};

}  // namespace lca
