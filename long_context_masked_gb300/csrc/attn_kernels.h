// Host-side launchers and argument blocks of the attention kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lca_types.h"

namespace lca {

struct FwdArgs {
  AttnDims dims;
  PlanDev plan;
  MaskDev mask;
  __nv_bfloat16* o;
  float* lse;
  int64_t o_row_stride;
  unsigned int* err;
  uint64_t timeout_ns;
  int n_units;                  // (query tile, query head, batch entry) units
  unsigned int* unit_counter;   // next unit to hand out (zeroed before the launch)
};

struct BwdArgs {
  AttnDims dims;
  PlanDev plan;
  MaskDev mask;
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;         // forward LSE, [B, H_q, S]
  float* lse2;              // workspace: LSE * log2(e) (+inf for rows without keys and
                            // padding), [B, H_q, s_pad]
  float* dsum;              // workspace: D = rowsum(dO * O) (0 on padding), [B, H_q, s_pad]
  int64_t s_pad;            // seqlen rounded up to the 128-row tile
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int64_t o_row_stride;     // O
  int64_t do_row_stride;    // dO
  int64_t dq_row_stride;    // dQ
  int64_t dk_row_stride;    // dK
  int64_t dv_row_stride;    // dV
  unsigned int* err;
  uint64_t timeout_ns;
};

size_t fwd_smem_bytes();
// n_ctas persistent CTAs (at most one per SM) take the args.n_units units from
// args.unit_counter, which the launch zeroes first on `st`.
cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& args, int n_ctas, cudaStream_t st);

cudaError_t launch_bwd_preprocess(const BwdArgs& args, cudaStream_t st);
// dK/dV (n_kv CTAs: one per KV head and key tile) and dQ (n_q CTAs: one per query head
// and query tile) in one launch.
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdArgs& args, int n_kv, int n_q,
                       cudaStream_t st);

cudaError_t launch_selftest_wait(unsigned int* err, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_selftest_umma(int variant, const CUtensorMap& ta, const CUtensorMap& tb,
                                 const __nv_bfloat16* a_rowmajor, float* c, unsigned int* err,
                                 cudaStream_t st);

}  // namespace lca
