// Host-side launchers of the block-score and top-k kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lca {

struct BlockScoreArgs {
  const __nv_bfloat16* q;   // [1, S, h_q, 128]
  const __nv_bfloat16* k;   // [1, S, h_kv, 128]
  int64_t q_row_stride, k_row_stride;
  int seqlen, block, n_blocks;
  int map_heads, heads_per_map, group;
  float scale;
  float* pooled;            // workspace [2][map_heads][n_blocks][128]
  float* scores;            // [map_heads][n_blocks][n_blocks]
};

size_t block_scores_workspace_bytes(int map_heads, int n_blocks);
cudaError_t launch_block_scores(const BlockScoreArgs& a, cudaStream_t st);
cudaError_t launch_block_topk(const float* scores, int rows, int n_cols, int k, uint8_t* map,
                              cudaStream_t st);

}  // namespace lca
