// Plain structs passed from the host side of the library to its kernels.
#pragma once

#include <stdint.h>

#include "../../include/lca.h"

namespace lca {

// Device error word bits.
constexpr unsigned int LCA_DEVERR_TIMEOUT = 1u;
constexpr unsigned int LCA_DEVERR_LAYOUT = 2u;   // shared-memory base not 1024-aligned

// Mask descriptor as the kernels see it (device arrays owned by the plan).
struct MaskDev {
  int type, seqlen, window, num_global, prefix_len, block, base_causal;
  int num_segments;
  const int32_t* cu;       // [num_segments + 1]
  int map_heads, n_rb, n_cb;
  const int32_t* row_off;  // [map_heads][n_rb + 1]
  const int32_t* col_off;  // [map_heads][n_cb + 1]
  const uint8_t* bmap;     // [map_heads][n_rb][n_cb]
};

// Tile plan as the kernels see it.
struct PlanDev {
  int tile_q, tile_k, n_qt, n_kt, map_heads;
  const uint8_t* cls;      // [map_heads][n_qt][n_kt]
  const int32_t* rowptr;   // [map_heads * n_qt + 1]
  const int32_t* kt_idx;   // [nnz]
  const uint8_t* kt_cls;   // [nnz]
  const int32_t* colptr;   // [map_heads * n_kt + 1]
  const int32_t* qt_idx;   // [nnz]
  const uint8_t* qt_cls;   // [nnz]
  const int32_t* work_q;   // [map_heads * n_qt]
  const int32_t* work_k;   // [map_heads * n_kt]
};

// Shape and head mapping shared by the attention kernels.
struct AttnDims {
  int batch, seqlen, h_q, h_kv, group;  // group = h_q / h_kv
  int heads_per_map;                    // query heads sharing one map head
  int kv_per_map;                       // KV heads per map head (0 when maps are per query head
                                        // and a KV group spans several maps)
  float scale;                          // softmax scale
  float scale_log2;                     // scale * log2(e)
  int chunk;                            // work items interleaved per launch-order group
  int head_dim;                         // 128 or 64
};

}  // namespace lca
