// Host-side launchers of the mask builder kernels (mask_build.cu).
#pragma once

#include <cuda_runtime.h>

#include "lca_types.h"

namespace lca {

cudaError_t launch_classify(const MaskDev& m, int tile_q, int tile_k, int n_qt, int n_kt,
                            uint8_t* cls, int32_t* rowlen, unsigned long long* n_valid,
                            unsigned long long* n_partial, cudaStream_t st);
cudaError_t launch_scan(const int32_t* len, int n, int32_t* ptr, cudaStream_t st);
cudaError_t launch_collen(const uint8_t* cls, int map_heads, int n_qt, int n_kt, int32_t* collen,
                          cudaStream_t st);
cudaError_t launch_fill(const uint8_t* cls, int map_heads, int n_qt, int n_kt,
                        const int32_t* rowptr, int32_t* kt_idx, uint8_t* kt_cls,
                        const int32_t* colptr, int32_t* qt_idx, uint8_t* qt_cls,
                        cudaStream_t st);
cudaError_t launch_lpt(const int32_t* rowptr, int n_rows, int max_rows, int32_t* work_q,
                       const int32_t* colptr, int n_cols, int max_cols, int32_t* work_k,
                       cudaStream_t st);

}  // namespace lca
