// Mask builder: the tile plan every attention kernel of the library walks.
//
// The benchmark feeds every kernel from one unified mask representation and its
// context-parallel framework precomputes its metadata once per mask
// ("Long-Context Attention Benchmark", summary page section 2.2; reading note, "Key
// design" 2-3).  Here that representation is a tile plan:
//   classify  - every (query tile, key tile) pair -> SKIP / FULL / PARTIAL and, for a
//               non-skipped tile, which of its key-column and query-row halves hold
//               no allowed pair (a kernel leaves those halves out), plus the exact
//               number of allowed pairs per map head and the list lengths;
//   scan      - CSR row pointers per (map head, query tile) and column pointers per
//               (map head, key tile);
//   fill      - ascending key-tile lists per row and query-tile lists per column;
//   lpt       - longest-first work orders (ties by index) for both lists.
// Classification evaluates each query row in closed form (two key intervals per row,
// restricted by the block map for the sparse masks), so no S x S mask is ever built.
#include <cuda_runtime.h>

#include <climits>

#include "lca_device.cuh"
#include "mask_build.h"

namespace lca {

namespace {

constexpr int KT_CHUNK = 1024;

__device__ __forceinline__ int overlap(int a, int b, int lo, int hi) {
  return max(0, min(b, hi) - max(a, lo));
}

template <int TQ, int TK>
__global__ void __launch_bounds__(TQ) classify_kernel(MaskDev m, int n_qt, int n_kt,
                                                      uint8_t* cls, int32_t* rowlen,
                                                      unsigned long long* n_valid,
                                                      unsigned long long* n_partial) {
  constexpr int NWARP = TQ / 32;
  constexpr int NW = TK / 32;
  __shared__ uint8_t s_any[NWARP][KT_CHUNK];   // bit 0 / 1: a pair in key half 0 / 1
  __shared__ uint8_t s_all[NWARP][KT_CHUNK];
  __shared__ unsigned long long s_red[NWARP];
  __shared__ int s_len[NWARP];
  __shared__ int s_part[NWARP];
  __shared__ int s_lo[NWARP], s_hi[NWARP];

  const int qt = blockIdx.x, hm = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = m.seqlen;
  const int i = qt * TQ + threadIdx.x;
  const bool valid = i < S;
  RowSpan sp{0, 0, 0, 0};
  if (valid) sp = row_span(m, i);
  const bool sparse = is_sparse(m.type);

  // Key tiles outside the hull of the block's allowed intervals are SKIP without any
  // per-row work (documents and windows leave most of a long row's tiles there).
  int lo = INT_MAX, hi = 0;
  if (valid) {
    if (sp.a0 < sp.b0) { lo = sp.a0; hi = sp.b0; }
    if (sp.a1 < sp.b1) { lo = min(lo, sp.a1); hi = max(hi, sp.b1); }
  }
  for (int off = 16; off > 0; off >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
    hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
  }
  if (lane == 0) { s_lo[warp] = lo; s_hi[warp] = hi; }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < NWARP; ++w) { lo = min(lo, s_lo[w]); hi = max(hi, s_hi[w]); }
  const int kt_lo = lo == INT_MAX ? n_kt : lo / TK;
  const int kt_hi = lo == INT_MAX ? n_kt : (hi + TK - 1) / TK;
  MapCursor mcur;

  unsigned long long my_count = 0;
  int my_len = 0, my_part = 0;
  uint8_t* cls_row = cls + (static_cast<size_t>(hm) * n_qt + qt) * n_kt;

  for (int k0 = 0; k0 < n_kt; k0 += KT_CHUNK) {
    const int k1 = min(n_kt, k0 + KT_CHUNK);
    for (int kt = k0; kt < k1; ++kt) {
      if (kt < kt_lo || kt >= kt_hi) {  // block-uniform
        if (lane == 0) {
          s_any[warp][kt - k0] = 0;
          s_all[warp][kt - k0] = 0;
        }
        continue;
      }
      const int c0 = kt * TK;
      const int width = min(TK, S - c0);
      const int cm = c0 + TK / 2;          // first key column of the second half
      int cnt0 = 0, cnt1 = 0;              // allowed pairs of this row in each key half
      if (valid) {
        if (sparse) {
          uint32_t bits[NW];
          row_tile_bits<NW>(m, hm, i, c0, sp, bits, &mcur);
#pragma unroll
          for (int w = 0; w < NW; ++w) (w < NW / 2 ? cnt0 : cnt1) += __popc(bits[w]);
        } else {
          const int ce = c0 + width;
          cnt0 = overlap(sp.a0, sp.b0, c0, min(cm, ce)) + overlap(sp.a1, sp.b1, c0, min(cm, ce));
          cnt1 = overlap(sp.a0, sp.b0, cm, ce) + overlap(sp.a1, sp.b1, cm, ce);
        }
      }
      const int cnt = cnt0 + cnt1;
      my_count += static_cast<unsigned long long>(cnt);
      const bool any0 = __any_sync(0xFFFFFFFFu, valid && cnt0 > 0);
      const bool any1 = __any_sync(0xFFFFFFFFu, valid && cnt1 > 0);
      const bool all_w = __all_sync(0xFFFFFFFFu, !valid || cnt == width);
      if (lane == 0) {
        s_any[warp][kt - k0] = static_cast<uint8_t>(any0 | (any1 << 1));
        s_all[warp][kt - k0] = all_w;
      }
    }
    __syncthreads();
    for (int kt = k0 + threadIdx.x; kt < k1; kt += TQ) {
      int keys = 0, top = 0, bottom = 0;   // key halves with a pair; rows of each half
      bool f = true;
#pragma unroll
      for (int w = 0; w < NWARP; ++w) {
        const int x = s_any[w][kt - k0];
        keys |= x;
        (w < NWARP / 2 ? top : bottom) |= x;
        f = f && s_all[w][kt - k0];
      }
      uint8_t c = LCA_TILE_SKIP;
      if (keys != 0) {
        c = f ? LCA_TILE_FULL : LCA_TILE_PARTIAL;
        if (!(keys & 1)) c |= LCA_TILE_KEY_HALF0_EMPTY;
        if (!(keys & 2)) c |= LCA_TILE_KEY_HALF1_EMPTY;
        if (!top) c |= LCA_TILE_QUERY_HALF0_EMPTY;
        if (!bottom) c |= LCA_TILE_QUERY_HALF1_EMPTY;
      }
      cls_row[kt] = c;
      my_len += (c != LCA_TILE_SKIP);
      my_part += ((c & LCA_TILE_CLASS_MASK) == LCA_TILE_PARTIAL);
    }
    __syncthreads();
  }
  // block reductions
  for (int off = 16; off > 0; off >>= 1) {
    my_count += __shfl_xor_sync(0xFFFFFFFFu, my_count, off);
    my_len += __shfl_xor_sync(0xFFFFFFFFu, my_len, off);
    my_part += __shfl_xor_sync(0xFFFFFFFFu, my_part, off);
  }
  if (lane == 0) {
    s_red[warp] = my_count;
    s_len[warp] = my_len;
    s_part[warp] = my_part;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long c = 0;
    int len = 0, part = 0;
    for (int w = 0; w < NWARP; ++w) {
      c += s_red[w];
      len += s_len[w];
      part += s_part[w];
    }
    rowlen[hm * n_qt + qt] = len;
    atomicAdd(n_valid + hm, c);
    atomicAdd(n_partial, static_cast<unsigned long long>(part));
  }
}

// Exclusive prefix sum of `len` [n] into `ptr` [n + 1] (one block).
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* len, int n, int32_t* ptr) {
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int idx = base + threadIdx.x;
    const int v = idx < n ? len[idx] : 0;
    int x = v;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = s_warp[lane];
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, w, off);
        if (lane >= off) w += y;
      }
      s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int warp_excl = warp > 0 ? s_warp[warp - 1] : 0;
    if (idx < n) ptr[idx] = s_carry + warp_excl + x - v;
    __syncthreads();
    if (threadIdx.x == 0) s_carry += s_warp[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) ptr[n] = s_carry;
}

// Number of non-skipped query tiles of every (map head, key tile) column.
__global__ void collen_kernel(const uint8_t* cls, int map_heads, int n_qt, int n_kt,
                              int32_t* collen) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= map_heads * n_kt) return;
  const int hm = c / n_kt, kt = c % n_kt;
  const uint8_t* base = cls + static_cast<size_t>(hm) * n_qt * n_kt + kt;
  int len = 0;
  for (int qt = 0; qt < n_qt; ++qt) len += base[static_cast<size_t>(qt) * n_kt] != 0;
  collen[c] = len;
}

// One warp per row: ascending key tiles and their classes.
__global__ void fill_rows_kernel(const uint8_t* cls, int n_rows, int n_kt, const int32_t* rowptr,
                                 int32_t* kt_idx, uint8_t* kt_cls) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= n_rows) return;
  const uint8_t* row = cls + static_cast<size_t>(r) * n_kt;
  int pos = rowptr[r];
  for (int k0 = 0; k0 < n_kt; k0 += 32) {
    const int kt = k0 + lane;
    const uint8_t c = kt < n_kt ? row[kt] : 0;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, c != 0);
    if (c != 0) {
      const int at = pos + __popc(bal & ((1u << lane) - 1u));
      kt_idx[at] = kt;
      kt_cls[at] = row_list_byte(c);
    }
    pos += __popc(bal);
  }
}

// One thread per column: ascending query tiles and their classes.
__global__ void fill_cols_kernel(const uint8_t* cls, int map_heads, int n_qt, int n_kt,
                                 const int32_t* colptr, int32_t* qt_idx, uint8_t* qt_cls) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= map_heads * n_kt) return;
  const int hm = c / n_kt, kt = c % n_kt;
  const uint8_t* base = cls + static_cast<size_t>(hm) * n_qt * n_kt + kt;
  int pos = colptr[c];
  for (int qt = 0; qt < n_qt; ++qt) {
    const uint8_t v = base[static_cast<size_t>(qt) * n_kt];
    if (v) {
      qt_idx[pos] = qt;
      qt_cls[pos] = col_list_byte(v);
      ++pos;
    }
  }
}

// Longest-first order of list indices, ties by ascending index (a stable counting
// sort by descending length).  Block 0 orders the rows, block 1 the columns; one warp
// each, histogram in shared memory.
__global__ void __launch_bounds__(32) lpt_kernel(const int32_t* rowptr, int n_rows, int max_rows,
                                                 int32_t* work_q, const int32_t* colptr,
                                                 int n_cols, int max_cols, int32_t* work_k) {
  extern __shared__ int hist[];
  const int32_t* ptr = blockIdx.x == 0 ? rowptr : colptr;
  const int n = blockIdx.x == 0 ? n_rows : n_cols;
  const int maxlen = blockIdx.x == 0 ? max_rows : max_cols;
  int32_t* work = blockIdx.x == 0 ? work_q : work_k;
  const int lane = threadIdx.x;
  for (int L = lane; L <= maxlen; L += 32) hist[L] = 0;
  __syncwarp();
  for (int r = lane; r < n; r += 32) atomicAdd(&hist[ptr[r + 1] - ptr[r]], 1);
  __syncwarp();
  // start offset of every length: number of lists strictly longer
  int carry = 0;
  for (int top = maxlen; top >= 0; top -= 32) {
    const int L = top - lane;
    const int v = L >= 0 ? hist[L] : 0;
    int x = v;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
      if (lane >= off) x += y;
    }
    __syncwarp();
    if (L >= 0) hist[L] = carry + x - v;
    carry += __shfl_sync(0xFFFFFFFFu, x, 31);
    __syncwarp();
  }
  for (int base = 0; base < n; base += 32) {
    const int r = base + lane;
    const bool act = r < n;
    const int L = act ? ptr[r + 1] - ptr[r] : -1 - lane;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, L);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int slot = 0;
    if (act) slot = hist[L] + rank;
    __syncwarp();
    if (act) {
      work[slot] = r;
      if (lane == __ffs(peers) - 1) hist[L] += __popc(peers);
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_classify(const MaskDev& m, int tile_q, int tile_k, int n_qt, int n_kt,
                            uint8_t* cls, int32_t* rowlen, unsigned long long* n_valid,
                            unsigned long long* n_partial, cudaStream_t st) {
  dim3 grid(n_qt, m.map_heads);
  if (tile_q == 128 && tile_k == 128)
    classify_kernel<128, 128><<<grid, 128, 0, st>>>(m, n_qt, n_kt, cls, rowlen, n_valid, n_partial);
  else if (tile_q == 128 && tile_k == 64)
    classify_kernel<128, 64><<<grid, 128, 0, st>>>(m, n_qt, n_kt, cls, rowlen, n_valid, n_partial);
  else if (tile_q == 64 && tile_k == 128)
    classify_kernel<64, 128><<<grid, 64, 0, st>>>(m, n_qt, n_kt, cls, rowlen, n_valid, n_partial);
  else
    classify_kernel<64, 64><<<grid, 64, 0, st>>>(m, n_qt, n_kt, cls, rowlen, n_valid, n_partial);
  return cudaGetLastError();
}

cudaError_t launch_scan(const int32_t* len, int n, int32_t* ptr, cudaStream_t st) {
  scan_kernel<<<1, 1024, 0, st>>>(len, n, ptr);
  return cudaGetLastError();
}

cudaError_t launch_collen(const uint8_t* cls, int map_heads, int n_qt, int n_kt, int32_t* collen,
                          cudaStream_t st) {
  const int n = map_heads * n_kt;
  collen_kernel<<<(n + 255) / 256, 256, 0, st>>>(cls, map_heads, n_qt, n_kt, collen);
  return cudaGetLastError();
}

cudaError_t launch_fill(const uint8_t* cls, int map_heads, int n_qt, int n_kt,
                        const int32_t* rowptr, int32_t* kt_idx, uint8_t* kt_cls,
                        const int32_t* colptr, int32_t* qt_idx, uint8_t* qt_cls,
                        cudaStream_t st) {
  const int n_rows = map_heads * n_qt;
  fill_rows_kernel<<<(n_rows * 32 + 255) / 256, 256, 0, st>>>(cls, n_rows, n_kt, rowptr, kt_idx,
                                                              kt_cls);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n_cols = map_heads * n_kt;
  fill_cols_kernel<<<(n_cols + 255) / 256, 256, 0, st>>>(cls, map_heads, n_qt, n_kt, colptr,
                                                         qt_idx, qt_cls);
  return cudaGetLastError();
}

cudaError_t launch_lpt(const int32_t* rowptr, int n_rows, int max_rows, int32_t* work_q,
                       const int32_t* colptr, int n_cols, int max_cols, int32_t* work_k,
                       cudaStream_t st) {
  const size_t smem = static_cast<size_t>(max(max_rows, max_cols) + 1) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(lpt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  lpt_kernel<<<2, 32, smem, st>>>(rowptr, n_rows, max_rows, work_q, colptr, n_cols, max_cols,
                                  work_k);
  return cudaGetLastError();
}

}  // namespace lca
