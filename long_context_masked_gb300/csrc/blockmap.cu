// Block-sparse maps from block scores: the step that turns a dynamic importance
// estimate into the block map the attention kernels consume.
//
// The benchmark builds its sparse masks by partitioning the attention map into
// query/key block grids, scoring every block pair and keeping the top-k key blocks of
// each query block, k following from the sparsity ratio ("Long-Context Attention
// Benchmark", summary page, appendix A.2: Block Partitioning, Score Calculation, Top-k
// Selection).  Its dynamic masks score blocks from the data; VSA's coarse stage
// mean-pools the tokens of each block and scores pooled queries against pooled keys
// (appendix A.3, "VSA").  Three kernels:
//   pool    mean of Q over the rows of a query block and the query heads of a map head,
//           and of K over the rows of a key block and those heads' KV heads (HBM-bound:
//           Q and K are read once, 16-byte loads, 16 row slots per CTA);
//   scores  scale * pooled Q . pooled K^T per map head (a small fp32 contraction,
//           2 * n_blocks^2 * d flops per map head, on the CUDA cores);
//   top-k   per (map head, query block) row: exact k-th largest score by a 4-pass
//           radix select on order-preserving 32-bit keys, then the row's entries above
//           it plus the lowest-index entries equal to it (descending score, ties by
//           ascending key block - a unique selection).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "blockmap.h"

namespace lca {

namespace {

constexpr int HD = 128;
constexpr int POOL_THREADS = 256;   // 16 row slots x 16 threads, 8 dims per thread
constexpr int SLOTS = POOL_THREADS / 16;

// grid (n_blocks, map_heads, 2): z = 0 pools Q, z = 1 pools K.
__global__ void __launch_bounds__(POOL_THREADS) pool_kernel(BlockScoreArgs a) {
  const int blk = blockIdx.x, hm = blockIdx.y, z = blockIdx.z;
  const int slot = threadIdx.x >> 4, part = threadIdx.x & 15;   // dims [8 part, 8 part + 8)
  const int r0 = blk * a.block, r1 = min(a.seqlen, r0 + a.block);
  const int hq0 = hm * a.heads_per_map;
  int h0, nh;
  const __nv_bfloat16* src;
  int64_t stride;
  if (z == 0) {
    h0 = hq0; nh = a.heads_per_map; src = a.q; stride = a.q_row_stride;
  } else {
    h0 = hq0 / a.group;
    nh = (hq0 + a.heads_per_map - 1) / a.group - h0 + 1;
    src = a.k; stride = a.k_row_stride;
  }
  const int items = (r1 - r0) * nh;
  float acc[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) acc[x] = 0.f;
  for (int it = slot; it < items; it += SLOTS) {
    const int r = r0 + it / nh, hh = h0 + it % nh;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + r * stride + hh * HD) + part);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 f = __bfloat1622float2(p[x]);
      acc[2 * x] += f.x;
      acc[2 * x + 1] += f.y;
    }
  }
  __shared__ float red[SLOTS][HD];
#pragma unroll
  for (int x = 0; x < 8; ++x) red[slot][part * 8 + x] = acc[x];
  __syncthreads();
  if (threadIdx.x < HD) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < SLOTS; ++w) s += red[w][threadIdx.x];
    const float inv = items > 0 ? 1.f / static_cast<float>(items) : 0.f;
    a.pooled[((static_cast<int64_t>(z) * a.map_heads + hm) * a.n_blocks + blk) * HD +
             threadIdx.x] = s * inv;
  }
}

// scores[hm][r][c] = scale * sum_x Qp[hm][r][x] Kp[hm][c][x]; 64 x 64 outputs per CTA,
// 4 x 4 per thread, 32-dim slices of both operands staged in shared memory.
constexpr int ST = 64, SK = 32;

__global__ void __launch_bounds__(256) score_kernel(BlockScoreArgs a) {
  const int hm = blockIdx.z;
  const int r0 = blockIdx.y * ST, c0 = blockIdx.x * ST;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* qp = a.pooled + static_cast<int64_t>(hm) * a.n_blocks * HD;
  const float* kp = a.pooled + (static_cast<int64_t>(a.map_heads) + hm) * a.n_blocks * HD;
  __shared__ float as[SK][ST + 1], bs[SK][ST + 1];
  float c[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) c[u][v] = 0.f;
  for (int k0 = 0; k0 < HD; k0 += SK) {
    for (int e = threadIdx.x; e < ST * SK; e += 256) {
      const int row = e / SK, kk = e % SK;
      const int gr = r0 + row, gc = c0 + row;
      as[kk][row] = gr < a.n_blocks ? qp[static_cast<int64_t>(gr) * HD + k0 + kk] : 0.f;
      bs[kk][row] = gc < a.n_blocks ? kp[static_cast<int64_t>(gc) * HD + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SK; ++kk) {
      float x[4], y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        x[u] = as[kk][ty * 4 + u];
        y[u] = bs[kk][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) c[u][v] = fmaf(x[u], y[v], c[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int r = r0 + ty * 4 + u;
    if (r >= a.n_blocks) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int cc = c0 + tx * 4 + v;
      if (cc < a.n_blocks)
        a.scores[(static_cast<int64_t>(hm) * a.n_blocks + r) * a.n_blocks + cc] =
            a.scale * c[u][v];
    }
  }
}

// 32-bit key whose unsigned order is the float order.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int TOPK_THREADS = 256;

// One CTA per (map head, row).
__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(const float* scores, int n_cols,
                                                            int k, uint8_t* map) {
  const int64_t row = blockIdx.x;
  const float* s = scores + row * n_cols;
  uint8_t* out = map + row * n_cols;
  __shared__ int hist[256];
  __shared__ int sh_sel, sh_remaining;
  __shared__ int warp_tot[TOPK_THREADS / 32];
  uint32_t prefix = 0u, mask = 0u;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int d = threadIdx.x; d < 256; d += TOPK_THREADS) hist[d] = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < n_cols; c += TOPK_THREADS) {
      const uint32_t key = order_key(__ldg(s + c));
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, sel = 0;
      for (int d = 255; d >= 0; --d) {
        if (cum + hist[d] >= remaining) { sel = d; break; }
        cum += hist[d];
      }
      sh_sel = sel;
      sh_remaining = remaining - cum;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sh_sel) << shift;
    mask |= 255u << shift;
    remaining = sh_remaining;
    __syncthreads();
  }
  // prefix = key of the k-th largest score; `remaining` entries equal to it are kept,
  // the lowest-index ones (exclusive scan over the row in index order)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int taken = 0;
  for (int base = 0; base < n_cols; base += TOPK_THREADS) {
    const int c = base + threadIdx.x;
    uint32_t key = 0u;
    if (c < n_cols) key = order_key(__ldg(s + c));
    const bool eq = c < n_cols && key == prefix;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, eq);
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = taken;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    before += __popc(bal & ((1u << lane) - 1u));
    int chunk_total = 0;
    for (int w = 0; w < TOPK_THREADS / 32; ++w) chunk_total += warp_tot[w];
    if (c < n_cols) out[c] = (key > prefix || (eq && before < remaining)) ? 1 : 0;
    taken += chunk_total;
    __syncthreads();
  }
}

}  // namespace

size_t block_scores_workspace_bytes(int map_heads, int n_blocks) {
  return 2 * static_cast<size_t>(map_heads) * n_blocks * HD * sizeof(float);
}

cudaError_t launch_block_scores(const BlockScoreArgs& a, cudaStream_t st) {
  pool_kernel<<<dim3(a.n_blocks, a.map_heads, 2), POOL_THREADS, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int g = (a.n_blocks + ST - 1) / ST;
  score_kernel<<<dim3(g, g, a.map_heads), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_block_topk(const float* scores, int rows, int n_cols, int k, uint8_t* map,
                              cudaStream_t st) {
  topk_kernel<<<rows, TOPK_THREADS, 0, st>>>(scores, n_cols, k, map);
  return cudaGetLastError();
}

}  // namespace lca
