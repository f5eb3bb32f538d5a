// C ABI of the library (include/lca.h): argument validation, the plan object, TMA
// tensor maps and kernel launches.  Host code only; every step of the computation
// runs in the kernels of mask_build.cu, attn_fwd.cu and attn_bwd.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "attn_kernels.h"
#include "blockmap.h"
#include "lca_types.h"
#include "mask_build.h"
#include "profile.h"

using namespace lca;

namespace {

__device__ unsigned int g_device_error = 0;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

constexpr int kMaxSeqlen = 1 << 20;
constexpr int kHeadDim = 128;

unsigned int* device_error_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
  return static_cast<unsigned int*>(p);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tensor map of a [B, S, H, 128] bf16 tensor (row stride in elements); a box is
// `box_rows` positions x one head x 64 elements, 128-byte swizzled (one half of a row).
bool make_tmap_bshd(CUtensorMap* m, const void* ptr, int batch, int seqlen, int heads,
                    int64_t row_stride, int box_rows, int head_dim = kHeadDim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(seqlen), static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(row_stride) * 2,
                           static_cast<cuuint64_t>(row_stride) * 2 * seqlen};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SMs of the current device (the persistent forward runs one CTA per SM).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}

bool is_sparse_type(int t) { return t == LCA_BLOCK_SPARSE_UNIFORM || t == LCA_BLOCK_SPARSE_VARIABLE; }

bool needs_segments(int t) {
  return t == LCA_FULL_DOCUMENT || t == LCA_CAUSAL_DOCUMENT || t == LCA_SHARED_QUESTION ||
         t == LCA_BLOCK_CAUSAL_DOCUMENT || t == LCA_SLIDING_WINDOW_DOCUMENT;
}

template <typename T>
bool copy_to_host(std::vector<T>& dst, const T* src, size_t n) {
  dst.resize(n);
  if (n == 0) return true;
  return cudaMemcpy(dst.data(), src, n * sizeof(T), cudaMemcpyDeviceToHost) == cudaSuccess;
}

bool offsets_ok(const std::vector<int32_t>& v, int n, int S) {
  if (v.empty() || v[0] != 0 || v[n] != S) return false;
  for (int k = 0; k < n; ++k)
    if (v[k + 1] < v[k]) return false;
  return true;
}

lca_status validate_desc(const lca_mask_desc* d, int tile_q, int tile_k) {
  if (!d) return LCA_ERR_INVALID_ARG;
  if ((tile_q != 64 && tile_q != 128) || (tile_k != 64 && tile_k != 128)) return LCA_ERR_UNSUPPORTED;
  if (d->type < LCA_FULL || d->type > LCA_SLIDING_WINDOW_DOCUMENT) return LCA_ERR_INVALID_ARG;
  const int S = d->seqlen;
  if (S < 1) return LCA_ERR_INVALID_ARG;
  if (S > kMaxSeqlen) return LCA_ERR_UNSUPPORTED;
  switch (d->type) {
    case LCA_SLIDING_WINDOW:
    case LCA_SLIDING_WINDOW_DOCUMENT:
      if (d->window < 1) return LCA_ERR_INVALID_ARG;
      break;
    case LCA_GLOBAL_SLIDING:
      if (d->window < 1 || d->num_global < 0) return LCA_ERR_INVALID_ARG;
      break;
    case LCA_PREFIX_LM:
      if (d->prefix_len < 0 || d->prefix_len > S) return LCA_ERR_INVALID_ARG;
      break;
    case LCA_CAUSAL_BLOCKWISE:
    case LCA_BLOCK_CAUSAL_DOCUMENT:
    case LCA_BLOCK_SPARSE_UNIFORM:
      if (d->block < 1) return LCA_ERR_INVALID_ARG;
      break;
    default:
      break;
  }
  const bool segs = needs_segments(d->type) || (is_sparse_type(d->type) && d->num_segments > 0);
  if (needs_segments(d->type) && d->num_segments < 1) return LCA_ERR_INVALID_ARG;
  if (segs) {
    if (!d->cu_seqlens || d->num_segments < 1) return LCA_ERR_INVALID_ARG;
    std::vector<int32_t> cu;
    if (!copy_to_host(cu, d->cu_seqlens, static_cast<size_t>(d->num_segments) + 1))
      return LCA_ERR_INVALID_ARG;
    if (!offsets_ok(cu, d->num_segments, S)) return LCA_ERR_INVALID_ARG;
  }
  if (is_sparse_type(d->type)) {
    if (d->map_heads < 1 || d->n_row_blocks < 1 || d->n_col_blocks < 1 || !d->block_map)
      return LCA_ERR_INVALID_ARG;
    if (d->type == LCA_BLOCK_SPARSE_UNIFORM) {
      const int nb = (S + d->block - 1) / d->block;
      if (d->n_row_blocks != nb || d->n_col_blocks != nb) return LCA_ERR_INVALID_ARG;
    } else {
      if (!d->row_block_offsets || !d->col_block_offsets) return LCA_ERR_INVALID_ARG;
      std::vector<int32_t> ro, co;
      const size_t nr = static_cast<size_t>(d->n_row_blocks) + 1;
      const size_t nc = static_cast<size_t>(d->n_col_blocks) + 1;
      if (!copy_to_host(ro, d->row_block_offsets, nr * d->map_heads) ||
          !copy_to_host(co, d->col_block_offsets, nc * d->map_heads))
        return LCA_ERR_INVALID_ARG;
      for (int h = 0; h < d->map_heads; ++h) {
        std::vector<int32_t> r(ro.begin() + h * nr, ro.begin() + (h + 1) * nr);
        std::vector<int32_t> c(co.begin() + h * nc, co.begin() + (h + 1) * nc);
        if (!offsets_ok(r, d->n_row_blocks, S) || !offsets_ok(c, d->n_col_blocks, S))
          return LCA_ERR_INVALID_ARG;
      }
    }
  }
  return LCA_OK;
}

}  // namespace

// Unit counters of the forward's persistent CTAs: a launch takes the next of
// kFwdCounters counters, so up to that many forward launches of one plan may overlap.
constexpr int kFwdCounters = 16;

struct lca_plan {
  lca_plan_info info{};
  MaskDev mask{};
  PlanDev dev{};
  unsigned long long* n_valid = nullptr;
  unsigned int* fwd_counters = nullptr;   // [kFwdCounters]
  std::atomic<unsigned int> fwd_next{0};
  std::vector<void*> allocs;
  size_t bytes = 0;   // device memory held by the plan

  ~lca_plan() {
    for (void* p : allocs) cudaFree(p);
  }
  template <typename T>
  T* alloc(size_t n) {
    void* p = nullptr;
    if (cudaMalloc(&p, (n ? n : 1) * sizeof(T)) != cudaSuccess) return nullptr;
    allocs.push_back(p);
    bytes += (n ? n : 1) * sizeof(T);
    return static_cast<T*>(p);
  }
};

extern "C" {

const char* lca_status_string(lca_status s) {
  switch (s) {
    case LCA_OK: return "ok";
    case LCA_ERR_INVALID_ARG: return "invalid argument";
    case LCA_ERR_UNSUPPORTED: return "unsupported configuration";
    case LCA_ERR_CUDA: return "CUDA error";
    case LCA_ERR_OOM: return "out of device memory";
    case LCA_ERR_TIMEOUT: return "device wait timed out";
    case LCA_ERR_PLAN_MISMATCH: return "plan does not match the shape";
  }
  return "unknown status";
}

void lca_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

lca_status lca_mask_build(const lca_mask_desc* desc, int tile_q, int tile_k, void* stream,
                          lca_plan** out) {
  if (!out) return LCA_ERR_INVALID_ARG;
  *out = nullptr;
  lca_status vs = validate_desc(desc, tile_q, tile_k);
  if (vs != LCA_OK) return vs;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  lca_plan* p = new (std::nothrow) lca_plan();
  if (!p) return LCA_ERR_OOM;

  const int S = desc->seqlen;
  const int t = desc->type;
  const bool sparse = is_sparse_type(t);
  const bool segs = needs_segments(t) || (sparse && desc->num_segments > 0);
  const int hm_n = sparse ? desc->map_heads : 1;
  const int n_qt = (S + tile_q - 1) / tile_q;
  const int n_kt = (S + tile_k - 1) / tile_k;

  MaskDev& m = p->mask;
  m.type = t;
  m.seqlen = S;
  m.window = desc->window;
  m.num_global = desc->num_global;
  m.prefix_len = desc->prefix_len;
  m.block = desc->block > 0 ? desc->block : 1;
  m.base_causal = desc->base_causal;
  m.num_segments = segs ? desc->num_segments : 0;
  m.map_heads = hm_n;
  m.n_rb = sparse ? desc->n_row_blocks : 0;
  m.n_cb = sparse ? desc->n_col_blocks : 0;

  auto fail = [&](lca_status s) {
    delete p;
    return s;
  };
  auto cuda_ok = [](cudaError_t e) { return e == cudaSuccess; };

  if (segs) {
    int32_t* cu = p->alloc<int32_t>(desc->num_segments + 1);
    if (!cu) return fail(LCA_ERR_OOM);
    if (!cuda_ok(cudaMemcpyAsync(cu, desc->cu_seqlens, (desc->num_segments + 1) * sizeof(int32_t),
                                 cudaMemcpyDeviceToDevice, st)))
      return fail(LCA_ERR_CUDA);
    m.cu = cu;
  }
  if (sparse) {
    const size_t nmap = static_cast<size_t>(hm_n) * m.n_rb * m.n_cb;
    uint8_t* bm = p->alloc<uint8_t>(nmap);
    if (!bm) return fail(LCA_ERR_OOM);
    if (!cuda_ok(cudaMemcpyAsync(bm, desc->block_map, nmap, cudaMemcpyDeviceToDevice, st)))
      return fail(LCA_ERR_CUDA);
    m.bmap = bm;
    if (t == LCA_BLOCK_SPARSE_VARIABLE) {
      const size_t nr = static_cast<size_t>(hm_n) * (m.n_rb + 1);
      const size_t nc = static_cast<size_t>(hm_n) * (m.n_cb + 1);
      int32_t* ro = p->alloc<int32_t>(nr);
      int32_t* co = p->alloc<int32_t>(nc);
      if (!ro || !co) return fail(LCA_ERR_OOM);
      if (!cuda_ok(cudaMemcpyAsync(ro, desc->row_block_offsets, nr * 4, cudaMemcpyDeviceToDevice, st)) ||
          !cuda_ok(cudaMemcpyAsync(co, desc->col_block_offsets, nc * 4, cudaMemcpyDeviceToDevice, st)))
        return fail(LCA_ERR_CUDA);
      m.row_off = ro;
      m.col_off = co;
    }
  }

  PlanDev& d = p->dev;
  d.tile_q = tile_q;
  d.tile_k = tile_k;
  d.n_qt = n_qt;
  d.n_kt = n_kt;
  d.map_heads = hm_n;
  const int n_rows = hm_n * n_qt, n_cols = hm_n * n_kt;
  uint8_t* cls = p->alloc<uint8_t>(static_cast<size_t>(n_rows) * n_kt);
  int32_t* rowlen = p->alloc<int32_t>(n_rows);
  int32_t* rowptr = p->alloc<int32_t>(n_rows + 1);
  int32_t* collen = p->alloc<int32_t>(n_cols);
  int32_t* colptr = p->alloc<int32_t>(n_cols + 1);
  int32_t* work_q = p->alloc<int32_t>(n_rows);
  int32_t* work_k = p->alloc<int32_t>(n_cols);
  unsigned long long* counters = p->alloc<unsigned long long>(hm_n + 1);
  p->fwd_counters = p->alloc<unsigned int>(kFwdCounters);
  if (!cls || !rowlen || !rowptr || !collen || !colptr || !work_q || !work_k || !counters ||
      !p->fwd_counters)
    return fail(LCA_ERR_OOM);
  p->n_valid = counters;
  if (!cuda_ok(cudaMemsetAsync(counters, 0, (hm_n + 1) * sizeof(unsigned long long), st)))
    return fail(LCA_ERR_CUDA);

  {
    ProfScope ps(K_CLASSIFY, st);
    if (!cuda_ok(launch_classify(m, tile_q, tile_k, n_qt, n_kt, cls, rowlen, counters,
                                 counters + hm_n, st)))
      return fail(LCA_ERR_CUDA);
  }
  {
    ProfScope ps(K_SCAN, st);
    if (!cuda_ok(launch_scan(rowlen, n_rows, rowptr, st))) return fail(LCA_ERR_CUDA);
  }
  {
    ProfScope ps(K_COLLEN, st);
    if (!cuda_ok(launch_collen(cls, hm_n, n_qt, n_kt, collen, st))) return fail(LCA_ERR_CUDA);
  }
  {
    ProfScope ps(K_SCAN, st);
    if (!cuda_ok(launch_scan(collen, n_cols, colptr, st))) return fail(LCA_ERR_CUDA);
  }

  int32_t nnz = 0;
  unsigned long long n_partial = 0;
  if (!cuda_ok(cudaMemcpyAsync(&nnz, rowptr + n_rows, sizeof(int32_t), cudaMemcpyDeviceToHost, st)) ||
      !cuda_ok(cudaMemcpyAsync(&n_partial, counters + hm_n, sizeof(n_partial),
                               cudaMemcpyDeviceToHost, st)) ||
      !cuda_ok(cudaStreamSynchronize(st)))
    return fail(LCA_ERR_CUDA);

  int32_t* kt_idx = p->alloc<int32_t>(nnz);
  uint8_t* kt_cls = p->alloc<uint8_t>(nnz);
  int32_t* qt_idx = p->alloc<int32_t>(nnz);
  uint8_t* qt_cls = p->alloc<uint8_t>(nnz);
  if (!kt_idx || !kt_cls || !qt_idx || !qt_cls) return fail(LCA_ERR_OOM);
  {
    ProfScope ps(K_FILL, st, 2);
    if (!cuda_ok(launch_fill(cls, hm_n, n_qt, n_kt, rowptr, kt_idx, kt_cls, colptr, qt_idx,
                             qt_cls, st)))
      return fail(LCA_ERR_CUDA);
  }
  {
    ProfScope ps(K_LPT, st);
    if (!cuda_ok(launch_lpt(rowptr, n_rows, n_kt, work_q, colptr, n_cols, n_qt, work_k, st)))
      return fail(LCA_ERR_CUDA);
  }

  d.cls = cls;
  d.rowptr = rowptr;
  d.kt_idx = kt_idx;
  d.kt_cls = kt_cls;
  d.colptr = colptr;
  d.qt_idx = qt_idx;
  d.qt_cls = qt_cls;
  d.work_q = work_q;
  d.work_k = work_k;

  lca_plan_info& info = p->info;
  info.seqlen = S;
  info.tile_q = tile_q;
  info.tile_k = tile_k;
  info.n_qt = n_qt;
  info.n_kt = n_kt;
  info.map_heads = hm_n;
  info.mask_type = t;
  info.nnz = nnz;
  info.n_partial = static_cast<int64_t>(n_partial);
  *out = p;
  return LCA_OK;
}

lca_status lca_plan_get_info(const lca_plan* plan, lca_plan_info* info) {
  if (!plan || !info) return LCA_ERR_INVALID_ARG;
  *info = plan->info;
  info->device_bytes = static_cast<int64_t>(plan->bytes);
  return LCA_OK;
}

lca_status lca_plan_export(const lca_plan* p, uint8_t* cls, int32_t* rowptr, int32_t* kt_idx,
                           uint8_t* kt_cls, int32_t* colptr, int32_t* qt_idx, uint8_t* qt_cls,
                           int32_t* work_q, int32_t* work_k, int64_t* n_valid) {
  if (!p) return LCA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return LCA_ERR_CUDA;
  const lca_plan_info& in = p->info;
  const size_t n_rows = static_cast<size_t>(in.map_heads) * in.n_qt;
  const size_t n_cols = static_cast<size_t>(in.map_heads) * in.n_kt;
  const size_t nnz = static_cast<size_t>(in.nnz);
  struct Item { void* dst; const void* src; size_t bytes; } items[] = {
      {cls, p->dev.cls, n_rows * in.n_kt},
      {rowptr, p->dev.rowptr, (n_rows + 1) * 4},
      {kt_idx, p->dev.kt_idx, nnz * 4},
      {kt_cls, p->dev.kt_cls, nnz},
      {colptr, p->dev.colptr, (n_cols + 1) * 4},
      {qt_idx, p->dev.qt_idx, nnz * 4},
      {qt_cls, p->dev.qt_cls, nnz},
      {work_q, p->dev.work_q, n_rows * 4},
      {work_k, p->dev.work_k, n_cols * 4},
      {n_valid, p->n_valid, static_cast<size_t>(in.map_heads) * 8},
  };
  for (const Item& it : items) {
    if (!it.dst || it.bytes == 0) continue;
    if (cudaMemcpy(it.dst, it.src, it.bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
      return LCA_ERR_CUDA;
  }
  return LCA_OK;
}

void lca_plan_destroy(lca_plan* plan) { delete plan; }

}  // extern "C"

namespace {

lca_status check_shape(const lca_plan* p, const lca_shape* s) {
  if (!p || !s) return LCA_ERR_INVALID_ARG;
  if (s->batch < 1 || s->seqlen < 1 || s->h_q < 1 || s->h_kv < 1 || s->head_dim < 1)
    return LCA_ERR_INVALID_ARG;
  if (s->h_q % s->h_kv != 0) return LCA_ERR_INVALID_ARG;
  if (s->head_dim != 128 && s->head_dim != 64) return LCA_ERR_UNSUPPORTED;
  const int64_t q_min = static_cast<int64_t>(s->h_q) * s->head_dim;
  const int64_t k_min = static_cast<int64_t>(s->h_kv) * s->head_dim;
  if (s->q_row_stride < q_min || s->o_row_stride < q_min || s->k_row_stride < k_min ||
      s->v_row_stride < k_min)
    return LCA_ERR_INVALID_ARG;
  if ((s->q_row_stride | s->o_row_stride | s->k_row_stride | s->v_row_stride) & 7)
    return LCA_ERR_INVALID_ARG;
  const lca_plan_info& in = p->info;
  if (in.seqlen != s->seqlen) return LCA_ERR_PLAN_MISMATCH;
  if (in.map_heads != 1 && in.map_heads != s->h_kv && in.map_heads != s->h_q)
    return LCA_ERR_PLAN_MISMATCH;
  const bool batched_ok = p->mask.num_segments == 0 && !is_sparse_type(in.mask_type);
  if (s->batch > 1 && !batched_ok) return LCA_ERR_UNSUPPORTED;
  if (in.tile_q != 128 || in.tile_k != 128) return LCA_ERR_UNSUPPORTED;
  return LCA_OK;
}

int64_t padded_seqlen(int seqlen) { return (static_cast<int64_t>(seqlen) + 127) / 128 * 128; }

// Row strides of dO, dQ, dK, dV: 0 takes the matching input's (dO as O, dQ as Q, dK as
// K, dV as V); each must cover its heads and be a multiple of 8 elements.
struct GradStrides { int64_t dout, dq, dk, dv; };

lca_status grad_strides(const lca_shape* s, GradStrides* g) {
  g->dout = s->do_row_stride ? s->do_row_stride : s->o_row_stride;
  g->dq = s->dq_row_stride ? s->dq_row_stride : s->q_row_stride;
  g->dk = s->dk_row_stride ? s->dk_row_stride : s->k_row_stride;
  g->dv = s->dv_row_stride ? s->dv_row_stride : s->v_row_stride;
  const int64_t q_min = static_cast<int64_t>(s->h_q) * s->head_dim;
  const int64_t k_min = static_cast<int64_t>(s->h_kv) * s->head_dim;
  if (g->dout < q_min || g->dq < q_min || g->dk < k_min || g->dv < k_min)
    return LCA_ERR_INVALID_ARG;
  if ((g->dout | g->dq | g->dk | g->dv) & 7) return LCA_ERR_INVALID_ARG;
  return LCA_OK;
}

AttnDims make_dims(const lca_plan* p, const lca_shape* s, float softmax_scale) {
  AttnDims d;
  d.batch = s->batch;
  d.seqlen = s->seqlen;
  d.h_q = s->h_q;
  d.h_kv = s->h_kv;
  d.group = s->h_q / s->h_kv;
  d.heads_per_map = s->h_q / p->info.map_heads;
  d.kv_per_map = p->info.map_heads <= s->h_kv ? s->h_kv / p->info.map_heads : 0;
  d.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(s->head_dim));
  d.scale_log2 = d.scale * 1.4426950408889634f;
  d.head_dim = s->head_dim;
  // 16 consecutive work items per launch-order group: MHA kernels then share K/V
  // (Q/dO) tiles in L2 across the resident CTAs; GQA is indifferent to it.
  d.chunk = 16;
  return d;
}

}  // namespace

extern "C" {

lca_status lca_attn_fwd(const lca_plan* plan, const lca_shape* shape, const void* q,
                        const void* k, const void* v, void* o, float* lse, float softmax_scale,
                        void* stream) {
  lca_status s = check_shape(plan, shape);
  if (s != LCA_OK) return s;
  if (!q || !k || !v || !o || !lse) return LCA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return LCA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bshd(&tq, q, shape->batch, shape->seqlen, shape->h_q, shape->q_row_stride, 128, shape->head_dim) ||
      !make_tmap_bshd(&tk, k, shape->batch, shape->seqlen, shape->h_kv, shape->k_row_stride, 128, shape->head_dim) ||
      !make_tmap_bshd(&tv, v, shape->batch, shape->seqlen, shape->h_kv, shape->v_row_stride, 128, shape->head_dim))
    return LCA_ERR_CUDA;
  FwdArgs a;
  a.dims = make_dims(plan, shape, softmax_scale);
  a.plan = plan->dev;
  a.mask = plan->mask;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.o_row_stride = shape->o_row_stride;
  a.err = device_error_ptr();
  a.timeout_ns = g_timeout_ns.load();
  if (!a.err) return LCA_ERR_CUDA;
  a.n_units = plan->info.n_qt * shape->h_q * shape->batch;
  lca_plan* mp = const_cast<lca_plan*>(plan);
  a.unit_counter = mp->fwd_counters + (mp->fwd_next.fetch_add(1) % kFwdCounters);
  const int sms = sm_count();
  if (sms <= 0) return LCA_ERR_CUDA;
  const int n_ctas = a.n_units < sms ? a.n_units : sms;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope ps(K_FWD, st);
  return launch_attn_fwd(tq, tk, tv, a, n_ctas, st) == cudaSuccess ? LCA_OK : LCA_ERR_CUDA;
}

size_t lca_attn_bwd_workspace(const lca_plan* plan, const lca_shape* shape, int flags) {
  (void)flags;
  if (!plan || !shape || shape->batch < 1 || shape->h_q < 1 || shape->seqlen < 1) return 0;
  // LSE2 and D rows, each padded to whole 128-row tiles
  return 2 * static_cast<size_t>(shape->batch) * shape->h_q * padded_seqlen(shape->seqlen) *
         sizeof(float);
}

lca_status lca_attn_bwd(const lca_plan* plan, const lca_shape* shape, const void* q,
                        const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, void* workspace,
                        size_t ws_bytes, float softmax_scale, int flags, void* stream) {
  lca_status s = check_shape(plan, shape);
  if (s != LCA_OK) return s;
  if (flags != 0) return LCA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return LCA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return LCA_ERR_INVALID_ARG;
  if (ws_bytes < lca_attn_bwd_workspace(plan, shape, flags)) return LCA_ERR_INVALID_ARG;
  GradStrides gs;
  s = grad_strides(shape, &gs);
  if (s != LCA_OK) return s;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bshd(&tq, q, shape->batch, shape->seqlen, shape->h_q, shape->q_row_stride, 128, shape->head_dim) ||
      !make_tmap_bshd(&tk, k, shape->batch, shape->seqlen, shape->h_kv, shape->k_row_stride, 128, shape->head_dim) ||
      !make_tmap_bshd(&tv, v, shape->batch, shape->seqlen, shape->h_kv, shape->v_row_stride, 128, shape->head_dim) ||
      !make_tmap_bshd(&tdo, dout, shape->batch, shape->seqlen, shape->h_q, gs.dout, 128, shape->head_dim))
    return LCA_ERR_CUDA;
  BwdArgs a;
  a.dims = make_dims(plan, shape, softmax_scale);
  a.plan = plan->dev;
  a.mask = plan->mask;
  a.o = static_cast<const __nv_bfloat16*>(o);
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.lse = lse;
  a.s_pad = padded_seqlen(shape->seqlen);
  a.lse2 = static_cast<float*>(workspace);
  a.dsum = a.lse2 + static_cast<size_t>(shape->batch) * shape->h_q * a.s_pad;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.o_row_stride = shape->o_row_stride;
  a.do_row_stride = gs.dout;
  a.dq_row_stride = gs.dq;
  a.dk_row_stride = gs.dk;
  a.dv_row_stride = gs.dv;
  a.err = device_error_ptr();
  a.timeout_ns = g_timeout_ns.load();
  if (!a.err) return LCA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    ProfScope ps(K_BWD_PRE, st);
    if (launch_bwd_preprocess(a, st) != cudaSuccess) return LCA_ERR_CUDA;
  }
  {
    ProfScope ps(K_BWD, st);
    const int n_kv_blocks = plan->info.n_kt * shape->h_kv * shape->batch;
    const int n_q_blocks = plan->info.n_qt * shape->h_q * shape->batch;
    if (launch_bwd(tq, tk, tv, tdo, a, n_kv_blocks, n_q_blocks, st) != cudaSuccess)
      return LCA_ERR_CUDA;
  }
  return LCA_OK;
}

size_t lca_block_scores_workspace(const lca_shape* shape, int block, int map_heads) {
  if (!shape || block < 1 || shape->seqlen < 1 || map_heads < 1) return 0;
  const int n_b = (shape->seqlen + block - 1) / block;
  return block_scores_workspace_bytes(map_heads, n_b);
}

lca_status lca_block_scores(const lca_shape* shape, const void* q, const void* k, int block,
                            int map_heads, float softmax_scale, float* scores, void* workspace,
                            size_t ws_bytes, void* stream) {
  if (!shape || !q || !k || !scores || !workspace) return LCA_ERR_INVALID_ARG;
  if (shape->batch != 1 || shape->head_dim != 128 || shape->seqlen < 1 || shape->h_q < 1 ||
      shape->h_kv < 1 || shape->h_q % shape->h_kv != 0)
    return LCA_ERR_INVALID_ARG;
  if (block < 1 || block > shape->seqlen) return LCA_ERR_INVALID_ARG;
  if (map_heads != 1 && map_heads != shape->h_kv && map_heads != shape->h_q)
    return LCA_ERR_INVALID_ARG;
  if (shape->q_row_stride < shape->h_q * 128 || shape->k_row_stride < shape->h_kv * 128 ||
      shape->q_row_stride % 8 != 0 || shape->k_row_stride % 8 != 0)
    return LCA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, scores, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return LCA_ERR_INVALID_ARG;
  if (ws_bytes < lca_block_scores_workspace(shape, block, map_heads)) return LCA_ERR_INVALID_ARG;
  BlockScoreArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.q_row_stride = shape->q_row_stride;
  a.k_row_stride = shape->k_row_stride;
  a.seqlen = shape->seqlen;
  a.block = block;
  a.n_blocks = (shape->seqlen + block - 1) / block;
  a.map_heads = map_heads;
  a.heads_per_map = shape->h_q / map_heads;
  a.group = shape->h_q / shape->h_kv;
  a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(128.0f);
  a.pooled = static_cast<float*>(workspace);
  a.scores = scores;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope ps(K_BLOCK_SCORES, st);
  return launch_block_scores(a, st) == cudaSuccess ? LCA_OK : LCA_ERR_CUDA;
}

lca_status lca_block_topk(const float* scores, int map_heads, int n_rows, int n_cols, int k,
                          uint8_t* block_map, void* stream) {
  if (!scores || !block_map || map_heads < 1 || n_rows < 1 || n_cols < 1) return LCA_ERR_INVALID_ARG;
  if (k < 1 || k > n_cols) return LCA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(map_heads) * n_rows > INT32_MAX) return LCA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope ps(K_BLOCK_TOPK, st);
  return launch_block_topk(scores, map_heads * n_rows, n_cols, k, block_map, st) == cudaSuccess
             ? LCA_OK
             : LCA_ERR_CUDA;
}

lca_status lca_get_last_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LCA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return LCA_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return LCA_ERR_CUDA;
  if (v & LCA_DEVERR_TIMEOUT) return LCA_ERR_TIMEOUT;
  return v ? LCA_ERR_CUDA : LCA_OK;
}

lca_status lca_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
  lca_status s = lca_get_last_device_error(stream);
  if (s == LCA_ERR_CUDA) return s;
  unsigned int* err = device_error_ptr();
  if (!err) return LCA_ERR_CUDA;
  if (launch_selftest_wait(err, timeout_ns, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LCA_ERR_CUDA;
  return lca_get_last_device_error(stream);
}

lca_status lca_selftest_umma(int variant, const void* a, const void* b, float* c, void* stream) {
  if (variant < 0 || variant > 4 || !a || !b || !c) return LCA_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  if (!make_tmap_bshd(&ta, a, 1, 128, 1, 128, 128) || !make_tmap_bshd(&tb, b, 1, 128, 1, 128, 128))
    return LCA_ERR_CUDA;
  unsigned int* err = device_error_ptr();
  if (!err) return LCA_ERR_CUDA;
  if (launch_selftest_umma(variant, ta, tb, static_cast<const __nv_bfloat16*>(a), c, err,
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LCA_ERR_CUDA;
  return lca_get_last_device_error(stream);
}

}  // extern "C"
