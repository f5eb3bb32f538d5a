// lca_attn_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.
//
// lca_attn_bwd needs a caller-provided workspace (per-row LSE*log2(e) and
// D = rowsum(dO * O), fp32, rows padded to whole 128-row tiles).  Some callers cannot
// call cudaMalloc at that point: code under a caching or pooled allocator that forbids
// allocations outside its pool, runtimes that hand out only the tensors of the op
// itself, or programs that reserve all device memory when they start.  This entry point takes the workspace from a
// fixed buffer compiled into the library instead, and otherwise runs exactly the
// lca_attn_bwd path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/lca.h"

namespace {

// Capacity of the built-in workspace: two fp32 values for each of 2^23 padded rows
// (batch * h_q * seqlen rounded up to 128), 64 MiB.
constexpr size_t kScratchFloats = size_t(1) << 24;

// The buffer lives in every GPU that loads the library, for the life of the process.
static __device__ __align__(256) float g_bwd_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;

// The device address of g_bwd_scratch, remembered per device together with the CUDA
// context it was looked up in: a context torn down and re-created (cudaDeviceReset)
// reloads the module, and the buffer may then sit at another address.
struct ScratchAddr {
  float* ptr = nullptr;
  unsigned long long ctx_id = 0;   // 0: unknown, look the address up again
};
std::mutex g_mu;
ScratchAddr g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Unique id of the calling thread's current context (false if there is none yet or the
// driver does not report one).
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// Device address of g_bwd_scratch on the current device.  In host code the symbol name
// is only a host-side handle, never a device address, so the address is asked of the
// runtime (with the device current) the first time and again whenever the context
// changed.
lca_status scratch_on_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LCA_ERR_CUDA;
  unsigned long long ctx = 0;
  const bool known = current_context_id(&ctx);
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& e = g_scratch[dev];
  if (!e.ptr || !known || e.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return LCA_ERR_CUDA;
    e.ptr = static_cast<float*>(p);
    e.ctx_id = 0;
    if (current_context_id(&ctx)) e.ctx_id = ctx;   // the lookup made the context current
  }
  *out = e.ptr;
  return LCA_OK;
}

}  // namespace

extern "C" lca_status lca_attn_bwd_noalloc(const lca_plan* plan, const lca_shape* shape,
                                           const void* q, const void* k, const void* v,
                                           const void* o, const void* dout, const float* lse,
                                           void* dq, void* dk, void* dv, float softmax_scale,
                                           void* stream) {
  if (!plan || !shape) return LCA_ERR_INVALID_ARG;
  if (shape->batch < 1 || shape->h_q < 1 || shape->seqlen < 1) return LCA_ERR_INVALID_ARG;
  if (lca_attn_bwd_workspace(plan, shape, 0) > kScratchFloats * sizeof(float))
    return LCA_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  lca_status s = scratch_on_current_device(&scratch);
  if (s != LCA_OK) return s;
  return lca_attn_bwd(plan, shape, q, k, v, o, dout, lse, dq, dk, dv, scratch,
                      kScratchFloats * sizeof(float), softmax_scale, 0, stream);
}
