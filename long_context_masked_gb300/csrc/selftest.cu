// Self-check kernels behind the lca_selftest_* entry points: the bounded mbarrier wait
// and single 128 x 128 x 128 tcgen05 GEMMs that exercise each operand layout the
// attention kernels use (TMA-loaded K-major and MN-major tiles, and a K-major tile
// written by threads in the 128-byte swizzle).
#include <cuda_runtime.h>

#include "attn_kernels.h"
#include "lca_device.cuh"

namespace lca {

namespace {

__global__ void selftest_wait_kernel(unsigned int* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtx w{&abort_flag, err, timeout_ns};
  mbar_wait(&bar, 0, w);  // nothing arrives on this barrier: the wait must give up
}

constexpr uint32_t T_BYTES = 128 * 128 * 2;
constexpr uint32_t T_HALF = T_BYTES / 2;

// variant 0: C = A B^T, A and B K-major via TMA
// variant 1: C = A B,   A K-major via TMA, B MN-major via TMA
// variant 2: C = A B,   A K-major written by threads (swizzled stores), B MN-major via TMA
// variant 3: C = A B,   A MN-major via TMA (memory holds A^T), B MN-major via TMA
// variant 4: C = A B,   A in TMEM (rows written by the threads as bf16 pairs with
//                       tcgen05.st), B MN-major via TMA
__global__ void __launch_bounds__(128, 1)
selftest_umma_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                     const __nv_bfloat16* a_rm, float* c, int variant, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + 2 * T_BYTES);
  uint64_t* done = full + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  int* abort_flag = reinterpret_cast<int*>(tslot + 1);
  const int t = threadIdx.x, warp = t >> 5;

  if (t == 0) {
    mbar_init(full, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);   // D: columns 0-127; A (variant 4): columns 128-191
    tmem_relinquish();
  }
  if (variant == 2) {
    const __nv_bfloat16* src = a_rm + t * 128;
    for (int hh = 0; hh < 2; ++hh)
      for (int u = 0; u < 8; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + hh * 64 + u * 8);
        st_shared_v4(base_u32 + hh * T_HALF + sw128_offset(t, u), v.x, v.y, v.z, v.w);
      }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  WaitCtx wc{abort_flag, err, 2000000000ull};
  if (variant == 4) {
    uint32_t r[64];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a_rm + t * 128);
    for (int x = 0; x < 64; ++x) r[x] = src[x];
    tmem_st64(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 128, r);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();

  if (t == 0) {
    const uint32_t bytes = (variant == 2 || variant == 4 ? 1u : 2u) * T_BYTES;
    mbar_arrive_expect_tx(full, bytes);
    for (int hh = 0; hh < 2; ++hh) {
      if (variant != 2 && variant != 4) tma_load_4d(base + hh * T_HALF, &ta, full, hh * 64, 0, 0, 0);
      tma_load_4d(base + T_BYTES + hh * T_HALF, &tb, full, hh * 64, 0, 0, 0);
    }
    mbar_wait(full, 0, wc);
    tc_fence_after();
    const int a_mn = variant == 3 ? 1 : 0;
    const int b_mn = variant == 0 ? 0 : 1;
    const uint32_t idesc = idesc_bf16(128, 128, a_mn, b_mn);
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t ad = a_mn ? desc_mnmajor(base_u32, kk, T_HALF) : desc_kmajor(base_u32, kk, T_HALF);
      const uint64_t bd = b_mn ? desc_mnmajor(base_u32 + T_BYTES, kk, T_HALF)
                               : desc_kmajor(base_u32 + T_BYTES, kk, T_HALF);
      if (variant == 4)
        umma_bf16_ts(tmem, tmem + 128 + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
      else
        umma_bf16_ss(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
    }
    umma_commit(done);
  }
  __syncwarp();
  mbar_wait(done, 0, wc);
  __syncwarp();
  tc_fence_after();
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t r[32];
    tmem_ld32(lane_addr + cc * 32, r);
    for (int x = 0; x < 32; ++x) c[t * 128 + cc * 32 + x] = __uint_as_float(r[x]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned int* err, uint64_t timeout_ns, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_selftest_umma(int variant, const CUtensorMap& ta, const CUtensorMap& tb,
                                 const __nv_bfloat16* a_rowmajor, float* c, unsigned int* err,
                                 cudaStream_t st) {
  const int smem = 2 * T_BYTES + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(selftest_umma_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  selftest_umma_kernel<<<1, 128, smem, st>>>(ta, tb, a_rowmajor, c, variant, err);
  return cudaGetLastError();
}

}  // namespace lca
