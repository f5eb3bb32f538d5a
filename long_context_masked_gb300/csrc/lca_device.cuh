// Device-side building blocks shared by the library's kernels: inline PTX for
// mbarriers, TMA tile loads and the 5th-generation tensor cores (tcgen05 MMA with
// TMEM accumulators), bounded waits, and the closed-form mask evaluation used by
// the mask builder and by the attention kernels on partial tiles.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "lca_types.h"

namespace lca {

// ------------------------------------------------------------------ misc

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t elect_lane0() { return (threadIdx.x & 31) == 0; }

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait state of one CTA: every wait is bounded by `timeout_ns`; the first wait that
// runs out raises the CTA's abort flag (shared memory) and the device error word, and
// every later wait of the CTA returns at once, so all threads drain to the end of the
// kernel instead of hanging.
struct WaitCtx {
  volatile int* abort;    // shared memory, 0 = running
  unsigned int* err;      // device error word
  uint64_t timeout_ns;
};

static __device__ __noinline__ void mbar_wait_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_test(bar, parity)) {
    if (*w.abort) return;
    if ((++spins & 15u) == 0 && globaltimer_ns() - t0 > w.timeout_ns) {
      *w.abort = 1;
      atomicOr(w.err, LCA_DEVERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ void mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (!mbar_test(bar, parity)) mbar_wait_slow(bar, parity, w);
}

// A last bounded wait that ignores the abort flag (used to let copies in flight land
// before the CTA exits).
static __device__ __noinline__ void mbar_wait_final(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

// ------------------------------------------------------------------ fences

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Barrier among `count` threads (a multiple of 32) of the CTA on hardware barrier `id`.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load (coordinates innermost first) completing on `bar` with byte count.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

// Untiled bulk copy of `bytes` from global to shared memory, completing on `bar` like
// a tensor load (both addresses 16-byte aligned, `bytes` a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch a 4-D tile into L2 (no shared memory, no completion tracking): issued a few
// steps ahead of the real load so that load hits in L2.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
// Bits: [0,14) start address >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte
// offset >> 4, [46,49) fixed 0b001, [61,64) swizzle mode (2 = 128-byte swizzle).
// Tiles are 1024-byte aligned so the base-offset field stays 0.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Descriptors of a 128-element-wide bf16 operand tile stored as two halves of 64
// elements (128 bytes) per row, each half 128-byte swizzled, `half_bytes` apart
// (rows * 128).  K-major: rows are M/N, the 128 elements are K; k-step kk (16
// elements) starts kk%4 * 32 bytes into half kk/4 (leading offset unused).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk, uint32_t half_bytes) {
  return sdesc_sw128(tile + (kk >> 2) * half_bytes + (kk & 3) * 32, 16, 1024);
}
// MN-major: rows are K, the 128 elements are M/N; the two halves are the leading-offset
// step along M/N and 8-row groups (1024 bytes) the stride-offset step along K; k-step kk
// starts 16 rows = 2048 bytes further.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk, uint32_t half_bytes) {
  return sdesc_sw128(tile + kk * 2048, half_bytes, 1024);
}

// The same descriptors as a base (k-step 0 of stage 0) plus constant increments, so an
// issuing thread builds each 64-bit descriptor once and steps it with an integer add:
// the start-address field is the low 14 bits in 16-byte units and shared-memory
// addresses stay below 2^18, so the increments never carry out of the field.
__host__ __device__ constexpr uint64_t kmajor_step(int kk, uint32_t half_bytes) {
  return ((kk >> 2) * half_bytes + (kk & 3) * 32) >> 4;
}
__host__ __device__ constexpr uint64_t mnmajor_step(int kk) { return (kk * 2048) >> 4; }
__host__ __device__ constexpr uint64_t stage_step(uint32_t bytes) { return bytes >> 4; }

// Instruction descriptor of kind::f16 with bf16 A/B and fp32 accumulation.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format,
// 15/16 A/B major (0 = K-major, 1 = MN-major), [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.  A (M = 128 rows) lives in
// TMEM: lane m holds row m, 32-bit column c holds the bf16 pair (k = 2c, 2c + 1), so
// a K = 16 step reads 8 columns starting at `a_tmem`.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

#define LCA_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                  "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define LCA_W8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                  "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

// 32 consecutive 32-bit TMEM columns of this thread's lane (lane = warp's quarter
// base + lane id), waiting for completion inside the same asm statement.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : LCA_R8(0), LCA_R8(8), LCA_R8(16), LCA_R8(24)
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      LCA_W8(0), LCA_W8(8), LCA_W8(16), LCA_W8(24)
      : "memory");
}

// 64 consecutive 32-bit TMEM columns of this thread's lane, waited on in the same
// asm statement.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

// Two 64-column loads (e.g. S and dP of the same rows) behind a single wait.
__device__ __forceinline__ void tmem_ld64x2(uint32_t ta, uint32_t tb, uint32_t (&a)[64],
                                            uint32_t (&b)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%129];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(a[32]), "=r"(a[33]), "=r"(a[34]), "=r"(a[35]), "=r"(a[36]), "=r"(a[37]), "=r"(a[38]), "=r"(a[39]), "=r"(a[40]), "=r"(a[41]), "=r"(a[42]), "=r"(a[43]), "=r"(a[44]), "=r"(a[45]), "=r"(a[46]), "=r"(a[47]), "=r"(a[48]), "=r"(a[49]), "=r"(a[50]), "=r"(a[51]), "=r"(a[52]), "=r"(a[53]), "=r"(a[54]), "=r"(a[55]), "=r"(a[56]), "=r"(a[57]), "=r"(a[58]), "=r"(a[59]), "=r"(a[60]), "=r"(a[61]), "=r"(a[62]), "=r"(a[63]),
        "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31]), "=r"(b[32]), "=r"(b[33]), "=r"(b[34]), "=r"(b[35]), "=r"(b[36]), "=r"(b[37]), "=r"(b[38]), "=r"(b[39]), "=r"(b[40]), "=r"(b[41]), "=r"(b[42]), "=r"(b[43]), "=r"(b[44]), "=r"(b[45]), "=r"(b[46]), "=r"(b[47]), "=r"(b[48]), "=r"(b[49]), "=r"(b[50]), "=r"(b[51]), "=r"(b[52]), "=r"(b[53]), "=r"(b[54]), "=r"(b[55]), "=r"(b[56]), "=r"(b[57]), "=r"(b[58]), "=r"(b[59]), "=r"(b[60]), "=r"(b[61]), "=r"(b[62]), "=r"(b[63])
      : "r"(ta), "r"(tb)
      : "memory");
}

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}

#undef LCA_R8
#undef LCA_W8

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Byte offset of the 16-byte unit `u` (0..7) of row `r` inside a [rows][64] bf16 tile
// stored with the 128-byte swizzle (the layout TMA writes for a 128-byte-wide box).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t u) {
  return r * 128u + ((u ^ (r & 7u)) << 4);
}

// ------------------------------------------------------------------ masks

// Launch order of the per-head CTAs of a work list.  CTA blk maps to work item `item`
// (an index into the longest-first list) and replica `rem` (query or KV head within
// the map head, times batch).  The replicas of `chunk` consecutive items are
// interleaved item-fastest, so the CTAs resident at one time cover several items of
// the same head: for MHA they then stream the same K/V (or Q/dO) tiles together and
// share them in L2, where head-fastest order would give every CTA its own stream.
__device__ __forceinline__ void chunked_item(int blk, int per_item, int n_items, int chunk,
                                             int& item, int& rem) {
  const int span = chunk * per_item;
  const int c = blk / span;
  const int first = c * chunk;
  const int cn = min(chunk, n_items - first);
  const int w = blk - c * span;
  item = first + w % cn;
  rem = w / cn;
}

// Index s of the segment [cu[s], cu[s+1]) holding x, for 0 <= x < cu[n].
__device__ __forceinline__ int seg_find(const int32_t* cu, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// seg_find for an ascending x sequence: starts at `hint` (any index; the answer from
// the previous, smaller x) and gallops upward, so a cursor that moves by a few blocks
// costs a few loads.  Falls back to the full search when the hint is past x.
__device__ __forceinline__ int seg_find_from(const int32_t* cu, int n, int hint, int x) {
  if (hint < 0 || hint >= n || __ldg(cu + hint) > x) return seg_find(cu, n, x);
  int lo = hint, step = 1;
  while (lo + step <= n - 1 && __ldg(cu + lo + step) <= x) {
    lo += step;
    step <<= 1;
  }
  int hi = min(n - 1, lo + step - 1);
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Tile bytes of the plan (class in bits 0-1, empty-half flags in bits 2-5) and the
// entries of its row and column lists.
__host__ __device__ __forceinline__ uint8_t row_list_byte(uint8_t c) {
  return static_cast<uint8_t>(c & (LCA_TILE_CLASS_MASK | LCA_TILE_KEY_HALF0_EMPTY |
                                   LCA_TILE_KEY_HALF1_EMPTY));
}
__host__ __device__ __forceinline__ uint8_t col_list_byte(uint8_t c) {
  return static_cast<uint8_t>((c & LCA_TILE_CLASS_MASK) | ((c >> 4) << 2));
}
// Empty halves of a list entry: bit 0 the first half, bit 1 the second (key columns
// in a row list, query rows in a column list).
__device__ __forceinline__ int entry_empty_halves(int e) { return (e >> 2) & 3; }
__device__ __forceinline__ int entry_class(int e) { return e & LCA_TILE_CLASS_MASK; }
// Both empty-half flags of a list entry (bits 2-3 in row and column lists alike).
constexpr int kEntryHalfFlags = LCA_TILE_KEY_HALF0_EMPTY | LCA_TILE_KEY_HALF1_EMPTY;

// Whether a list of n plan entries runs the half-width path: it is long (at least 64
// entries) and at least 1/share of its entries flag an empty half.  The flag-aware loops
// cost a few percent per tile over the plain ones, and short lists are bound by load
// and MMA round-trip latency, where half-width tiles were measured slower; other lists
// run the plain loops (which treat a flagged tile as a partial full-width one).  The
// forward passes share 4, the backward kernels (whose half-width tiles save less) 2.
// The MMA issuer and the softmax warps of a CTA decide alike.
__device__ __forceinline__ bool half_path(int flagged, int n, int share) {
  return n >= 64 && share * flagged >= n;
}
// half_path over the n entries at e.  Warp-wide: every lane calls it and gets the same
// answer.
__device__ __forceinline__ bool use_half_path(const uint8_t* e, int n, int share, int lane) {
  int f = 0;
  for (int x = lane; x < n; x += 32) f += (__ldg(e + x) & kEntryHalfFlags) != 0;
  return half_path(__reduce_add_sync(0xFFFFFFFFu, f), n, share);
}

// Per-thread search hints of the variable block-sparse map: the row block of the last
// row and the column block of the last column window looked up.  Only speed depends
// on them; start them at -1.
struct MapCursor { int rb = -1, cb = -1; };

// Allowed keys of query row i as two disjoint half-open intervals inside [0, S):
// [a0, b0) and [a1, b1) (either may be empty).  Block-sparse masks return their base
// interval (documents / causal), which the block map further restricts.
struct RowSpan { int a0, b0, a1, b1; };

__device__ __forceinline__ RowSpan row_span(const MaskDev& m, int i) {
  RowSpan r{0, 0, 0, 0};
  const int S = m.seqlen;
  switch (m.type) {
    case LCA_FULL: r.b0 = S; break;
    case LCA_CAUSAL: r.b0 = i + 1; break;
    case LCA_SLIDING_WINDOW: r.a0 = max(0, i - m.window + 1); r.b0 = i + 1; break;
    case LCA_FULL_DOCUMENT: {
      const int d = seg_find(m.cu, m.num_segments, i);
      r.a0 = __ldg(m.cu + d); r.b0 = __ldg(m.cu + d + 1);
    } break;
    case LCA_CAUSAL_DOCUMENT: {
      const int d = seg_find(m.cu, m.num_segments, i);
      r.a0 = __ldg(m.cu + d); r.b0 = i + 1;
    } break;
    case LCA_SLIDING_WINDOW_DOCUMENT: {
      const int d = seg_find(m.cu, m.num_segments, i);
      r.a0 = max(__ldg(m.cu + d), i - m.window + 1); r.b0 = i + 1;
    } break;
    case LCA_PREFIX_LM: r.b0 = min(S, max(m.prefix_len, i + 1)); break;
    case LCA_SHARED_QUESTION: {
      const int s = seg_find(m.cu, m.num_segments, i);
      if (s == 0) {
        r.b0 = i + 1;
      } else {
        r.b0 = __ldg(m.cu + 1);
        r.a1 = __ldg(m.cu + s); r.b1 = i + 1;
      }
    } break;
    case LCA_GLOBAL_SLIDING: {
      if (m.base_causal) {
        const int g = min(m.num_global, i + 1);
        const int wlo = max(0, i - m.window + 1);
        if (wlo <= g) { r.b0 = i + 1; }
        else { r.b0 = g; r.a1 = wlo; r.b1 = i + 1; }
      } else if (i < m.num_global) {
        r.b0 = S;
      } else {
        const int g = min(m.num_global, S);
        const int wlo = max(0, i - m.window + 1);
        const int whi = static_cast<int>(min(static_cast<long long>(S),
                                             static_cast<long long>(i) + m.window));
        if (wlo <= g) { r.b0 = whi; }
        else { r.b0 = g; r.a1 = wlo; r.b1 = whi; }
      }
    } break;
    case LCA_CAUSAL_BLOCKWISE:
      r.b0 = static_cast<int>(min(static_cast<long long>(S),
                                  (static_cast<long long>(i / m.block) + 1) * m.block));
      break;
    case LCA_BLOCK_CAUSAL_DOCUMENT: {
      const int d = seg_find(m.cu, m.num_segments, i);
      const int st = __ldg(m.cu + d), en = __ldg(m.cu + d + 1);
      r.a0 = st;
      r.b0 = static_cast<int>(min(static_cast<long long>(en),
                                  st + (static_cast<long long>((i - st) / m.block) + 1) * m.block));
    } break;
    default: {  // block-sparse base
      int lo = 0, hi = S;
      if (m.num_segments > 0) {
        const int d = seg_find(m.cu, m.num_segments, i);
        lo = __ldg(m.cu + d); hi = __ldg(m.cu + d + 1);
      }
      if (m.base_causal) hi = min(hi, i + 1);
      r.a0 = lo; r.b0 = hi;
    } break;
  }
  if (r.b0 < r.a0) r.b0 = r.a0;
  if (r.b1 < r.a1) r.b1 = r.a1;
  return r;
}

// Allowed queries of key column j as two disjoint half-open intervals inside [0, S):
// the column view of row_span, for kernels whose threads own key rows.  Block-sparse
// masks return their base interval (documents / causal), which the block map further
// restricts.
__device__ __forceinline__ RowSpan col_span(const MaskDev& m, int j) {
  RowSpan r{0, 0, 0, 0};
  const int S = m.seqlen;
  const auto clip = [S](long long x) { return static_cast<int>(min(static_cast<long long>(S), x)); };
  switch (m.type) {
    case LCA_FULL: r.b0 = S; break;
    case LCA_CAUSAL: r.a0 = j; r.b0 = S; break;
    case LCA_SLIDING_WINDOW:  // j <= i < j + w
      r.a0 = j; r.b0 = clip(static_cast<long long>(j) + m.window);
      break;
    case LCA_FULL_DOCUMENT: {
      const int d = seg_find(m.cu, m.num_segments, j);
      r.a0 = __ldg(m.cu + d); r.b0 = __ldg(m.cu + d + 1);
    } break;
    case LCA_CAUSAL_DOCUMENT: {
      const int d = seg_find(m.cu, m.num_segments, j);
      r.a0 = j; r.b0 = __ldg(m.cu + d + 1);
    } break;
    case LCA_SLIDING_WINDOW_DOCUMENT: {   // j <= i < min(end of doc(j), j + w)
      const int d = seg_find(m.cu, m.num_segments, j);
      r.a0 = j;
      r.b0 = static_cast<int>(min(static_cast<long long>(__ldg(m.cu + d + 1)),
                                  static_cast<long long>(j) + m.window));
    } break;
    case LCA_PREFIX_LM:       // prefix keys are seen by every query
      r.a0 = j < m.prefix_len ? 0 : j; r.b0 = S;
      break;
    case LCA_SHARED_QUESTION: {
      const int s = seg_find(m.cu, m.num_segments, j);
      r.a0 = j;               // question keys: every later query; answer keys: own answer
      r.b0 = s == 0 ? S : __ldg(m.cu + s + 1);
    } break;
    case LCA_GLOBAL_SLIDING: {
      if (m.base_causal) {
        r.a0 = j;
        r.b0 = j < m.num_global ? S : clip(static_cast<long long>(j) + m.window);
      } else if (j < m.num_global) {
        r.b0 = S;
      } else {                // global queries, plus the symmetric window |i - j| < w
        const int g = min(m.num_global, S);
        const int wlo = max(0, j - m.window + 1);
        const int whi = clip(static_cast<long long>(j) + m.window);
        if (wlo <= g) { r.b0 = whi; }
        else { r.b0 = g; r.a1 = wlo; r.b1 = whi; }
      }
    } break;
    case LCA_CAUSAL_BLOCKWISE:
      r.a0 = (j / m.block) * m.block; r.b0 = S;
      break;
    case LCA_BLOCK_CAUSAL_DOCUMENT: {
      const int d = seg_find(m.cu, m.num_segments, j);
      const int st = __ldg(m.cu + d);
      r.a0 = st + ((j - st) / m.block) * m.block; r.b0 = __ldg(m.cu + d + 1);
    } break;
    default: {  // block-sparse base
      int lo = 0, hi = S;
      if (m.num_segments > 0) {
        const int d = seg_find(m.cu, m.num_segments, j);
        lo = __ldg(m.cu + d); hi = __ldg(m.cu + d + 1);
      }
      r.a0 = m.base_causal ? max(lo, j) : lo; r.b0 = hi;
    } break;
  }
  if (r.b0 < r.a0) r.b0 = r.a0;
  if (r.b1 < r.a1) r.b1 = r.a1;
  return r;
}

__device__ __forceinline__ bool is_sparse(int type) {
  return type == LCA_BLOCK_SPARSE_UNIFORM || type == LCA_BLOCK_SPARSE_VARIABLE;
}

// Bits of the columns [lo, hi) that fall into the 32 columns starting at ws.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int ws) {
  const int a = max(lo - ws, 0);
  const int b = min(hi - ws, 32);
  if (b <= a) return 0u;
  const uint32_t upper = (b >= 32) ? 0xFFFFFFFFu : ((1u << b) - 1u);
  const uint32_t lower = (1u << a) - 1u;
  return upper & ~lower;
}

// Allowed-key bits of row i over the NW*32 columns starting at c0 (bit c of word w =
// column c0 + 32w + c).  Columns >= S are never allowed.
template <int NW>
__device__ __forceinline__ void row_tile_bits(const MaskDev& m, int h_m, int i, int c0,
                                              const RowSpan& sp, uint32_t (&bits)[NW],
                                              MapCursor* cur = nullptr) {
#pragma unroll
  for (int w = 0; w < NW; ++w)
    bits[w] = range_bits(sp.a0, sp.b0, c0 + 32 * w) | range_bits(sp.a1, sp.b1, c0 + 32 * w);
  if (!is_sparse(m.type)) return;
  uint32_t mb[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) mb[w] = 0u;
  const int c1 = min(c0 + NW * 32, m.seqlen);
  if (m.type == LCA_BLOCK_SPARSE_UNIFORM) {
    const int rb = i / m.block;
    const uint8_t* row = m.bmap + (static_cast<size_t>(h_m) * m.n_rb + rb) * m.n_cb;
    for (int cb = c0 / m.block; cb * m.block < c1; ++cb) {
      if (__ldg(row + cb)) {
        const int lo = cb * m.block, hi = lo + m.block;
#pragma unroll
        for (int w = 0; w < NW; ++w) mb[w] |= range_bits(lo, hi, c0 + 32 * w);
      }
    }
  } else {
    const int32_t* ro = m.row_off + static_cast<size_t>(h_m) * (m.n_rb + 1);
    const int32_t* co = m.col_off + static_cast<size_t>(h_m) * (m.n_cb + 1);
    int rb, cb0;
    if (cur != nullptr) {
      rb = cur->rb = seg_find_from(ro, m.n_rb, cur->rb, i);
      cb0 = cur->cb = seg_find_from(co, m.n_cb, cur->cb, c0);
    } else {
      rb = seg_find(ro, m.n_rb, i);
      cb0 = seg_find(co, m.n_cb, c0);
    }
    const uint8_t* row = m.bmap + (static_cast<size_t>(h_m) * m.n_rb + rb) * m.n_cb;
    for (int cb = cb0; cb < m.n_cb; ++cb) {
      const int lo = __ldg(co + cb);
      if (lo >= c1) break;
      if (__ldg(row + cb)) {
        const int hi = __ldg(co + cb + 1);
#pragma unroll
        for (int w = 0; w < NW; ++w) mb[w] |= range_bits(lo, hi, c0 + 32 * w);
      }
    }
  }
#pragma unroll
  for (int w = 0; w < NW; ++w) bits[w] &= mb[w];
}

// Allowed-query bits of key column j over the NW*32 queries starting at r0 (bit r of
// word w = query r0 + 32w + r), from the column span `sp` and, for the sparse masks,
// the block map's column of j.  Queries >= S are never allowed.
template <int NW>
__device__ __forceinline__ void col_tile_bits(const MaskDev& m, int h_m, int j, int r0,
                                              const RowSpan& sp, uint32_t (&bits)[NW],
                                              MapCursor* cur) {
#pragma unroll
  for (int w = 0; w < NW; ++w)
    bits[w] = range_bits(sp.a0, sp.b0, r0 + 32 * w) | range_bits(sp.a1, sp.b1, r0 + 32 * w);
  if (!is_sparse(m.type)) return;
  uint32_t mb[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) mb[w] = 0u;
  const int r1 = min(r0 + NW * 32, m.seqlen);
  const uint8_t* map = m.bmap + static_cast<size_t>(h_m) * m.n_rb * m.n_cb;
  if (m.type == LCA_BLOCK_SPARSE_UNIFORM) {
    const int cb = j / m.block;
    for (int rb = r0 / m.block; rb * m.block < r1; ++rb) {
      if (__ldg(map + static_cast<size_t>(rb) * m.n_cb + cb)) {
        const int lo = rb * m.block, hi = lo + m.block;
#pragma unroll
        for (int w = 0; w < NW; ++w) mb[w] |= range_bits(lo, hi, r0 + 32 * w);
      }
    }
  } else {
    const int32_t* ro = m.row_off + static_cast<size_t>(h_m) * (m.n_rb + 1);
    const int32_t* co = m.col_off + static_cast<size_t>(h_m) * (m.n_cb + 1);
    const int cb = cur->cb = seg_find_from(co, m.n_cb, cur->cb, j);
    const int rb0 = cur->rb = seg_find_from(ro, m.n_rb, cur->rb, r0);
    for (int rb = rb0; rb < m.n_rb; ++rb) {
      const int lo = __ldg(ro + rb);
      if (lo >= r1) break;
      if (__ldg(map + static_cast<size_t>(rb) * m.n_cb + cb)) {
        const int hi = __ldg(ro + rb + 1);
#pragma unroll
        for (int w = 0; w < NW; ++w) mb[w] |= range_bits(lo, hi, r0 + 32 * w);
      }
    }
  }
#pragma unroll
  for (int w = 0; w < NW; ++w) bits[w] &= mb[w];
}

}  // namespace lca
