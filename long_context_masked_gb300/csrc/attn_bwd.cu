// Backward pass of mask-aware exact softmax attention on sm_103a.
//
// The benchmark singles the backward pass out as the bottleneck of attention training
// ("Long-Context Attention Benchmark": summary page, TL;DR and section 3.2; reading note,
// key findings).  Given the forward's LSE, with P = exp(scale * Q K^T - LSE) under the
// mask and D = rowsum(dO * O):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dK = scale dS^T Q,  dQ = scale dS K.
// Deterministic and free of floating-point atomics, in two launches: the preprocess,
// then one launch whose first CTAs run the dK/dV pass and the rest the dQ pass (neither
// reads the other's output, so dQ CTAs fill the SMs the last dK/dV CTAs leave idle):
//   preprocess  D for every (b, h, i) row and LSE * log2(e), into padded workspace
//               rows (HBM-bound);
//   dK/dV       one CTA per (KV head, key tile), key rows on the TMEM lanes: loops over
//               the query tiles that attend to the key tile (the plan's transposed
//               lists) for every query head of the KV group, recomputing S^T and dP^T
//               with tcgen05, writing P^T and dS^T back into TMEM and accumulating dV
//               and dK there with TS MMAs;
//   dQ          one CTA per (query head, query tile), query rows on the TMEM lanes:
//               loops over the tile's key tiles, recomputing S, dP and dS and
//               accumulating dQ in TMEM; dO and dS live in TMEM (bf16 pairs) and feed
//               the dP and dQ MMAs from there.
// Warp roles as in the forward: warps 8 and 10 issue TMA loads, warp 9 owns TMEM and
// issues the MMAs, warps 0-7 (two threads per TMEM lane, 64 columns each) turn S/dP
// into P/dS.  Where a CTA walks at least 64 plan entries and at least half of them flag
// one half of their tile as empty (query rows for dK/dV, key columns for dQ), such a
// tile runs at half width: N = 64 recompute MMAs, half the k-steps of the accumulating MMAs, and the
// softmax warps of that half stay idle.
// All waits are bounded.
#include <cuda_runtime.h>

#include <type_traits>

#include "attn_kernels.h"
#include "lca_device.cuh"

namespace lca {

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr uint32_t HALF = BM * 64 * 2;   // one 128-byte-swizzled 64-column half, 16 KB
constexpr uint64_t ROWS64_STEP = (64 * 128) >> 4;   // descriptor step to row 64 of a half
constexpr float LOG2E = 1.4426950408889634f;
constexpr int HALF_SHARE = 2;   // half-width path: half of a list's entries flagged

// ------------------------------------------------------------------ preprocess

template <int HD>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(BwdArgs a) {
  constexpr int TPR = HD / 8;   // threads per row, 8 elements each
  // One TPR-thread group per (b, i, h) row of the padded workspace, h fastest so the O
  // and dO reads coalesce; rows i >= S only write the padding values.
  const int S = a.dims.seqlen, hq = a.dims.h_q;
  const int64_t rows = static_cast<int64_t>(a.dims.batch) * a.s_pad * hq;
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / TPR;
  const int part = threadIdx.x % TPR;
  const int h = static_cast<int>(r % hq);
  const int64_t bi = r / hq;
  const int64_t b = bi / a.s_pad, i = bi % a.s_pad;
  const bool live = r < rows && i < S;
  float acc = 0.f;
  if (live) {
    const int64_t off = (b * S + i) * a.o_row_stride + h * HD + part * 8;
    const int64_t goff = (b * S + i) * a.do_row_stride + h * HD + part * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(a.o + off);
    const uint4 gv = *reinterpret_cast<const uint4*>(a.dout + goff);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 of = __bfloat1622float2(o2[x]);
      const float2 gf = __bfloat1622float2(g2[x]);
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (part == 0 && r < rows) {
    const int64_t w = (b * hq + h) * a.s_pad + i;
    float l2 = INFINITY;
    if (live) {
      const float l = a.lse[(b * hq + h) * S + i];
      if (l != -INFINITY) l2 = l * LOG2E;
    }
    a.dsum[w] = acc;
    a.lse2[w] = l2;
  }
}

// ------------------------------------------------------------------ shared pieces

constexpr int KV_THREADS = 352;      // dK/dV: 8 softmax warps, Q producer, MMA issuer, dO producer
constexpr int DQ_THREADS = 352;      // dQ: the same plus a second producer warp
constexpr int SOFTMAX_THREADS = 256;
constexpr int WARP_PRODUCER = 8, WARP_MMA = 9, WARP_PRODUCER_2 = 10;

// Half a row (64 key columns) of dS = P (dP - D), P = exp2(s * scale_log2 - lse_log2)
// on allowed entries, packed to bf16 pairs.
__device__ __forceinline__ void ds_half(const uint32_t (&sr)[64], const uint32_t (&dr)[64],
                                        bool masked, const uint32_t (&bits)[2], float sl2,
                                        float lse2, float dsum, uint32_t (&dk)[32]) {
#pragma unroll
  for (int x = 0; x < 64; x += 2) {
    float p0 = ex2_approx(fmaf(__uint_as_float(sr[x]), sl2, -lse2));
    float p1 = ex2_approx(fmaf(__uint_as_float(sr[x + 1]), sl2, -lse2));
    if (masked) {
      if (!((bits[x >> 5] >> (x & 31)) & 1u)) p0 = 0.f;
      if (!((bits[x >> 5] >> ((x + 1) & 31)) & 1u)) p1 = 0.f;
    }
    dk[x / 2] = pack_bf16x2(p0 * (__uint_as_float(dr[x]) - dsum),
                            p1 * (__uint_as_float(dr[x + 1]) - dsum));
  }
}

// N consecutive 32-bit TMEM columns (N = 16, 32 or 64) of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 32 || N == 64, "32 or 64 columns");
  if constexpr (N == 64) tmem_ld64(taddr, r); else tmem_ld32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) {
    tmem_st32(taddr, r);
  } else {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
  }
}

// Read N fp32 accumulator columns of this thread's lane, scale, store N bf16.
template <int N>
__device__ __forceinline__ void store_acc_half(uint32_t taddr, bool have, float scale,
                                               __nv_bfloat16* dst, bool write) {
  uint32_t r[N];
  if (have) {
    tmem_ldn<N>(taddr, r);
  } else {
#pragma unroll
    for (int x = 0; x < N; ++x) r[x] = 0u;
  }
  if (write) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < N / 8; ++v) {
      const int x = v * 8;
      uint4 w;
      w.x = pack_bf16x2(__uint_as_float(r[x + 0]) * scale, __uint_as_float(r[x + 1]) * scale);
      w.y = pack_bf16x2(__uint_as_float(r[x + 2]) * scale, __uint_as_float(r[x + 3]) * scale);
      w.z = pack_bf16x2(__uint_as_float(r[x + 4]) * scale, __uint_as_float(r[x + 5]) * scale);
      w.w = pack_bf16x2(__uint_as_float(r[x + 6]) * scale, __uint_as_float(r[x + 7]) * scale);
      d4[v] = w;
    }
  }
}

// ------------------------------------------------------------------ dK / dV
//
// Key-major orientation: the CTA's 128 key rows are the TMEM lanes, so
//   S^T = K Q^T, dP^T = V dO^T           SS MMAs, both operands K-major, N = 128
//   P^T = exp2(S^T scale_log2 - LSE2),   dS^T = P^T (dP^T - D)
//   dV += P^T dO, dK += dS^T Q           TS MMAs: P^T / dS^T from TMEM, dO / Q MN-major
// A softmax thread owns one key row and 64 query columns; it writes P^T (dS^T) back as
// bf16 pairs into the first 32 of its own 64 S^T (dP^T) columns, so P and dS never pass
// through shared memory.  The next S^T (dP^T) overwrites P^T (dS^T), so it is issued
// once dV (dK) of the previous step completed; the issue order dV(t), dK(t), S^T(t+1),
// dP^T(t+1) keeps the tensor pipe fed across those waits.  LSE2 = LSE log2(e) and D of
// the step's 128 queries arrive in shared memory with the Q and dO tiles (bulk copies
// from the padded workspace rows).  Both stages are released when dK completes (the
// softmax reads D until it hands over dS^T); Q gets three stages, dO two.

constexpr int KV_QST = 3;
constexpr int KV_DOST = 2;
constexpr uint32_t ROWV = BM * 4;                   // one step's LSE2 or D values
constexpr uint32_t KV_TM_S = 0, KV_TM_DP = 128, KV_TM_DV = 256, KV_TM_DK = 384;

// Head-dim dependent layouts (head_dim 128 or 64): a Q/K/V/dO tile is 128 rows x HD
// columns in HD / 64 swizzled halves; shared-memory offsets from a 1024-aligned base.
template <int HD_>
struct BwdCfg {
  static constexpr int HD = HD_;
  static constexpr int NH = HD / 64;
  static constexpr int ACOLS = HD / 2;      // accumulator columns per thread (2 per lane)
  static constexpr uint32_t TILE = BM * HD * 2;
  static constexpr uint32_t KV_OFF_K = 0;
  static constexpr uint32_t KV_OFF_V = TILE;
  static constexpr uint32_t KV_OFF_Q = 2 * TILE;
  static constexpr uint32_t KV_OFF_DO = KV_OFF_Q + KV_QST * TILE;
  static constexpr uint32_t KV_OFF_LSE = KV_OFF_DO + KV_DOST * TILE;   // one per Q stage
  static constexpr uint32_t KV_OFF_D = KV_OFF_LSE + KV_QST * ROWV;     // one per dO stage
  static constexpr uint32_t KV_OFF_BAR = KV_OFF_D + KV_DOST * ROWV;
  static constexpr uint32_t KV_SMEM = KV_OFF_BAR + 256;
  static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
  static_assert(KV_SMEM <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

struct KvBars {
  uint64_t kv_full;
  uint64_t q_full[KV_QST], q_empty[KV_QST], do_full[KV_DOST], do_empty[KV_DOST];
  uint64_t s_full, dp_full, p_ready, ds_ready, dv_done, dk_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(KvBars) <= 256, "barrier block overflows its shared-memory slot");

// TMEM column of the bf16 pairs of queries [16 kk, 16 kk + 16) in a P^T / dS^T region:
// queries 0-63 sit in columns 0-31 (written by the half-0 threads), queries 64-127 in
// columns 64-95 (half 1), each inside the columns its writer has already read.
__host__ __device__ constexpr uint32_t kv_pair_col(int kk) {
  return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8;
}

// Walks the (query head, query tile) pairs feeding one key tile: every query head of
// the KV group, each with the transposed list of its map head (head-major: measured
// faster than query-tile-major on the GQA 64:8 workload).
struct ColWalk {
  const PlanDev* pl;
  int kt, hk, group, heads_per_map, n_kt;
  int gi, pos, end;
  __device__ void start_head() {
    const int h = hk * group + gi;
    const int col = (h / heads_per_map) * n_kt + kt;
    pos = __ldg(pl->colptr + col);
    end = __ldg(pl->colptr + col + 1);
  }
  __device__ void init(const PlanDev* p, int kt_, int hk_, const AttnDims& d) {
    pl = p; kt = kt_; hk = hk_; group = d.group; heads_per_map = d.heads_per_map; n_kt = p->n_kt;
    gi = 0;
    start_head();
  }
  // Next pair; false when done.
  __device__ bool next(int& h, int& qt, int& cls) {
    while (pos >= end) {
      if (++gi >= group) return false;
      start_head();
    }
    h = hk * group + gi;
    qt = __ldg(pl->qt_idx + pos);
    cls = __ldg(pl->qt_cls + pos);
    ++pos;
    return true;
  }
};

// use_half_path over the column lists a dK/dV CTA walks.  Warp-wide.
__device__ __forceinline__ bool walk_use_half_path(const PlanDev& pl, int kt, int hk,
                                                   const AttnDims& d, int lane) {
  int f = 0, n = 0;
  int prev = -1;
  for (int gi = 0; gi < d.group; ++gi) {
    const int col = ((hk * d.group + gi) / d.heads_per_map) * pl.n_kt + kt;
    if (col == prev) continue;   // query heads sharing a map share its list
    prev = col;
    const int p0 = __ldg(pl.colptr + col), p1 = __ldg(pl.colptr + col + 1);
    n += p1 - p0;
    for (int x = p0 + lane; x < p1; x += 32)
      f += (__ldg(pl.qt_cls + x) & kEntryHalfFlags) != 0;
  }
  return half_path(__reduce_add_sync(0xFFFFFFFFu, f), n, HALF_SHARE);
}

template <int HD_>
__device__ __forceinline__ void dkdv_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                         const CUtensorMap& tm_v, const CUtensorMap& tm_do,
                                         const BwdArgs& a, int blk) {
  using C = BwdCfg<HD_>;
  constexpr int HD = C::HD, NH = C::NH, ACOLS = C::ACOLS;
  constexpr uint32_t TILE = C::TILE;
  constexpr uint32_t KV_OFF_K = C::KV_OFF_K, KV_OFF_V = C::KV_OFF_V, KV_OFF_Q = C::KV_OFF_Q,
                     KV_OFF_DO = C::KV_OFF_DO, KV_OFF_LSE = C::KV_OFF_LSE, KV_OFF_D = C::KV_OFF_D,
                     KV_OFF_BAR = C::KV_OFF_BAR;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  if (base_u32 & 1023u) {
    if (threadIdx.x == 0) atomicOr(a.err, LCA_DEVERR_LAYOUT);
    return;
  }
  uint8_t* base = smem_raw;
  KvBars& bar = *reinterpret_cast<KvBars*>(base + KV_OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnDims& dm = a.dims;
  const PlanDev& pl = a.plan;
  const int S = dm.seqlen;

  int b, hk, kt;
  if (dm.kv_per_map > 0) {
    const int per_item = dm.kv_per_map * dm.batch;
    int item, rem;
    chunked_item(blk, per_item, pl.map_heads * pl.n_kt, dm.chunk, item, rem);
    const int col = __ldg(pl.work_k + item);
    const int hm = col / pl.n_kt;
    kt = col - hm * pl.n_kt;
    hk = hm * dm.kv_per_map + rem % dm.kv_per_map;
    b = rem / dm.kv_per_map;
  } else {
    kt = blk % pl.n_kt;
    const int rest = blk / pl.n_kt;
    hk = rest % dm.h_kv;
    b = rest / dm.h_kv;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bar.kv_full, 1);
    for (int s = 0; s < KV_QST; ++s) {
      mbar_init(&bar.q_full[s], 1);
      mbar_init(&bar.q_empty[s], 1);
    }
    for (int s = 0; s < KV_DOST; ++s) {
      mbar_init(&bar.do_full[s], 1);
      mbar_init(&bar.do_empty[s], 1);
    }
    mbar_init(&bar.s_full, 1);
    mbar_init(&bar.dp_full, 1);
    mbar_init(&bar.p_ready, SOFTMAX_THREADS);
    mbar_init(&bar.ds_ready, SOFTMAX_THREADS);
    mbar_init(&bar.dv_done, 1);
    mbar_init(&bar.dk_done, 1);
    bar.abort = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&bar.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  WaitCtx wc{&bar.abort, a.err, a.timeout_ns};
  ColWalk walk;
  walk.init(&pl, kt, hk, dm);
  const int64_t row0 = static_cast<int64_t>(b) * dm.h_q;   // workspace row of head 0

  if (warp == WARP_PRODUCER) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      mbar_arrive_expect_tx(&bar.kv_full, 2 * TILE);
      for (int c = 0; c < NH; ++c) {
        tma_load_4d(base + KV_OFF_K + c * HALF, &tm_k, &bar.kv_full, c * 64, hk, kt * BN, b);
        tma_load_4d(base + KV_OFF_V + c * HALF, &tm_v, &bar.kv_full, c * 64, hk, kt * BN, b);
      }
      int h, qt, cls, t = 0;
      ColWalk ahead = walk;   // L2 prefetch of the Q tile KV_QST steps ahead
      int ha, qa, ca;
      for (int k = 0; k < KV_QST && ahead.next(ha, qa, ca); ++k)
        for (int c = 0; c < NH; ++c) tma_prefetch_l2_4d(&tm_q, c * 64, ha, qa * BM, b);
      while (walk.next(h, qt, cls)) {
        const int st = t % KV_QST;
        const uint32_t ph = (t / KV_QST) & 1;
        if (ahead.next(ha, qa, ca))
          for (int c = 0; c < NH; ++c) tma_prefetch_l2_4d(&tm_q, c * 64, ha, qa * BM, b);
        if (t >= KV_QST) mbar_wait(&bar.q_empty[st], ph ^ 1u, wc);
        mbar_arrive_expect_tx(&bar.q_full[st], TILE + ROWV);
        for (int c = 0; c < NH; ++c)
          tma_load_4d(base + KV_OFF_Q + st * TILE + c * HALF, &tm_q, &bar.q_full[st], c * 64, h,
                      qt * BM, b);
        bulk_load(base + KV_OFF_LSE + st * ROWV,
                  a.lse2 + (row0 + h) * a.s_pad + static_cast<int64_t>(qt) * BM, ROWV,
                  &bar.q_full[st]);
        ++t;
      }
      if (bar.abort) {
        mbar_wait_final(&bar.kv_full, 0, a.timeout_ns);
        for (int n = max(0, t - KV_QST); n < t; ++n)
          mbar_wait_final(&bar.q_full[n % KV_QST], (n / KV_QST) & 1, a.timeout_ns);
      }
    }
  } else if (warp == WARP_PRODUCER_2) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_do);
      int h, qt, cls, t = 0;
      ColWalk ahead = walk;   // L2 prefetch of the dO tile KV_QST steps ahead
      int ha, qa, ca;
      for (int k = 0; k < KV_QST && ahead.next(ha, qa, ca); ++k)
        for (int c = 0; c < NH; ++c) tma_prefetch_l2_4d(&tm_do, c * 64, ha, qa * BM, b);
      while (walk.next(h, qt, cls)) {
        const int st = t % KV_DOST;
        const uint32_t ph = (t / KV_DOST) & 1;
        if (ahead.next(ha, qa, ca))
          for (int c = 0; c < NH; ++c) tma_prefetch_l2_4d(&tm_do, c * 64, ha, qa * BM, b);
        if (t >= KV_DOST) mbar_wait(&bar.do_empty[st], ph ^ 1u, wc);
        mbar_arrive_expect_tx(&bar.do_full[st], TILE + ROWV);
        for (int c = 0; c < NH; ++c)
          tma_load_4d(base + KV_OFF_DO + st * TILE + c * HALF, &tm_do, &bar.do_full[st], c * 64,
                      h, qt * BM, b);
        bulk_load(base + KV_OFF_D + st * ROWV,
                  a.dsum + (row0 + h) * a.s_pad + static_cast<int64_t>(qt) * BM, ROWV,
                  &bar.do_full[st]);
        ++t;
      }
      if (bar.abort) {
        for (int n = max(0, t - KV_DOST); n < t; ++n)
          mbar_wait_final(&bar.do_full[n % KV_DOST], (n / KV_DOST) & 1, a.timeout_ns);
      }
    }
  } else if (warp == WARP_MMA) {
    const bool halves = walk_use_half_path(pl, kt, hk, dm, lane);
    if (lane == 0) {
      constexpr uint32_t IDESC_SS = idesc_bf16(BN, BM, 0, 0);  // S^T, dP^T
      constexpr uint32_t IDESC_SS_HALF = idesc_bf16(BN, BM / 2, 0, 0);
      constexpr uint32_t IDESC_TS = idesc_bf16(BN, HD, 0, 1);  // dV, dK (B MN-major)
      const uint64_t dk_ = desc_kmajor(base_u32 + KV_OFF_K, 0, HALF);
      const uint64_t dv_ = desc_kmajor(base_u32 + KV_OFF_V, 0, HALF);
      const uint64_t dq_k0 = desc_kmajor(base_u32 + KV_OFF_Q, 0, HALF);
      const uint64_t ddo_k0 = desc_kmajor(base_u32 + KV_OFF_DO, 0, HALF);
      const uint64_t dq_m0 = desc_mnmajor(base_u32 + KV_OFF_Q, 0, HALF);
      const uint64_t ddo_m0 = desc_mnmajor(base_u32 + KV_OFF_DO, 0, HALF);
      int total = 0;
      {
        ColWalk w2 = walk;
        int h, qt, cls;
        while (w2.next(h, qt, cls)) ++total;
      }
      // A step whose entry flags a query half as empty recomputes S^T / dP^T for the
      // other half only (N = 64 on its 64 Q / dO rows, into its 64 columns) and gives
      // dV / dK only that half's k-steps.
      auto recompute = [&](uint32_t tcol, uint64_t da, uint64_t db, int empty) {
        uint32_t idesc = IDESC_SS;
        if (empty != 0) {
          const int hf = empty == 1 ? 1 : 0;
          idesc = IDESC_SS_HALF;
          tcol += hf * 64;
          db += hf * ROWS64_STEP;
        }
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_ss(tmem + tcol, da + kmajor_step(kk, HALF), db + kmajor_step(kk, HALF), idesc,
                       kk > 0 ? 1u : 0u);
      };
      auto accumulate = [&](uint32_t dcol, uint32_t acol, uint64_t db, int empty, bool first) {
        if (empty == 0) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_bf16_ts(tmem + dcol, tmem + acol + kv_pair_col(kk), db + mnmajor_step(kk),
                         IDESC_TS, (!first || kk > 0) ? 1u : 0u);
        } else {
          // the four k-steps of the other query half only
          const int k0 = empty == 1 ? 4 : 0;
          const uint32_t a0 = tmem + acol + kv_pair_col(k0);
          const uint64_t b0 = db + mnmajor_step(k0);
#pragma unroll
          for (int kk = 0; kk < BM / 32; ++kk)
            umma_bf16_ts(tmem + dcol, a0 + kk * 8, b0 + mnmajor_step(kk), IDESC_TS,
                         (!first || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_s = [&](int t, int empty) {
        tc_fence_after();
        recompute(KV_TM_S, dk_, dq_k0 + (t % KV_QST) * stage_step(TILE), empty);
        umma_commit(&bar.s_full);
      };
      auto issue_dp = [&](int t, int empty) {
        tc_fence_after();
        recompute(KV_TM_DP, dv_, ddo_k0 + (t % KV_DOST) * stage_step(TILE), empty);
        umma_commit(&bar.dp_full);
      };
      auto issue_dv = [&](int t, int empty) {
        tc_fence_after();
        accumulate(KV_TM_DV, KV_TM_S, ddo_m0 + (t % KV_DOST) * stage_step(TILE), empty, t == 0);
        umma_commit(&bar.dv_done);
      };
      auto issue_dk = [&](int t, int empty) {
        const int st = t % KV_QST;
        tc_fence_after();
        accumulate(KV_TM_DK, KV_TM_DP, dq_m0 + st * stage_step(TILE), empty, t == 0);
        umma_commit(&bar.dk_done);
        umma_commit(&bar.q_empty[st]);
        umma_commit(&bar.do_empty[t % KV_DOST]);   // D(t) is read until ds_ready(t)
      };
      // Key tiles that walk_use_half_path turns down run the loop without any flag
      // handling (a separate instantiation; the issue loop is sensitive to extra work).
      // In the flag-aware loop the steps' entries come from the issuer's own walk, one
      // step ahead of use: a load consumed right away holds the issue of the next MMAs
      // back.
      auto run = [&](auto halves_c) {
        constexpr bool HALVES = decltype(halves_c)::value;
        ColWalk iw = walk;
        int e_next = 0;
        auto fetch = [&]() {
          int h, qt, cls;
          if (iw.next(h, qt, cls)) e_next = cls;
        };
        int eh = 0;          // empty halves of step t
        mbar_wait(&bar.kv_full, 0, wc);
        if (total > 0) {
          if constexpr (HALVES) {
            fetch();
            eh = entry_empty_halves(e_next);
            fetch();
          }
          mbar_wait(&bar.q_full[0], 0, wc);
          issue_s(0, eh);
          mbar_wait(&bar.do_full[0], 0, wc);
          issue_dp(0, eh);
        }
        // Issue order dV(t), S^T(t+1), dK(t), dP^T(t+1): S^T(t+1) runs while the softmax
        // still turns dP^T(t) into dS^T(t).  S^T(t+1) overwrites P^T(t) and dP^T(t+1)
        // overwrites dS^T(t); tcgen05 MMAs of one thread run in issue order, so dV(t)
        // (dK(t)) has read them by then.
        for (int t = 0; t < total && !bar.abort; ++t) {
          const int eh_t = eh;
          mbar_wait(&bar.p_ready, t & 1, wc);
          issue_dv(t, eh_t);
          const int n = t + 1;
          if (n < total) {
            if constexpr (HALVES) {
              eh = entry_empty_halves(e_next);
              fetch();
            }
            mbar_wait(&bar.q_full[n % KV_QST], (n / KV_QST) & 1, wc);
            issue_s(n, eh);
          }
          mbar_wait(&bar.ds_ready, t & 1, wc);
          issue_dk(t, eh_t);
          if (n < total) {
            mbar_wait(&bar.do_full[n % KV_DOST], (n / KV_DOST) & 1, wc);
            issue_dp(n, eh);
          }
        }
      };
      if (halves) run(std::true_type{}); else run(std::false_type{});
    }
  } else {
    // ------------------------------------------------ softmax warps 0-7
    const int quarter = warp & 3, half = warp >> 2;
    const int jl = quarter * 32 + lane;              // key row within the tile = TMEM lane
    const int j = kt * BN + jl;
    const bool jvalid = j < S;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * 64;
    const float sl2 = dm.scale_log2;
    const RowSpan cs = col_span(a.mask, min(j, S - 1));
    MapCursor mcur;
    int t = 0;
    // Key tiles that walk_use_half_path turns down run the loop without the idle check
    // (a separate instantiation).
    auto steps = [&](auto halves_c) {
      constexpr bool HALVES = decltype(halves_c)::value;
      int h, qt, cls;
      while (walk.next(h, qt, cls)) {
        // this warp's query half holds no pair of the tile: nothing to read or write
        const bool idle = HALVES && ((entry_empty_halves(cls) >> half) & 1);
        const bool masked =
            entry_class(cls) != LCA_TILE_FULL || kt * BN + BN > S || qt * BM + BM > S;
        uint32_t bits[2] = {0u, 0u};
        if (masked && jvalid && !idle)
          col_tile_bits<2>(a.mask, h / dm.heads_per_map, j, qt * BM + half * 64, cs, bits, &mcur);
        const float* lse2 =
            reinterpret_cast<const float*>(base + KV_OFF_LSE + (t % KV_QST) * ROWV) + half * 64;
        const float* dsum =
            reinterpret_cast<const float*>(base + KV_OFF_D + (t % KV_DOST) * ROWV) + half * 64;

        // The LSE2 / D rows were written by bulk copies that complete on q_full / do_full;
        // observing those phases here (already complete: the stages are refilled only
        // after this step's ds_ready) makes the rows visible to this thread.
        mbar_wait(&bar.s_full, t & 1, wc);
        mbar_wait(&bar.q_full[t % KV_QST], (t / KV_QST) & 1, wc);
        __syncwarp();
        tc_fence_after();
        if (idle) {
          tc_fence_before();
          mbar_arrive(&bar.p_ready);
          mbar_wait(&bar.dp_full, t & 1, wc);
          mbar_wait(&bar.do_full[t % KV_DOST], (t / KV_DOST) & 1, wc);
          tc_fence_before();
          mbar_arrive(&bar.ds_ready);
          ++t;
          continue;
        }
        uint32_t r[64];
        tmem_ld64(lane_addr + KV_TM_S, r);
        float p[64];
#pragma unroll
        for (int x = 0; x < 64; x += 4) {
          const float4 l = *reinterpret_cast<const float4*>(lse2 + x);
          p[x + 0] = ex2_approx(fmaf(__uint_as_float(r[x + 0]), sl2, -l.x));
          p[x + 1] = ex2_approx(fmaf(__uint_as_float(r[x + 1]), sl2, -l.y));
          p[x + 2] = ex2_approx(fmaf(__uint_as_float(r[x + 2]), sl2, -l.z));
          p[x + 3] = ex2_approx(fmaf(__uint_as_float(r[x + 3]), sl2, -l.w));
        }
        if (masked) {
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (!((bits[x >> 5] >> (x & 31)) & 1u)) p[x] = 0.f;
        }
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) pk[x] = pack_bf16x2(p[2 * x], p[2 * x + 1]);
        tmem_st32(lane_addr + KV_TM_S, pk);
        tc_fence_before();
        mbar_arrive(&bar.p_ready);

        mbar_wait(&bar.dp_full, t & 1, wc);
        mbar_wait(&bar.do_full[t % KV_DOST], (t / KV_DOST) & 1, wc);
        __syncwarp();
        tc_fence_after();
        tmem_ld64(lane_addr + KV_TM_DP, r);
#pragma unroll
        for (int x = 0; x < 64; x += 4) {
          const float4 dd = *reinterpret_cast<const float4*>(dsum + x);
          p[x + 0] *= __uint_as_float(r[x + 0]) - dd.x;
          p[x + 1] *= __uint_as_float(r[x + 1]) - dd.y;
          p[x + 2] *= __uint_as_float(r[x + 2]) - dd.z;
          p[x + 3] *= __uint_as_float(r[x + 3]) - dd.w;
        }
#pragma unroll
        for (int x = 0; x < 32; ++x) pk[x] = pack_bf16x2(p[2 * x], p[2 * x + 1]);
        tmem_st32(lane_addr + KV_TM_DP, pk);
        tc_fence_before();
        mbar_arrive(&bar.ds_ready);
        ++t;
      }
    };
    if (walk_use_half_path(pl, kt, hk, dm, lane)) steps(std::true_type{});
    else steps(std::false_type{});
    if (t > 0) {
      mbar_wait(&bar.dv_done, (t - 1) & 1, wc);
      mbar_wait(&bar.dk_done, (t - 1) & 1, wc);
      __syncwarp();
      tc_fence_after();
    }
    const int64_t col = static_cast<int64_t>(hk) * HD + half * ACOLS;
    const int64_t pos = static_cast<int64_t>(b) * S + j;
    const uint32_t acc_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * ACOLS;
    store_acc_half<ACOLS>(acc_addr + KV_TM_DV, t > 0, 1.f, a.dv + pos * a.dv_row_stride + col,
                          jvalid);
    store_acc_half<ACOLS>(acc_addr + KV_TM_DK, t > 0, dm.scale,
                          a.dk + pos * a.dk_row_stride + col, jvalid);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dQ

// dO only ever feeds dP = dO V^T as the A operand, so it sits in TMEM (bf16 pairs, 64
// columns, stored once per CTA by the softmax threads) and dP is a TS MMA; the shared
// memory it frees gives the K and V rings three stages each.
constexpr int DQ_KST = 3;                        // K stages (K is held until the dQ MMA)
constexpr int DQ_VST = 3;                        // V stages (V is released after dP)

template <int HD_>
struct DqCfg {
  static constexpr uint32_t TILE = BwdCfg<HD_>::TILE;
  static constexpr uint32_t DQ_OFF_Q = 0;
  static constexpr uint32_t DQ_OFF_K = TILE;
  static constexpr uint32_t DQ_OFF_V = DQ_OFF_K + DQ_KST * TILE;
  static constexpr uint32_t DQ_OFF_BAR = DQ_OFF_V + DQ_VST * TILE;
  static constexpr uint32_t DQ_SMEM = DQ_OFF_BAR + 256;   // the dynamic base is 1024-aligned
  static_assert(DQ_SMEM <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};
constexpr uint32_t DQ_TM_S = 0, DQ_TM_DP = 128, DQ_TM_DQ = 256, DQ_TM_DS = 384, DQ_TM_DO = 448;

struct DqBars {
  uint64_t q_full, do_ready;
  uint64_t k_full[DQ_KST], k_empty[DQ_KST], v_full[DQ_VST], v_empty[DQ_VST];
  uint64_t sdp_full, sdp_free, ds_ready, dq_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqBars) <= 256, "barrier block overflows its shared-memory slot");

template <int HD_>
__device__ __forceinline__ void dq_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                       const CUtensorMap& tm_v, const CUtensorMap& tm_do,
                                       const BwdArgs& a, int blk) {
  using C = BwdCfg<HD_>;
  using D = DqCfg<HD_>;
  constexpr int HD = C::HD, NH = C::NH, ACOLS = C::ACOLS;
  constexpr uint32_t TILE = C::TILE;
  constexpr uint32_t DQ_OFF_Q = D::DQ_OFF_Q, DQ_OFF_K = D::DQ_OFF_K, DQ_OFF_V = D::DQ_OFF_V,
                     DQ_OFF_BAR = D::DQ_OFF_BAR;
  constexpr int DOC = HD / 4;   // TMEM columns of this thread's half row of dO (bf16 pairs)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  if (base_u32 & 1023u) {   // the swizzled tiles need a 1024-byte-aligned base
    if (threadIdx.x == 0) atomicOr(a.err, LCA_DEVERR_LAYOUT);
    return;
  }
  uint8_t* base = smem_raw;
  DqBars& bar = *reinterpret_cast<DqBars*>(base + DQ_OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnDims& dm = a.dims;
  const PlanDev& pl = a.plan;
  const int S = dm.seqlen;

  const int per_item = dm.heads_per_map * dm.batch;
  int item, rem;
  chunked_item(blk, per_item, pl.map_heads * pl.n_qt, dm.chunk, item, rem);
  const int row = __ldg(pl.work_q + item);
  const int hm = row / pl.n_qt;
  const int qt = row - hm * pl.n_qt;
  const int h = hm * dm.heads_per_map + rem % dm.heads_per_map;
  const int b = rem / dm.heads_per_map;
  const int hk = h / dm.group;
  const int beg = __ldg(pl.rowptr + row);
  const int n_tiles = __ldg(pl.rowptr + row + 1) - beg;
  const auto tile = [&](int n) { return beg + n; };

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.do_ready, SOFTMAX_THREADS);
    for (int s = 0; s < DQ_KST; ++s) {
      mbar_init(&bar.k_full[s], 1);
      mbar_init(&bar.k_empty[s], 1);
    }
    for (int s = 0; s < DQ_VST; ++s) {
      mbar_init(&bar.v_full[s], 1);
      mbar_init(&bar.v_empty[s], 1);
    }
    mbar_init(&bar.sdp_full, 1);
    mbar_init(&bar.sdp_free, SOFTMAX_THREADS);
    mbar_init(&bar.ds_ready, SOFTMAX_THREADS);
    mbar_init(&bar.dq_done, 1);
    bar.abort = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&bar.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  WaitCtx wc{&bar.abort, a.err, a.timeout_ns};

  if (warp == WARP_PRODUCER) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar.q_full, TILE);
      for (int c = 0; c < NH; ++c)
        tma_load_4d(base + DQ_OFF_Q + c * HALF, &tm_q, &bar.q_full, c * 64, h, qt * BM, b);
      for (int n = 0; n < n_tiles; ++n) {
        const int kt = __ldg(pl.kt_idx + tile(n));
        const int st = n % DQ_KST;
        if (n + DQ_KST < n_tiles) {
          const int ka = __ldg(pl.kt_idx + tile(n + DQ_KST));
          for (int c = 0; c < NH; ++c) tma_prefetch_l2_4d(&tm_k, c * 64, hk, ka * BN, b);
        }
        if (n >= DQ_KST) mbar_wait(&bar.k_empty[st], (n / DQ_KST - 1) & 1, wc);
        mbar_arrive_expect_tx(&bar.k_full[st], TILE);
        for (int c = 0; c < NH; ++c)
          tma_load_4d(base + DQ_OFF_K + st * TILE + c * HALF, &tm_k, &bar.k_full[st], c * 64, hk,
                      kt * BN, b);
      }
      if (bar.abort) {
        mbar_wait_final(&bar.q_full, 0, a.timeout_ns);
        for (int n = max(0, n_tiles - DQ_KST); n < n_tiles; ++n)
          mbar_wait_final(&bar.k_full[n % DQ_KST], (n / DQ_KST) & 1, a.timeout_ns);
      }
    }
  } else if (warp == WARP_PRODUCER_2) {
    if (lane == 0) {
      // V stages are released after dP, earlier than K stages (released after dQ):
      // a separate warp keeps V loads from queueing behind K releases
      for (int n = 0; n < n_tiles; ++n) {
        const int kt = __ldg(pl.kt_idx + tile(n));
        const int st = n % DQ_VST;
        if (n + DQ_VST < n_tiles) {
          const int ka = __ldg(pl.kt_idx + tile(n + DQ_VST));
          for (int c = 0; c < NH; ++c) tma_prefetch_l2_4d(&tm_v, c * 64, hk, ka * BN, b);
        }
        if (n >= DQ_VST) mbar_wait(&bar.v_empty[st], (n / DQ_VST - 1) & 1, wc);
        mbar_arrive_expect_tx(&bar.v_full[st], TILE);
        for (int c = 0; c < NH; ++c)
          tma_load_4d(base + DQ_OFF_V + st * TILE + c * HALF, &tm_v, &bar.v_full[st], c * 64, hk,
                      kt * BN, b);
      }
      if (bar.abort) {
        for (int n = max(0, n_tiles - DQ_VST); n < n_tiles; ++n)
          mbar_wait_final(&bar.v_full[n % DQ_VST], (n / DQ_VST) & 1, a.timeout_ns);
      }
    }
  } else if (warp == WARP_MMA) {
    const bool halves = use_half_path(pl.kt_cls + beg, n_tiles, HALF_SHARE, lane);
    if (lane == 0) {
      constexpr uint32_t IDESC_NT = idesc_bf16(BM, BN, 0, 0);  // S, dP
      constexpr uint32_t IDESC_NT_HALF = idesc_bf16(BM, BN / 2, 0, 0);
      constexpr uint32_t IDESC_NN = idesc_bf16(BM, HD, 0, 1);  // dQ (B = K MN-major)
      const uint64_t dq_ = desc_kmajor(base_u32 + DQ_OFF_Q, 0, HALF);
      const uint64_t dk_k0 = desc_kmajor(base_u32 + DQ_OFF_K, 0, HALF);
      const uint64_t dk_m0 = desc_mnmajor(base_u32 + DQ_OFF_K, 0, HALF);
      const uint64_t dv_k0 = desc_kmajor(base_u32 + DQ_OFF_V, 0, HALF);
      // Two MMA groups per key tile n: SdP(n) = {S, dP} and dQ(n), issued as soon as
      // their inputs are ready so that a late K/V tile for SdP(n+1) never holds back
      // dQ(n).  SdP(n+1) needs the softmax's release of S/dP(n); the softmax writes
      // dS(n+1) only after dQ(n) completed, so ds_ready is at most one phase ahead.
      // dP first: its commit releases the V stage half a group earlier, and S (the last
      // reader of K until dQ) gets its K tile later.
      auto issue_sdp = [&](int n, int empty) {
        uint64_t dk = dk_k0 + (n % DQ_KST) * stage_step(TILE);
        uint64_t dv = dv_k0 + (n % DQ_VST) * stage_step(TILE);
        uint32_t idesc = IDESC_NT, col = 0;
        if (empty != 0) {   // one key half only: its 64 K / V rows into its 64 columns
          const int hf = empty == 1 ? 1 : 0;
          idesc = IDESC_NT_HALF;
          col = hf * 64;
          dk += hf * ROWS64_STEP;
          dv += hf * ROWS64_STEP;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_ts(tmem + DQ_TM_DP + col, tmem + DQ_TM_DO + kk * 8,
                       dv + kmajor_step(kk, HALF), idesc, kk > 0 ? 1u : 0u);
        umma_commit(&bar.v_empty[n % DQ_VST]);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_ss(tmem + DQ_TM_S + col, dq_ + kmajor_step(kk, HALF),
                       dk + kmajor_step(kk, HALF), idesc, kk > 0 ? 1u : 0u);
        umma_commit(&bar.sdp_full);
      };
      auto issue_dq = [&](int n, int empty) {
        const uint64_t dk = dk_m0 + (n % DQ_KST) * stage_step(TILE);
        tc_fence_after();
        if (empty == 0) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_bf16_ts(tmem + DQ_TM_DQ, tmem + DQ_TM_DS + kk * 8, dk + mnmajor_step(kk),
                         IDESC_NN, (n > 0 || kk > 0) ? 1u : 0u);
        } else {
          // the four k-steps of the other key half only
          const int k0 = empty == 1 ? 4 : 0;
#pragma unroll
          for (int kk = 0; kk < BN / 32; ++kk)
            umma_bf16_ts(tmem + DQ_TM_DQ, tmem + DQ_TM_DS + (k0 + kk) * 8,
                         dk + mnmajor_step(k0 + kk), IDESC_NN, (n > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bar.dq_done);
        umma_commit(&bar.k_empty[n % DQ_KST]);
      };
      // Rows that use_half_path turns down run the loop without any flag handling (a
      // separate instantiation; the issue loop is sensitive to extra work).  In the
      // flag-aware loop the entry of tile n_sdp is loaded one SdP issue ahead of use (a
      // load consumed right away holds the issue of the next MMAs back), then kept for
      // dQ in a register ring, two bits at (n % 16) (the two counters stay a few tiles
      // apart).
      auto run = [&](auto halves_c) {
        constexpr bool HALVES = decltype(halves_c)::value;
        mbar_wait(&bar.q_full, 0, wc);
        mbar_wait(&bar.do_ready, 0, wc);
        int n_sdp = 0, n_dq = 0;
        int e_sdp = (HALVES && n_tiles > 0) ? __ldg(pl.kt_cls + tile(0)) : 0;
        uint32_t ring = 0u;
        uint64_t idle_since = 0;
        while (n_dq < n_tiles && !bar.abort) {
          bool progress = false;
          if (n_sdp < n_tiles && (n_sdp == 0 || mbar_test(&bar.sdp_free, (n_sdp - 1) & 1)) &&
              mbar_test(&bar.k_full[n_sdp % DQ_KST], (n_sdp / DQ_KST) & 1) &&
              mbar_test(&bar.v_full[n_sdp % DQ_VST], (n_sdp / DQ_VST) & 1)) {
            if constexpr (HALVES) {
              const int empty = entry_empty_halves(e_sdp);
              const int sh = 2 * (n_sdp % 16);
              ring = (ring & ~(3u << sh)) | (static_cast<uint32_t>(empty) << sh);
              issue_sdp(n_sdp++, empty);
              if (n_sdp < n_tiles) e_sdp = __ldg(pl.kt_cls + tile(n_sdp));
            } else {
              issue_sdp(n_sdp++, 0);
            }
            progress = true;
          }
          if (n_dq < n_sdp && mbar_test(&bar.ds_ready, n_dq & 1)) {
            issue_dq(n_dq, HALVES ? static_cast<int>((ring >> (2 * (n_dq % 16))) & 3) : 0);
            ++n_dq;
            progress = true;
          }
          if (progress) {
            idle_since = 0;
          } else if (idle_since == 0) {
            idle_since = globaltimer_ns();
          } else if (globaltimer_ns() - idle_since > a.timeout_ns) {
            bar.abort = 1;
            atomicOr(a.err, LCA_DEVERR_TIMEOUT);
          }
        }
      };
      if (halves) run(std::true_type{}); else run(std::false_type{});
    }
  } else {
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const int i = qt * BM + row;
    const bool valid = i < S;
    const uint32_t quarter_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t lane_addr = quarter_addr + half * 64;
    const float sl2 = dm.scale_log2;
    // padded workspace rows: +inf / 0 on rows without keys and past S
    const int64_t rowi = (static_cast<int64_t>(b) * dm.h_q + h) * a.s_pad + i;
    const float lse2 = __ldg(a.lse2 + rowi);
    const float dsum = __ldg(a.dsum + rowi);
    const int64_t pos = static_cast<int64_t>(b) * S + i;
    const int64_t col = static_cast<int64_t>(h) * HD + half * ACOLS;
    {
      // this thread's half row of dO (HD / 2 bf16) into TMEM columns
      // [DQ_TM_DO + DOC half, + DOC)
      uint32_t v[DOC];
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(a.dout + pos * a.do_row_stride + col);
#pragma unroll
        for (int u = 0; u < DOC / 4; ++u) {
          const uint4 w = __ldg(src + u);
          v[4 * u] = w.x; v[4 * u + 1] = w.y; v[4 * u + 2] = w.z; v[4 * u + 3] = w.w;
        }
      } else {
#pragma unroll
        for (int u = 0; u < DOC; ++u) v[u] = 0u;
      }
      tmem_stn<DOC>(quarter_addr + DQ_TM_DO + half * DOC, v);
      tc_fence_before();
      mbar_arrive(&bar.do_ready);
    }
    const RowSpan sp = row_span(a.mask, min(i, S - 1));
    MapCursor mcur;
    // One key tile; IDLE: this warp's key half holds no pair of the tile (nothing to read
    // or write, only the barrier protocol).  Two instantiations keep the common path's
    // code exactly that of a full-width tile.
    auto tile_step = [&](int n, auto idle_c) {
      constexpr bool IDLE = decltype(idle_c)::value;
      if constexpr (!IDLE) {
        const int kt = __ldg(pl.kt_idx + tile(n));
        const int e = __ldg(pl.kt_cls + tile(n));
        const bool masked =
            entry_class(e) != LCA_TILE_FULL || kt * BN + BN > S || qt * BM + BM > S;
        uint32_t bits[2] = {0u, 0u};
        if (masked && valid) row_tile_bits<2>(a.mask, hm, i, kt * BN + half * 64, sp, bits, &mcur);
        mbar_wait(&bar.sdp_full, n & 1, wc);
        __syncwarp();
        tc_fence_after();
        uint32_t sr[64], dr[64];
        tmem_ld64x2(lane_addr + DQ_TM_S, lane_addr + DQ_TM_DP, sr, dr);
        tc_fence_before();
        mbar_arrive(&bar.sdp_free);
        uint32_t dk[32];
        ds_half(sr, dr, masked, bits, sl2, lse2, dsum, dk);
        if (n >= 1) mbar_wait(&bar.dq_done, (n - 1) & 1, wc);   // dQ_{n-1} read dS_{n-1}
        __syncwarp();
        tc_fence_after();
        tmem_st32(quarter_addr + DQ_TM_DS + half * 32, dk);
      } else {
        mbar_wait(&bar.sdp_full, n & 1, wc);
        mbar_arrive(&bar.sdp_free);
        if (n >= 1) mbar_wait(&bar.dq_done, (n - 1) & 1, wc);
      }
      tc_fence_before();
      mbar_arrive(&bar.ds_ready);
    };
    if (!use_half_path(pl.kt_cls + beg, n_tiles, HALF_SHARE, lane)) {
      for (int n = 0; n < n_tiles; ++n) tile_step(n, std::false_type{});
    } else {
      for (int n = 0; n < n_tiles; ++n) {
        if ((entry_empty_halves(__ldg(pl.kt_cls + tile(n))) >> half) & 1)
          tile_step(n, std::true_type{});
        else
          tile_step(n, std::false_type{});
      }
    }
    if (n_tiles > 0) {
      mbar_wait(&bar.dq_done, (n_tiles - 1) & 1, wc);
      __syncwarp();
      tc_fence_after();
    }
    store_acc_half<ACOLS>(quarter_addr + DQ_TM_DQ + half * ACOLS, n_tiles > 0, dm.scale,
                          a.dq + pos * a.dq_row_stride + col, valid);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The two passes in one launch: CTAs [0, n_kv) run dK/dV (the longest, launched
// first), the rest dQ.  Neither pass reads the other's output (both read only the
// preprocess rows), so dQ CTAs take over the SMs that the last wave of dK/dV CTAs
// leaves idle, with no drain and launch gap between two kernels.
template <int HD_>
__global__ void __launch_bounds__(KV_THREADS, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
           BwdArgs a, int n_kv) {
  static_assert(KV_THREADS == DQ_THREADS, "one block shape for both passes");
  if (static_cast<int>(blockIdx.x) < n_kv)
    dkdv_cta<HD_>(tm_q, tm_k, tm_v, tm_do, a, blockIdx.x);
  else
    dq_cta<HD_>(tm_q, tm_k, tm_v, tm_do, a, blockIdx.x - n_kv);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(a.dims.batch) * a.s_pad * a.dims.h_q;
  const int tpr = a.dims.head_dim / 8;
  const int64_t blocks = (rows * tpr + 255) / 256;
  if (a.dims.head_dim == 64)
    bwd_preprocess_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  else
    bwd_preprocess_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int HD>
static cudaError_t launch_bwd_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const BwdArgs& a, int n_kv, int n_q,
                                 cudaStream_t st) {
  constexpr uint32_t smem = BwdCfg<HD>::KV_SMEM > DqCfg<HD>::DQ_SMEM ? BwdCfg<HD>::KV_SMEM
                                                                      : DqCfg<HD>::DQ_SMEM;
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel<HD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_kernel<HD><<<n_kv + n_q, KV_THREADS, smem, st>>>(tq, tk, tv, tdo, a, n_kv);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdArgs& a, int n_kv, int n_q,
                       cudaStream_t st) {
  if (n_kv + n_q == 0) return cudaSuccess;
  if (a.dims.head_dim == 64) return launch_bwd_hd<64>(tq, tk, tv, tdo, a, n_kv, n_q, st);
  return launch_bwd_hd<128>(tq, tk, tv, tdo, a, n_kv, n_q, st);
}

}  // namespace lca
