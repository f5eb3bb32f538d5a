// Forward pass of mask-aware exact softmax attention on sm_103a.
//
// Computes O = softmax(scale * Q K^T + mask) V and LSE per query row, the operation
// the LongCA-bench kernels are measured on ("Long-Context Attention Benchmark":
// summary page, abstract and sections 2.2 / 3.1; reading note, "Key design" 2).
//
// Persistent CTAs, at most one per SM, work through units (one 128-row query tile of
// one query head and batch entry, with the tile's list of non-skipped key tiles from
// the tile plan).  Units are handed out in longest-first order by a global counter: the
// K producer warp takes the next unit when it starts loading that unit's K tiles,
// decodes it and passes it to the other roles through a ring of shared-memory slots, so
// an SM moves on to its next unit without a CTA exit, launch and prologue, and the next
// unit's loads, first S MMAs and first softmax tile overlap the end of the current one.
// Roles:
//   warp 8      unit fetcher and K producer: the K tiles of every unit into a 3-stage
//               ring (the ring and every barrier phase follow one tile counter across
//               units), the next unit's Q prefetched into L2;
//   warp 10     Q and V producer: a unit's Q once the previous unit's last S has read
//               the Q buffer, then its V tiles into a 3-stage ring;
//   warp 9      TMEM owner and MMA issuer: S_n = Q K_n^T (tcgen05, both operands in
//               shared memory, fp32 in TMEM, three buffers) and O += P_{n-2} V_{n-2}
//               with P read from TMEM (accumulated in TMEM).  PV trails S by two
//               tiles so that S_{n+1} is computed while the softmax works on S_n.  A
//               unit's first PV (which overwrites O) waits until the softmax warps have
//               read the previous unit's O; its first two S MMAs do not;
//   warps 0-7   softmax, two threads per query row (warps w and w+4 share TMEM lanes
//               and take key columns 0-63 / 64-127): read S_n from TMEM, apply the mask
//               bits only on partial or ragged tiles, combine the two halves' row
//               maxima through shared memory, online softmax in fp32 with exp2, write P
//               (bf16 pairs) back into the TMEM columns of S_n for the PV MMA, rescale
//               the O accumulator in TMEM when the running max moves by more than 2^8
//               (exact after the final 1/l normalisation); the next unit's first tile,
//               then this unit's epilogue.
// In a row of at least 64 plan entries of which at least a quarter flag one key half of
// their tile as empty (no allowed pair: block maps on a grid finer than the tile, ragged tails),
// such a tile runs at half width: S is an N = 64 MMA on the other half's keys, PV takes
// only that half's k-steps, and the softmax warps of the empty half only join the
// row-max exchange.  Other rows run loops without any flag handling.
// Keeping P in TMEM matters on this part: an M = N = 128 MMA with both operands in
// shared memory reads 128 B/clk, the whole shared-memory bandwidth of the SM.
// Tile = 128 x 128, head_dim 128 or 64.  All waits are bounded.
#include <cuda_runtime.h>

#include <type_traits>

#include "attn_kernels.h"
#include "lca_device.cuh"

namespace lca {

namespace {

constexpr int BM = 128;              // query rows per tile
constexpr int BN = 128;              // keys per tile
constexpr uint32_t HALF_BYTES = BM * 64 * 2;   // one 128-byte-swizzled 64-column half, 16 KB
constexpr uint64_t ROWS64_STEP = (64 * 128) >> 4;   // descriptor step to row 64 of a half
constexpr float RESCALE_THRESHOLD = 8.0f;      // log2 units
constexpr int HALF_SHARE = 4;   // half-width path: a quarter of a row's entries flagged

constexpr int NUM_THREADS = 352;     // 8 softmax warps, MMA issuer, K and V producers
constexpr int SOFTMAX_THREADS = 256;
constexpr int WARP_PRODUCER = 8, WARP_MMA = 9, WARP_PRODUCER_V = 10;
constexpr int BAR_SOFTMAX = 1;        // named barrier of the softmax warps

constexpr int KST = 3;                // K stages
constexpr int VST = 3;                // V stages
constexpr int NSB = 3;                // S buffers in TMEM

// Head-dim dependent layout (head_dim 128 or 64).  A Q/K/V tile is 128 rows x HD
// columns, stored as HD / 64 swizzled halves; shared memory offsets from a 1024-aligned
// base.
template <int HD_>
struct Cfg {
  static constexpr int HD = HD_;
  static constexpr int NH = HD / 64;                          // swizzled halves per tile
  static constexpr uint32_t TILE_BYTES = BM * HD * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;       // KST stages
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE_BYTES; // VST stages
  static constexpr uint32_t OFF_BAR = OFF_V + VST * TILE_BYTES;
  static constexpr uint32_t OFF_RED = OFF_BAR + 400;          // row-max / row-sum exchange
  static constexpr uint32_t SMEM_BYTES = OFF_RED + 2 * 2 * BM * 4;
  static constexpr int OCOLS = HD / 2;                        // O columns per softmax thread
  static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
  static_assert(SMEM_BYTES <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

// TMEM columns
constexpr uint32_t TM_S0 = 0, TM_O = NSB * BN, TM_COLS = 512;
static_assert(TM_O + 128 <= TM_COLS, "TMEM columns");

// N consecutive 32-bit TMEM columns (N = 32 or 64) of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 64) tmem_ld64(taddr, r); else tmem_ld32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 64) tmem_st64(taddr, r); else tmem_st32(taddr, r);
}

constexpr int UR = 4;                 // unit ring slots
constexpr int UNIT_READERS = 10;      // V producer, MMA warp, eight softmax warps

// A unit as the fetcher decodes it: query head, KV head, map head, query tile, batch
// entry, its row list [beg, beg + n) in the plan, and whether that list runs the
// half-width path.  n < 0 marks the end of the work.
struct Unit { int h, hk, hm, qt, b, beg, n, halves; };

struct Bars {
  uint64_t q_full, q_empty, o_free;
  uint64_t unit_full[UR], unit_empty[UR];
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[NSB], p_ready[NSB], pv_done[NSB];
  uint32_t tmem_base;
  int abort;
  Unit unit[UR];
};
static_assert(sizeof(Bars) <= 400, "barrier block overflows its shared-memory slot");

// use_half_path for the unit fetcher, which runs it while the K ring drains: lists too
// short for the half-width path are not read at all, longer ones with eight loads in
// flight per lane.
__device__ __forceinline__ bool fetch_half_path(const uint8_t* e, int n, int lane) {
  if (n < 64) return false;   // half_path() needs at least 64 entries
  int f = 0;
  for (int x0 = 0; x0 < n; x0 += 256) {
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int x = x0 + 32 * j + lane;
      v[j] = x < n ? __ldg(e + x) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) f += (v[j] & kEntryHalfFlags) != 0;
  }
  return half_path(__reduce_add_sync(0xFFFFFFFFu, f), n, HALF_SHARE);
}

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return desc_kmajor(tile, kk, HALF_BYTES);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
  return desc_mnmajor(tile, kk, HALF_BYTES);
}

template <int HD_>
__global__ void __launch_bounds__(NUM_THREADS, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, FwdArgs a) {
  using C = Cfg<HD_>;
  constexpr int HD = C::HD;
  constexpr uint32_t TILE_BYTES = C::TILE_BYTES;
  constexpr uint32_t OFF_Q = C::OFF_Q, OFF_K = C::OFF_K, OFF_V = C::OFF_V, OFF_BAR = C::OFF_BAR,
                     OFF_RED = C::OFF_RED;
  constexpr int OCOLS = C::OCOLS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  if (base_u32 & 1023u) {   // the swizzled tiles need a 1024-byte-aligned base
    if (threadIdx.x == 0) atomicOr(a.err, LCA_DEVERR_LAYOUT);
    return;
  }
  uint8_t* base = smem_raw;
  Bars& bar = *reinterpret_cast<Bars*>(base + OFF_BAR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AttnDims& dm = a.dims;
  const PlanDev& pl = a.plan;
  const int S = dm.seqlen;
  const int n_units = a.n_units;

  // A unit is one (query tile, query head, batch entry).  Units are handed out in
  // longest-first order by a global counter: the K producer warp takes the next unit when
  // it starts loading that unit's K tiles, decodes it (its list pointers and half-width
  // decision come from global memory) and passes the decoded unit to the other roles
  // through a ring of UR shared-memory slots, so no other role waits for those loads.
  auto decode = [&](int u) {
    const int per_item = dm.heads_per_map * dm.batch;
    int item, rem;
    chunked_item(u, per_item, pl.map_heads * pl.n_qt, dm.chunk, item, rem);
    Unit w;
    const int row = __ldg(pl.work_q + item);
    w.hm = row / pl.n_qt;
    w.qt = row - w.hm * pl.n_qt;
    w.h = w.hm * dm.heads_per_map + rem % dm.heads_per_map;
    w.b = rem / dm.heads_per_map;
    w.hk = w.h / dm.group;
    w.beg = __ldg(pl.rowptr + row);
    w.n = __ldg(pl.rowptr + row + 1) - w.beg;
    w.halves = 0;
    return w;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    mbar_init(&bar.o_free, SOFTMAX_THREADS);
    for (int s = 0; s < UR; ++s) {
      mbar_init(&bar.unit_full[s], 1);
      mbar_init(&bar.unit_empty[s], UNIT_READERS);
    }
    for (int s = 0; s < KST; ++s) {
      mbar_init(&bar.k_full[s], 1);
      mbar_init(&bar.k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&bar.v_full[s], 1);
      mbar_init(&bar.v_empty[s], 1);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&bar.s_full[s], 1);
      mbar_init(&bar.p_ready[s], SOFTMAX_THREADS);
      mbar_init(&bar.pv_done[s], 1);
    }
    bar.abort = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(&bar.tmem_base, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  WaitCtx wc{&bar.abort, a.err, a.timeout_ns};

  // The k-th unit of this CTA sits in ring slot k % UR.  Readers other than the fetcher:
  // the V producer, the MMA warp and the eight softmax warps (lane 0 of each arrives once
  // its warp has read the slot).  A unit with n < 0 ends every role's loop.
  // WHOLE: called by all 32 lanes of a warp (lane 0 arrives after the warp has read the
  // slot); otherwise by one lane alone, which arrives itself.
  auto take_unit = [&](int k, bool whole) {
    const int slot = k % UR;
    mbar_wait(&bar.unit_full[slot], (k / UR) & 1, wc);
    Unit w = bar.unit[slot];
    if (bar.abort) w.n = -1;
    if (whole) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.unit_empty[slot]);
    } else {
      mbar_arrive(&bar.unit_empty[slot]);
    }
    return w;
  };

  // The K/V rings, the S buffers and every barrier phase follow one tile counter g across
  // units; every role walks the same unit sequence, so the counters agree.
  if (warp == WARP_PRODUCER) {
    // ------------------------------------------------ unit fetcher and K producer
    // The whole warp fetches and decodes a unit (the half-width scan is warp-wide); lane
    // 0 publishes it and loads its K tiles while the other lanes wait at the __syncwarp.
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_q);
    }
    int g = 0;
    for (int k = 0;; ++k) {
      const int slot = k % UR;
      if (k >= UR) mbar_wait(&bar.unit_empty[slot], (k / UR - 1) & 1, wc);
      int u = 0;
      if (lane == 0) u = bar.abort ? n_units : static_cast<int>(atomicAdd(a.unit_counter, 1u));
      u = __shfl_sync(0xFFFFFFFFu, u, 0);
      Unit w{};
      w.n = -1;
      if (u < n_units) {
        w = decode(u);
        w.halves = fetch_half_path(pl.kt_cls + w.beg, w.n, lane);
      }
      if (lane == 0) {
        bar.unit[slot] = w;
        mbar_arrive(&bar.unit_full[slot]);
      }
      if (u >= n_units) break;
      if (lane == 0) {
        // the unit's Q is loaded only after the previous unit's last S; prefetching it into
        // L2 now (this thread runs a few tiles ahead) shortens that load
        if (w.n > 0)
          for (int c = 0; c < C::NH; ++c) tma_prefetch_l2_4d(&tm_q, c * 64, w.h, w.qt * BM, w.b);
        for (int n = 0; n < w.n; ++n, ++g) {
          const int kt = __ldg(pl.kt_idx + w.beg + n);
          const int ks = g % KST;
          if (n + KST < w.n) {   // L2 prefetch one ring ahead
            const int ka = __ldg(pl.kt_idx + w.beg + n + KST);
            for (int c = 0; c < C::NH; ++c) tma_prefetch_l2_4d(&tm_k, c * 64, w.hk, ka * BN, w.b);
          }
          if (g >= KST) mbar_wait(&bar.k_empty[ks], (g / KST - 1) & 1, wc);
          mbar_arrive_expect_tx(&bar.k_full[ks], TILE_BYTES);
          for (int c = 0; c < C::NH; ++c)
            tma_load_4d(base + OFF_K + ks * TILE_BYTES + c * HALF_BYTES, &tm_k, &bar.k_full[ks],
                        c * 64, w.hk, kt * BN, w.b);
        }
      }
      __syncwarp();
    }
    if (lane == 0 && bar.abort) {  // let copies in flight land before the CTA exits
      for (int n = max(0, g - KST); n < g; ++n)
        mbar_wait_final(&bar.k_full[n % KST], (n / KST) & 1, a.timeout_ns);
    }
  } else if (warp == WARP_PRODUCER_V) {
    // ------------------------------------------------ Q and V producer
    // A unit's Q is loaded once the previous unit's last S MMA has read its Q (q_empty).
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_v);
      int g = 0, nq = 0;
      for (int k = 0;; ++k) {
        const Unit w = take_unit(k, false);
        if (w.n < 0) break;
        if (w.n == 0) continue;
        if (nq > 0) mbar_wait(&bar.q_empty, (nq - 1) & 1, wc);
        mbar_arrive_expect_tx(&bar.q_full, TILE_BYTES);
        for (int c = 0; c < C::NH; ++c)
          tma_load_4d(base + OFF_Q + c * HALF_BYTES, &tm_q, &bar.q_full, c * 64, w.h, w.qt * BM,
                      w.b);
        ++nq;
        for (int n = 0; n < w.n; ++n, ++g) {
          const int kt = __ldg(pl.kt_idx + w.beg + n);
          const int vs = g % VST;
          if (n + VST < w.n) {
            const int ka = __ldg(pl.kt_idx + w.beg + n + VST);
            for (int c = 0; c < C::NH; ++c) tma_prefetch_l2_4d(&tm_v, c * 64, w.hk, ka * BN, w.b);
          }
          if (g >= VST) mbar_wait(&bar.v_empty[vs], (g / VST - 1) & 1, wc);
          mbar_arrive_expect_tx(&bar.v_full[vs], TILE_BYTES);
          for (int c = 0; c < C::NH; ++c)
            tma_load_4d(base + OFF_V + vs * TILE_BYTES + c * HALF_BYTES, &tm_v, &bar.v_full[vs],
                        c * 64, w.hk, kt * BN, w.b);
        }
      }
      if (bar.abort) {
        if (nq > 0) mbar_wait_final(&bar.q_full, (nq - 1) & 1, a.timeout_ns);
        for (int n = max(0, g - VST); n < g; ++n)
          mbar_wait_final(&bar.v_full[n % VST], (n / VST) & 1, a.timeout_ns);
      }
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------ MMA issuer
    // The per-tile issue loops are those of a one-unit CTA (the issue loop is sensitive to
    // any per-tile extra work); unit transitions sit outside them.  A unit's first two S
    // MMAs go out as soon as its Q has landed; its first PV (which overwrites O) waits
    // until the softmax warps have read the previous unit's O (o_free), so those S MMAs
    // overlap the previous unit's epilogue.  The whole warp walks the units
    // (use_half_path is warp-wide); lane 0 issues.
    constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0, 0);
    constexpr uint32_t IDESC_QK_HALF = idesc_bf16(BM, BN / 2, 0, 0);
    constexpr uint32_t IDESC_PV = idesc_bf16(BM, HD, 0, 1);
    const uint64_t dq0 = kmajor_desc(base_u32 + OFF_Q, 0);
    const uint64_t dk0 = kmajor_desc(base_u32 + OFF_K, 0);
    const uint64_t dv0 = mnmajor_desc(base_u32 + OFF_V, 0);
    // P_j sits (bf16 pairs) in the first 64 TMEM columns of S buffer j % 3.  S_{j+3}
    // reuses that buffer; it is issued after PV_j and tcgen05 MMAs of one thread run
    // in issue order, so PV_j has read P_j before S_{j+3} overwrites it.
    auto issue_pv = [&](int j, int j0, int empty) {
      const int sb = j % NSB;
      const int vs = j % VST;
      mbar_wait(&bar.p_ready[sb], (j / NSB) & 1, wc);
      mbar_wait(&bar.v_full[vs], (j / VST) & 1, wc);
      tc_fence_after();
      const uint64_t dv = dv0 + vs * stage_step(TILE_BYTES);
      const uint32_t ta = tmem + TM_S0 + sb * BN;
      if (empty == 0) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_bf16_ts(tmem + TM_O, ta + kk * 8, dv + mnmajor_step(kk), IDESC_PV,
                       (j > j0 || kk > 0) ? 1u : 0u);
      } else {
        const int k0 = empty == 1 ? 4 : 0;
#pragma unroll
        for (int kk = 0; kk < BN / 32; ++kk)
          umma_bf16_ts(tmem + TM_O, ta + (k0 + kk) * 8, dv + mnmajor_step(k0 + kk), IDESC_PV,
                       (j > j0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&bar.pv_done[sb]);
      umma_commit(&bar.v_empty[vs]);
    };
    auto issue_s = [&](int n, int empty) {
      const int sb = n % NSB;
      const int ks = n % KST;
      mbar_wait(&bar.k_full[ks], (n / KST) & 1, wc);
      tc_fence_after();
      const uint64_t dk = dk0 + ks * stage_step(TILE_BYTES);
      const uint32_t td = tmem + TM_S0 + sb * BN;
      if (empty == 0) {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_ss(td, dq0 + kmajor_step(kk, HALF_BYTES), dk + kmajor_step(kk, HALF_BYTES),
                       IDESC_QK, kk > 0 ? 1u : 0u);
      } else {
        const int hf = empty == 1 ? 1 : 0;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_bf16_ss(td + hf * 64, dq0 + kmajor_step(kk, HALF_BYTES),
                       dk + hf * ROWS64_STEP + kmajor_step(kk, HALF_BYTES), IDESC_QK_HALF,
                       kk > 0 ? 1u : 0u);
      }
      umma_commit(&bar.s_full[sb]);
      umma_commit(&bar.k_empty[ks]);
    };
    int g = 0, nq = 0;
    for (int k = 0;; ++k) {
      const Unit w = take_unit(k, true);
      if (w.n < 0) break;
      if (w.n == 0) continue;
      const bool halves = w.halves != 0;
      if (lane == 0 && !bar.abort) {
        mbar_wait(&bar.q_full, nq & 1, wc);
        const int g0 = g, g1 = g + w.n;
        const int gs = min(g0 + 2, g1);   // the S MMAs issued before the o_free wait
        if (!halves) {
          for (int n = g0; n < gs; ++n) issue_s(n, 0);
          if (nq > 0) mbar_wait(&bar.o_free, (nq - 1) & 1, wc);
          for (int n = gs; n < g1; ++n) {
            issue_s(n, 0);
            issue_pv(n - 2, g0, 0);
          }
          umma_commit(&bar.q_empty);   // the unit's last S has read Q
          for (int j = max(g0, g1 - 2); j < g1; ++j) issue_pv(j, g0, 0);
        } else {
          // flags one tile ahead of use, then a register history for the PV two tiles later
          int e_next = __ldg(pl.kt_cls + w.beg);
          uint32_t hist = 0u;
          for (int n = g0; n < g1; ++n) {
            const int empty = entry_empty_halves(e_next);
            hist = (hist << 2) | static_cast<uint32_t>(empty);
            if (n + 1 < g1) e_next = __ldg(pl.kt_cls + w.beg + (n + 1 - g0));
            issue_s(n, empty);
            if (n == gs - 1 && nq > 0) mbar_wait(&bar.o_free, (nq - 1) & 1, wc);
            if (n >= g0 + 2) issue_pv(n - 2, g0, (hist >> 4) & 3);
          }
          umma_commit(&bar.q_empty);
          for (int j = max(g0, g1 - 2); j < g1; ++j)
            issue_pv(j, g0, (hist >> (2 * (g1 - 1 - j))) & 3);
        }
      }
      // the other lanes wait here, suspended, instead of spinning on the next unit's slot
      // while lane 0 issues (divergent lanes of a warp share its issue slots)
      __syncwarp();
      g += w.n;
      ++nq;
    }
  } else {
    // ------------------------------------------------ softmax warps 0-7
    const int quarter = warp & 3;          // TMEM lane quarter
    const int half = warp >> 2;            // key columns [64 * half, 64 * half + 64)
    const int t = quarter * 32 + lane;     // row within the tile = TMEM lane
    const uint32_t quarter_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t lane_addr = quarter_addr + half * 64;
    const float sl2 = dm.scale_log2;
    float* red = reinterpret_cast<float*>(base + OFF_RED);  // [parity][half][row]
    int xc = 0;   // row-max / row-sum exchanges so far; its parity picks the red half

    // This thread's row of one unit: running max (log2 units) and sum, allowed key span,
    // block-map search hints.
    struct RowState {
      float m_run, l_run;
      RowSpan sp;
      MapCursor mcur;
    };
    auto start_row = [&](const Unit& w, RowState& rs) {
      rs.m_run = -INFINITY;
      rs.l_run = 0.f;
      rs.sp = row_span(a.mask, min(w.qt * BM + t, S - 1));
      rs.mcur = MapCursor{};
    };
    // Key tile n of unit w, whose tiles start at tile counter g0; IDLE: this warp's key
    // half holds no pair of the tile (only the barrier protocol).
    auto tile_step = [&](const Unit& w, int g0, int n, RowState& rs, auto idle_c) {
      constexpr bool IDLE = decltype(idle_c)::value;
      const int i = w.qt * BM + t;
      const int gn = g0 + n;
      const int st = gn % NSB;             // S buffer
      const uint32_t ph = (gn / NSB) & 1;
      const int rp = xc & 1;
      ++xc;
      float s[64];
      float mx = -INFINITY;
      if constexpr (!IDLE) {
        const int kt = __ldg(pl.kt_idx + w.beg + n);
        const int e = __ldg(pl.kt_cls + w.beg + n);
        const int c0 = kt * BN + half * 64;
        const bool masked = entry_class(e) != LCA_TILE_FULL || kt * BN + BN > S;
        uint32_t bits[2] = {0u, 0u};
        if (masked && i < S) row_tile_bits<2>(a.mask, w.hm, i, c0, rs.sp, bits, &rs.mcur);
        mbar_wait(&bar.s_full[st], ph, wc);
        __syncwarp();
        tc_fence_after();
        uint32_t r[64];
        tmem_ld64(lane_addr + TM_S0 + st * BN, r);
#pragma unroll
        for (int xx = 0; xx < 64; ++xx) s[xx] = __uint_as_float(r[xx]);
        if (masked) {
#pragma unroll
          for (int xx = 0; xx < 64; ++xx)
            if (!((bits[xx >> 5] >> (xx & 31)) & 1u)) s[xx] = -INFINITY;
        }
        float mq[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mq[kk] = s[kk];
#pragma unroll
        for (int xx = 8; xx < 64; xx += 8)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mq[kk] = fmaxf(mq[kk], s[xx + kk]);
        mx = fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])),
                   fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7])));
      } else {
        mbar_wait(&bar.s_full[st], ph, wc);
      }
      red[(rp * 2 + half) * BM + t] = mx;
      named_bar_sync(BAR_SOFTMAX, SOFTMAX_THREADS);
      mx = fmaxf(mx, red[(rp * 2 + (half ^ 1)) * BM + t]);
      const float mt = mx * sl2;
      float alpha = 1.f;
      bool rescale = false;
      if (mt > rs.m_run + RESCALE_THRESHOLD) {
        rescale = (rs.m_run != -INFINITY);
        alpha = ex2_approx(rs.m_run - mt);
        rs.l_run *= alpha;
        rs.m_run = mt;
      }
      // never on a unit's first tile (m_run starts at -inf), so never while O still holds
      // the previous unit's result
      if (__any_sync(0xFFFFFFFFu, rescale)) {
        // O holds this unit's P V so far: wait for its last PV, scale, store back
        const int pj = gn - 1;
        mbar_wait(&bar.pv_done[pj % NSB], (pj / NSB) & 1, wc);
        __syncwarp();
        tc_fence_after();
        const float f = rescale ? alpha : 1.f;
        uint32_t o[OCOLS];
        tmem_ldn<OCOLS>(quarter_addr + TM_O + half * OCOLS, o);
#pragma unroll
        for (int xx = 0; xx < OCOLS; ++xx) o[xx] = __float_as_uint(__uint_as_float(o[xx]) * f);
        tmem_stn<OCOLS>(quarter_addr + TM_O + half * OCOLS, o);
      }
      if constexpr (!IDLE) {
        const float m_use = (rs.m_run == -INFINITY) ? 0.f : rs.m_run;
        float ls[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) ls[kk] = 0.f;
#pragma unroll
        for (int xx = 0; xx < 64; ++xx) {
          s[xx] = ex2_approx(fmaf(s[xx], sl2, -m_use));
          ls[xx & 7] += s[xx];
        }
        rs.l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        uint32_t pk[32];
#pragma unroll
        for (int xx = 0; xx < 32; ++xx) pk[xx] = pack_bf16x2(s[2 * xx], s[2 * xx + 1]);
        tmem_st32(quarter_addr + TM_S0 + st * BN + half * 32, pk);
      }
      tc_fence_before();
      mbar_arrive(&bar.p_ready[st]);
    };
    // tiles [n0, w.n) of unit w; rows whose list runs the half-width path check each
    // tile's flags, the others run the loop without any flag handling
    auto run_tiles = [&](const Unit& w, int g0, int n0, RowState& rs) {
      if (!w.halves) {
        for (int n = n0; n < w.n; ++n) tile_step(w, g0, n, rs, std::false_type{});
      } else {
        for (int n = n0; n < w.n; ++n) {
          if ((entry_empty_halves(__ldg(pl.kt_cls + w.beg + n)) >> half) & 1)
            tile_step(w, g0, n, rs, std::true_type{});
          else
            tile_step(w, g0, n, rs, std::false_type{});
        }
      }
    };
    // Epilogue, first part (no wait on the MMAs): l over the whole row, LSE =
    // (m + log2 l) * ln 2 stored; returns 1 / l (0 for a row without allowed keys).
    auto epilogue_sum = [&](const Unit& w, const RowState& rs) {
      const int i = w.qt * BM + t;
      const int pe = xc & 1;
      ++xc;
      red[(pe * 2 + half) * BM + t] = rs.l_run;
      named_bar_sync(BAR_SOFTMAX, SOFTMAX_THREADS);
      const float l_tot = rs.l_run + red[(pe * 2 + (half ^ 1)) * BM + t];
      if (i < S && half == 0) {
        const float lse = (l_tot > 0.f) ? (rs.m_run + __log2f(l_tot)) * 0.69314718055994531f
                                        : -INFINITY;
        a.lse[(static_cast<int64_t>(w.b) * dm.h_q + w.h) * S + i] = lse;
      }
      return (l_tot > 0.f) ? 1.f / l_tot : 0.f;
    };
    // Epilogue, second part: after the unit's last PV, O = acc / l (bf16) to orow (null
    // past S); then O is free for the next unit.
    auto epilogue_out = [&](int last_tile, float inv, __nv_bfloat16* orow) {
      mbar_wait(&bar.pv_done[last_tile % NSB], (last_tile / NSB) & 1, wc);
      __syncwarp();
      tc_fence_after();
      uint32_t o[OCOLS];
      tmem_ldn<OCOLS>(quarter_addr + TM_O + half * OCOLS, o);
      tc_fence_before();
      mbar_arrive(&bar.o_free);
      if (orow != nullptr) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int v = 0; v < OCOLS / 8; ++v) {
          const int xx = v * 8;
          uint4 ww;
          ww.x = pack_bf16x2(__uint_as_float(o[xx + 0]) * inv, __uint_as_float(o[xx + 1]) * inv);
          ww.y = pack_bf16x2(__uint_as_float(o[xx + 2]) * inv, __uint_as_float(o[xx + 3]) * inv);
          ww.z = pack_bf16x2(__uint_as_float(o[xx + 4]) * inv, __uint_as_float(o[xx + 5]) * inv);
          ww.w = pack_bf16x2(__uint_as_float(o[xx + 6]) * inv, __uint_as_float(o[xx + 7]) * inv);
          dst[v] = ww;
        }
      }
    };

    // Unit transitions: the next unit's row set-up and first tile run between the two
    // parts of the current unit's epilogue.  Its S is computed by then (the MMA warp
    // issues a unit's first S MMAs as soon as its Q has landed), and the first tile never
    // touches O, so the wait for the last PV and the set-up's global loads overlap work
    // the tensor pipe can use.
    int g = 0;    // tile counter (S buffers, barrier phases)
    int k = 0;
    Unit w = take_unit(0, true);
    RowState rs{};
    bool started = false;   // rs holds w's row and w's first tile has run
    while (w.n >= 0) {
      if (w.n == 0) {   // no allowed key anywhere in the tile: O = 0, LSE = -inf
        const int i = w.qt * BM + t;
        if (i < S) {
          uint4* dst = reinterpret_cast<uint4*>(a.o + (static_cast<int64_t>(w.b) * S + i) *
                                                          a.o_row_stride +
                                                static_cast<int64_t>(w.h) * HD + half * OCOLS);
#pragma unroll
          for (int v = 0; v < OCOLS / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
          if (half == 0) a.lse[(static_cast<int64_t>(w.b) * dm.h_q + w.h) * S + i] = -INFINITY;
        }
        w = take_unit(++k, true);
        started = false;
        continue;
      }
      if (!started) start_row(w, rs);
      run_tiles(w, g, started ? 1 : 0, rs);   // one call site: one copy of the loops
      const float inv = epilogue_sum(w, rs);
      const int iw = w.qt * BM + t;
      __nv_bfloat16* orow = iw < S ? a.o + (static_cast<int64_t>(w.b) * S + iw) * a.o_row_stride +
                                         static_cast<int64_t>(w.h) * HD + half * OCOLS
                                   : nullptr;
      const int last_tile = g + w.n - 1;
      const Unit wn = take_unit(++k, true);
      RowState rn{};
      started = false;
      if (wn.n > 0) {
        // a tile with an empty key half is partial, so this warp's half is masked out
        // in full there: the full-width step is correct for it too
        start_row(wn, rn);
        tile_step(wn, g + w.n, 0, rn, std::false_type{});
        started = true;
      }
      epilogue_out(last_tile, inv, orow);
      g += w.n;
      w = wn;
      rs = rn;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

}  // namespace

size_t fwd_smem_bytes() { return Cfg<128>::SMEM_BYTES; }

template <int HD>
static cudaError_t launch_fwd_hd(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const FwdArgs& args, int n_ctas,
                                 cudaStream_t st) {
  constexpr uint32_t smem = Cfg<HD>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<HD><<<n_ctas, NUM_THREADS, smem, st>>>(tq, tk, tv, args);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& args, int n_ctas, cudaStream_t st) {
  if (args.n_units == 0) return cudaSuccess;
  // the unit counter starts at 0 for every launch
  cudaError_t e = cudaMemsetAsync(args.unit_counter, 0, sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  if (args.dims.head_dim == 64) return launch_fwd_hd<64>(tq, tk, tv, args, n_ctas, st);
  return launch_fwd_hd<128>(tq, tk, tv, args, n_ctas, st);
}

}  // namespace lca
