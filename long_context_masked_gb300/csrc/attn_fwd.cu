// Forward pass of mask-aware exact softmax attention on sm_103a.
//
// Computes O = softmax(scale * Q K^T + mask) V and LSE per query row, the operation
// the LongCA-bench kernels are measured on ("Long-Context Attention Benchmark":
// summary page, abstract and sections 2.2 / 3.1; reading note, "Key design" 2).
//
// One CTA owns one 128-row query tile of one query head and walks that tile's list
// of non-skipped key tiles (from the tile plan, longest lists launched first):
//   warps 8, 10 TMA producers: Q once and the K tiles (warp 8), the V tiles (warp 10),
//               each into a 3-stage ring;
//   warp 9      TMEM owner and MMA issuer: S_n = Q K_n^T (tcgen05, both operands in
//               shared memory, fp32 in TMEM, three buffers) and O += P_{n-2} V_{n-2}
//               with P read from TMEM (accumulated in TMEM).  PV trails S by two
//               tiles so that S_{n+1} is computed while the softmax works on S_n;
//   warps 0-7   softmax, two threads per query row (warps w and w+4 share TMEM lanes
//               and take key columns 0-63 / 64-127): read S_n from TMEM, apply the mask
//               bits only on partial or ragged tiles, combine the two halves' row
//               maxima through shared memory, online softmax in fp32 with exp2, write P
//               (bf16 pairs) back into the TMEM columns of S_n for the PV MMA, rescale
//               the O accumulator in TMEM when the running max moves by more than 2^8
//               (exact after the final 1/l normalisation), then the epilogue.
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
  static constexpr uint32_t OFF_RED = OFF_BAR + 256;          // row-max / row-sum exchange
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

struct Bars {
  uint64_t q_full;
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[NSB], p_ready[NSB], pv_done[NSB];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block overflows its shared-memory slot");

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

  // ---- work item
  const AttnDims& dm = a.dims;
  const PlanDev& pl = a.plan;
  const int per_item = dm.heads_per_map * dm.batch;
  int item, rem;
  chunked_item(blockIdx.x, per_item, pl.map_heads * pl.n_qt, dm.chunk, item, rem);
  const int sub = rem % dm.heads_per_map;
  const int b = rem / dm.heads_per_map;
  const int row = __ldg(pl.work_q + item);
  const int hm = row / pl.n_qt;
  const int qt = row - hm * pl.n_qt;
  const int h = hm * dm.heads_per_map + sub;
  const int hk = h / dm.group;
  const int beg = __ldg(pl.rowptr + row);
  const int n_tiles = __ldg(pl.rowptr + row + 1) - beg;
  const int S = dm.seqlen;

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
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

  if (warp == WARP_PRODUCER || warp == WARP_PRODUCER_V) {
    // ------------------------------------------------ TMA producers
    // one warp streams Q and the K tiles, another the V tiles, so a K load never
    // queues behind the release of a V stage (V stages are freed two tiles later).
    if (warp == WARP_PRODUCER && lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(&bar.q_full, TILE_BYTES);
      for (int c = 0; c < C::NH; ++c)
        tma_load_4d(base + OFF_Q + c * HALF_BYTES, &tm_q, &bar.q_full, c * 64, h, qt * BM, b);
      for (int n = 0; n < n_tiles; ++n) {
        const int kt = __ldg(pl.kt_idx + beg + n);
        const int ks = n % KST;
        if (n + KST < n_tiles) {   // L2 prefetch one ring ahead
          const int ka = __ldg(pl.kt_idx + beg + n + KST);
          for (int c = 0; c < C::NH; ++c) tma_prefetch_l2_4d(&tm_k, c * 64, hk, ka * BN, b);
        }
        if (n >= KST) mbar_wait(&bar.k_empty[ks], (n / KST - 1) & 1, wc);
        mbar_arrive_expect_tx(&bar.k_full[ks], TILE_BYTES);
        for (int c = 0; c < C::NH; ++c)
          tma_load_4d(base + OFF_K + ks * TILE_BYTES + c * HALF_BYTES, &tm_k, &bar.k_full[ks],
                      c * 64, hk, kt * BN, b);
      }
      if (bar.abort) {  // let copies in flight land before the CTA exits
        mbar_wait_final(&bar.q_full, 0, a.timeout_ns);
        for (int n = max(0, n_tiles - KST); n < n_tiles; ++n)
          mbar_wait_final(&bar.k_full[n % KST], (n / KST) & 1, a.timeout_ns);
      }
    } else if (warp == WARP_PRODUCER_V && lane == 0) {
      tma_prefetch_desc(&tm_v);
      for (int n = 0; n < n_tiles; ++n) {
        const int kt = __ldg(pl.kt_idx + beg + n);
        const int vs = n % VST;
        if (n + VST < n_tiles) {
          const int ka = __ldg(pl.kt_idx + beg + n + VST);
          for (int c = 0; c < C::NH; ++c) tma_prefetch_l2_4d(&tm_v, c * 64, hk, ka * BN, b);
        }
        if (n >= VST) mbar_wait(&bar.v_empty[vs], (n / VST - 1) & 1, wc);
        mbar_arrive_expect_tx(&bar.v_full[vs], TILE_BYTES);
        for (int c = 0; c < C::NH; ++c)
          tma_load_4d(base + OFF_V + vs * TILE_BYTES + c * HALF_BYTES, &tm_v, &bar.v_full[vs],
                      c * 64, hk, kt * BN, b);
      }
      if (bar.abort) {
        for (int n = max(0, n_tiles - VST); n < n_tiles; ++n)
          mbar_wait_final(&bar.v_full[n % VST], (n / VST) & 1, a.timeout_ns);
      }
    }
  } else if (warp == WARP_MMA) {
    // ------------------------------------------------ MMA issuer
    // Rows that use_half_path turns down (every dense mask) run the plain loop; the
    // flag-aware loop is a separate instantiation, so the plain one carries no per-tile
    // flag handling (the issue loop is sensitive to any extra work).
    const bool halves = use_half_path(pl.kt_cls + beg, n_tiles, HALF_SHARE, lane);
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t IDESC_QK_HALF = idesc_bf16(BM, BN / 2, 0, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16(BM, HD, 0, 1);
      const uint64_t dq0 = kmajor_desc(base_u32 + OFF_Q, 0);
      const uint64_t dk0 = kmajor_desc(base_u32 + OFF_K, 0);
      const uint64_t dv0 = mnmajor_desc(base_u32 + OFF_V, 0);
      // P_j sits (bf16 pairs) in the first 64 TMEM columns of S buffer j % 3.  S_{j+3}
      // reuses that buffer; it is issued after PV_j and tcgen05 MMAs of one thread run
      // in issue order, so PV_j has read P_j before S_{j+3} overwrites it (and PV_j
      // waited for the softmax of tile j, so S_j was consumed).
      auto issue_pv = [&](int j, int empty) {
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
                         (j > 0 || kk > 0) ? 1u : 0u);
        } else {
          // the four k-steps of the other key half only
          const int k0 = empty == 1 ? 4 : 0;
#pragma unroll
          for (int kk = 0; kk < BN / 32; ++kk)
            umma_bf16_ts(tmem + TM_O, ta + (k0 + kk) * 8, dv + mnmajor_step(k0 + kk), IDESC_PV,
                         (j > 0 || kk > 0) ? 1u : 0u);
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
          // one key half only: its 64 K rows into its 64 S columns
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
      mbar_wait(&bar.q_full, 0, wc);
      if (!halves) {
        for (int n = 0; n < n_tiles; ++n) {
          issue_s(n, 0);
          if (n >= 2) issue_pv(n - 2, 0);
        }
        for (int j = max(0, n_tiles - 2); j < n_tiles; ++j) issue_pv(j, 0);
      } else {
        // The flags reach the issuer one tile ahead of use (a load consumed right away
        // holds the issue of the next MMAs back) and stay in a register history, two
        // bits per tile, for the PV MMA two tiles later.
        int e_next = n_tiles > 0 ? __ldg(pl.kt_cls + beg) : 0;
        uint32_t hist = 0u;
        for (int n = 0; n < n_tiles; ++n) {
          const int empty = entry_empty_halves(e_next);
          hist = (hist << 2) | static_cast<uint32_t>(empty);
          if (n + 1 < n_tiles) e_next = __ldg(pl.kt_cls + beg + n + 1);
          issue_s(n, empty);
          if (n >= 2) issue_pv(n - 2, (hist >> 4) & 3);
        }
        for (int j = max(0, n_tiles - 2); j < n_tiles; ++j)
          issue_pv(j, (hist >> (2 * (n_tiles - 1 - j))) & 3);
      }
    }
  } else {
    // ------------------------------------------------ softmax warps 0-7
    const int quarter = warp & 3;          // TMEM lane quarter
    const int half = warp >> 2;            // key columns [64 * half, 64 * half + 64)
    const int t = quarter * 32 + lane;     // row within the tile = TMEM lane
    const int i = qt * BM + t;
    const uint32_t quarter_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t lane_addr = quarter_addr + half * 64;
    const RowSpan sp = row_span(a.mask, min(i, S - 1));
    MapCursor mcur;
    const float sl2 = dm.scale_log2;
    float* red = reinterpret_cast<float*>(base + OFF_RED);  // [parity][half][row]
    float m_run = -INFINITY;
    float l_run = 0.f;

    // One key tile; IDLE: this warp's key half holds no pair of the tile (no S to read,
    // no P to write, only the row-max exchange and the O rescale).  Two instantiations
    // keep the common path's code exactly that of a full-width tile.
    auto tile_step = [&](int n, auto idle_c) {
      constexpr bool IDLE = decltype(idle_c)::value;
      const int st = n % NSB;             // S buffer
      const uint32_t ph = (n / NSB) & 1;
      const int rp = n & 1;               // max-exchange parity
      float s[64];
      float mx = -INFINITY;
      if constexpr (!IDLE) {
        const int kt = __ldg(pl.kt_idx + beg + n);
        const int e = __ldg(pl.kt_cls + beg + n);
        const int c0 = kt * BN + half * 64;
        const bool masked = entry_class(e) != LCA_TILE_FULL || kt * BN + BN > S;
        uint32_t bits[2] = {0u, 0u};
        if (masked && i < S) row_tile_bits<2>(a.mask, hm, i, c0, sp, bits, &mcur);
        mbar_wait(&bar.s_full[st], ph, wc);
        __syncwarp();
        tc_fence_after();
        uint32_t r[64];
        tmem_ld64(lane_addr + TM_S0 + st * BN, r);
#pragma unroll
        for (int x = 0; x < 64; ++x) s[x] = __uint_as_float(r[x]);
        if (masked) {
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (!((bits[x >> 5] >> (x & 31)) & 1u)) s[x] = -INFINITY;
        }
        float mq[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mq[k] = s[k];
#pragma unroll
        for (int x = 8; x < 64; x += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) mq[k] = fmaxf(mq[k], s[x + k]);
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
      if (mt > m_run + RESCALE_THRESHOLD) {
        rescale = (m_run != -INFINITY);
        alpha = ex2_approx(m_run - mt);
        l_run *= alpha;
        m_run = mt;
      }
      if (__any_sync(0xFFFFFFFFu, rescale)) {
        // O holds P_0..P_{n-1} V: wait for the last PV, scale this half row, store back
        const int pj = n - 1;
        mbar_wait(&bar.pv_done[pj % NSB], (pj / NSB) & 1, wc);
        __syncwarp();
        tc_fence_after();
        const float f = rescale ? alpha : 1.f;
        uint32_t o[OCOLS];
        tmem_ldn<OCOLS>(quarter_addr + TM_O + half * OCOLS, o);
#pragma unroll
        for (int x = 0; x < OCOLS; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
        tmem_stn<OCOLS>(quarter_addr + TM_O + half * OCOLS, o);
      }
      if constexpr (!IDLE) {
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        float ls[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ls[k] = 0.f;
#pragma unroll
        for (int x = 0; x < 64; ++x) {
          s[x] = ex2_approx(fmaf(s[x], sl2, -m_use));
          ls[x & 7] += s[x];
        }
        l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        // P (bf16 pairs) into the first 64 columns of this S buffer; both halves of the
        // row finished reading S before the max exchange barrier above
        uint32_t pk[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) pk[x] = pack_bf16x2(s[2 * x], s[2 * x + 1]);
        tmem_st32(quarter_addr + TM_S0 + st * BN + half * 32, pk);
      }
      tc_fence_before();
      mbar_arrive(&bar.p_ready[st]);
    };
    if (!use_half_path(pl.kt_cls + beg, n_tiles, HALF_SHARE, lane)) {
      for (int n = 0; n < n_tiles; ++n) tile_step(n, std::false_type{});
    } else {
      for (int n = 0; n < n_tiles; ++n) {
        if ((entry_empty_halves(__ldg(pl.kt_cls + beg + n)) >> half) & 1)
          tile_step(n, std::true_type{});
        else
          tile_step(n, std::false_type{});
      }
    }

    // ---- epilogue: O = acc / l (bf16), LSE = (m + log2 l) * ln 2
    if (n_tiles > 0) {
      const int pj = n_tiles - 1;
      mbar_wait(&bar.pv_done[pj % NSB], (pj / NSB) & 1, wc);
      __syncwarp();
      tc_fence_after();
    }
    // row-sum exchange in the slots of parity n_tiles & 1: last written for tile
    // n_tiles - 2, whose reads both threads finished before the last tile's barrier
    const int pe = n_tiles & 1;
    red[(pe * 2 + half) * BM + t] = l_run;
    named_bar_sync(BAR_SOFTMAX, SOFTMAX_THREADS);
    const float l_tot = l_run + red[(pe * 2 + (half ^ 1)) * BM + t];
    const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
    uint32_t o[OCOLS];
    if (n_tiles > 0) {
      tmem_ldn<OCOLS>(quarter_addr + TM_O + half * OCOLS, o);
    } else {
#pragma unroll
      for (int x = 0; x < OCOLS; ++x) o[x] = 0u;
    }
    if (i < S) {
      __nv_bfloat16* orow = a.o + (static_cast<int64_t>(b) * S + i) * a.o_row_stride +
                            static_cast<int64_t>(h) * HD + half * OCOLS;
      uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int v = 0; v < OCOLS / 8; ++v) {
        const int x = v * 8;
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(o[x + 0]) * inv, __uint_as_float(o[x + 1]) * inv);
        w.y = pack_bf16x2(__uint_as_float(o[x + 2]) * inv, __uint_as_float(o[x + 3]) * inv);
        w.z = pack_bf16x2(__uint_as_float(o[x + 4]) * inv, __uint_as_float(o[x + 5]) * inv);
        w.w = pack_bf16x2(__uint_as_float(o[x + 6]) * inv, __uint_as_float(o[x + 7]) * inv);
        dst[v] = w;
      }
      if (half == 0) {
        const float lse = (l_tot > 0.f) ? (m_run + __log2f(l_tot)) * 0.69314718055994531f
                                        : -INFINITY;
        a.lse[(static_cast<int64_t>(b) * dm.h_q + h) * S + i] = lse;
      }
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
                                 const CUtensorMap& tv, const FwdArgs& args, int n_blocks,
                                 cudaStream_t st) {
  constexpr uint32_t smem = Cfg<HD>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HD>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<HD><<<n_blocks, NUM_THREADS, smem, st>>>(tq, tk, tv, args);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& args, int n_blocks, cudaStream_t st) {
  if (n_blocks == 0) return cudaSuccess;
  if (args.dims.head_dim == 64) return launch_fwd_hd<64>(tq, tk, tv, args, n_blocks, st);
  return launch_fwd_hd<128>(tq, tk, tv, args, n_blocks, st);
}

}  // namespace lca
