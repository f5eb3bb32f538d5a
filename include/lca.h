/*
 * lca.h - C ABI of the GB300 (sm_103a) mask-aware exact softmax attention library.
 *
 * The operation is standard softmax attention under an attention mask, forward and
 * backward, the computation every kernel of the LongCA-bench benchmark performs
 * ("Long-Context Attention Benchmark: From Kernel Efficiency to Distributed Context
 * Parallelism": summary page, abstract and section 2.2 "Attention Kernel"; reading
 * note, "Key design" 1-2).  For batch b, query head h (KV head h / g, g = H_q / H_kv)
 * and the mask M of the head's map head:
 *
 *     s_ij = scale * <q_i, k_j>,  LSE_i = ln sum_{j: M_ij} exp(s_ij),
 *     P_ij = M_ij exp(s_ij - LSE_i),  O_i = sum_j P_ij v_j,
 *     dV_j = sum_i P_ij dO_i,  dP_ij = <dO_i, v_j>,  D_i = <dO_i, O_i>,
 *     dS_ij = P_ij (dP_ij - D_i),  dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i
 *
 * (dK/dV of a KV head sum over its g query heads).  A query row with no allowed key
 * gets O = 0, LSE = -inf and dQ = 0, and adds nothing to dK/dV.
 *
 * Conventions shared by every entry point:
 *  - Tensor arguments are DEVICE pointers owned by the caller.  The library owns only
 *    the plan (freed with lca_plan_destroy) and never frees caller memory.
 *  - Work is enqueued on the given cudaStream_t (passed as void*, NULL = legacy default
 *    stream).  lca_mask_build is the one call that synchronises the stream (it reads
 *    the size of the tile lists back to size them).
 *  - Arguments are validated on the host before anything is launched; a failed check
 *    returns LCA_ERR_INVALID_ARG / LCA_ERR_UNSUPPORTED / LCA_ERR_PLAN_MISMATCH and
 *    launches nothing.  No C++ exception crosses this interface.
 *  - Device-side waits inside the kernels are bounded; a wait that runs out sets a
 *    device error word, which lca_get_last_device_error reports as LCA_ERR_TIMEOUT.
 */
#ifndef LCA_H_
#define LCA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LCA_OK = 0,
  LCA_ERR_INVALID_ARG = 1,   /* null pointer, inconsistent size, bad descriptor         */
  LCA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim not 64 or 128) */
  LCA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed                       */
  LCA_ERR_OOM = 4,           /* device allocation for the plan failed                   */
  LCA_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out                      */
  LCA_ERR_PLAN_MISMATCH = 6  /* plan built for another seqlen / head layout             */
} lca_status;

/* Mask types: the benchmark's static masks and its two dynamic block-sparse masks
 * (summary page, section 2.1.1 "Input Mask Patterns"; reading note, "Key design" 1).
 * Query i may attend to key j when (0-indexed, S = seqlen):
 *   FULL                   always
 *   CAUSAL                 j <= i
 *   SLIDING_WINDOW         j <= i && i - j < window
 *   FULL_DOCUMENT          doc(i) == doc(j)                      (docs from cu_seqlens)
 *   CAUSAL_DOCUMENT        doc(i) == doc(j) && j <= i
 *   SLIDING_WINDOW_DOCUMENT doc(i) == doc(j) && j <= i && i - j < window
 *   PREFIX_LM              j < prefix_len || j <= i
 *   SHARED_QUESTION        j <= i && (seg(j) == seg(i) || seg(j) == 0)  (segment 0 = question)
 *   GLOBAL_SLIDING         base_causal: j <= i && (j < num_global || i - j < window)
 *                          otherwise:   j < num_global || i < num_global || |i - j| < window
 *   CAUSAL_BLOCKWISE       j / block <= i / block
 *   BLOCK_CAUSAL_DOCUMENT  doc(i) == doc(j) && (j - st) / block <= (i - st) / block,
 *                          st = start of the document
 *   BLOCK_SPARSE_UNIFORM   map[h_m][i / block][j / block]
 *   BLOCK_SPARSE_VARIABLE  map[h_m][rb(i)][cb(j)], rb/cb from the head's row/column offsets
 * Both block-sparse types are ANDed with j <= i when base_causal != 0 and with
 * doc(i) == doc(j) when cu_seqlens is given (num_segments > 0). */
typedef enum {
  LCA_FULL = 0,
  LCA_CAUSAL = 1,
  LCA_SLIDING_WINDOW = 2,
  LCA_FULL_DOCUMENT = 3,
  LCA_CAUSAL_DOCUMENT = 4,
  LCA_PREFIX_LM = 5,
  LCA_SHARED_QUESTION = 6,
  LCA_GLOBAL_SLIDING = 7,
  LCA_CAUSAL_BLOCKWISE = 8,
  LCA_BLOCK_CAUSAL_DOCUMENT = 9,
  LCA_BLOCK_SPARSE_UNIFORM = 10,
  LCA_BLOCK_SPARSE_VARIABLE = 11,
  LCA_SLIDING_WINDOW_DOCUMENT = 12   /* the sliding window inside each document */
} lca_mask_type;

/* Class of one (query tile, key tile) pair; tiles on the last row/column are clipped
 * at S and only in-range pairs count. */
typedef enum {
  LCA_TILE_SKIP = 0,    /* no allowed pair                */
  LCA_TILE_FULL = 1,    /* every in-range pair allowed    */
  LCA_TILE_PARTIAL = 2  /* some pairs allowed, some not   */
} lca_tile_class;

/* Tile byte: the class in bits 0-1 and, for a non-skipped tile, one flag per half of
 * the tile that holds no allowed in-range pair.  The benchmark's sparse masks keep
 * blocks of a grid finer than a 128 x 128 tile (64-token blocks; summary page,
 * appendix A.2 "Block Partitioning"), which leaves tiles with pairs in one half only;
 * the kernels leave an empty half out.  A skipped tile's byte is 0.
 *   cls     the whole tile byte (bits 0-5);
 *   kt_cls  row-list entry: the class and the key-half flags (tile byte & 15);
 *   qt_cls  column-list entry: the class and the query-half flags moved down to
 *           bits 2-3 ((byte & 3) | ((byte >> 4) << 2)).
 * In either list, bits 2-3 are the flags of the halves the list's kernel iterates
 * against: (entry >> 2) & 1 for the first half, (entry >> 3) & 1 for the second. */
enum {
  LCA_TILE_CLASS_MASK = 3,
  LCA_TILE_KEY_HALF0_EMPTY = 4,     /* key columns [0, tile_k / 2)      */
  LCA_TILE_KEY_HALF1_EMPTY = 8,     /* key columns [tile_k / 2, tile_k) */
  LCA_TILE_QUERY_HALF0_EMPTY = 16,  /* query rows [0, tile_q / 2)       */
  LCA_TILE_QUERY_HALF1_EMPTY = 32   /* query rows [tile_q / 2, tile_q)  */
};

/* Mask descriptor ("unified data format" of the benchmark: summary page, section 2.2;
 * reading note, "Key design" 2).  Fields a type does not use are ignored.
 * Device arrays are read during lca_mask_build only (the plan keeps its own copies). */
typedef struct {
  int32_t type;          /* lca_mask_type                                               */
  int32_t seqlen;        /* S, 1 <= S <= 2^20                                           */
  int32_t window;        /* SLIDING_WINDOW(_DOCUMENT), GLOBAL_SLIDING: >= 1             */
  int32_t num_global;    /* GLOBAL_SLIDING: >= 0                                        */
  int32_t prefix_len;    /* PREFIX_LM: 0 <= prefix_len <= S                             */
  int32_t block;         /* CAUSAL_BLOCKWISE, BLOCK_CAUSAL_DOCUMENT, BLOCK_SPARSE_UNIFORM */
  int32_t base_causal;   /* GLOBAL_SLIDING and block-sparse types (see above)           */
  int32_t num_segments;  /* entries of cu_seqlens minus one; 0 = no segments            */
  const int32_t* cu_seqlens;  /* device int32 [num_segments + 1], 0 = c_0 <= ... <= c_n = S;
                                 documents (DOCUMENT types incl. SLIDING_WINDOW_DOCUMENT, BLOCK_CAUSAL_DOCUMENT,
                                 optional for block-sparse) or segments (SHARED_QUESTION,
                                 segment 0 = question, >= 2 segments)                 */
  int32_t map_heads;     /* block-sparse: H_m = 1, H_kv (GQA: shared in a KV group) or H_q */
  int32_t n_row_blocks;  /* block-sparse: rows of each head's map                        */
  int32_t n_col_blocks;  /* block-sparse: columns of each head's map                     */
  const int32_t* row_block_offsets; /* VARIABLE: device int32 [map_heads][n_row_blocks+1],
                                       ascending from 0 to S per head (trailing entries
                                       equal to S pad heads with fewer blocks)           */
  const int32_t* col_block_offsets; /* VARIABLE: device int32 [map_heads][n_col_blocks+1] */
  const uint8_t* block_map;         /* block-sparse: device uint8 (0/1)
                                       [map_heads][n_row_blocks][n_col_blocks]           */
} lca_mask_desc;

/* Tensor shape.  Q, O, dO, dQ: [batch, seqlen, h_q, head_dim] bf16 with row stride
 * *_row_stride elements between consecutive positions (>= h_q * head_dim, multiple of
 * 8), heads packed (stride head_dim), batch stride seqlen * row_stride.  K, V, dK, dV:
 * [batch, seqlen, h_kv, head_dim] likewise.  Every tensor has its own row stride, so
 * inputs may be slices of a packed QKV (or KV) tensor while the gradients are separate
 * buffers, or the other way round.  The four gradient-side strides are read by
 * lca_attn_bwd only; 0 there means "the row stride of the matching input": dO as O,
 * dQ as Q, dK as K, dV as V.  LSE and D: [batch, h_q, seqlen] fp32, contiguous.  All
 * base pointers 16-byte aligned.  Masks with segments or block maps require
 * batch == 1. */
typedef struct {
  int32_t batch, seqlen, h_q, h_kv, head_dim;
  int64_t q_row_stride, k_row_stride, v_row_stride, o_row_stride;
  int64_t do_row_stride, dq_row_stride, dk_row_stride, dv_row_stride;
} lca_shape;

typedef struct lca_plan lca_plan; /* opaque; owns its device buffers */

/* Sizes of a plan's arrays, for lca_plan_export, and its device footprint. */
typedef struct {
  int32_t seqlen, tile_q, tile_k, n_qt, n_kt, map_heads, mask_type;
  int64_t nnz;         /* non-skipped tiles over all map heads                  */
  int64_t n_partial;   /* of which PARTIAL                                      */
  int64_t device_bytes;  /* device memory the plan holds (its arrays and the copies
                            of the descriptor's arrays)                          */
} lca_plan_info;

/* Build the tile plan of a mask (step "mask build": classify every (query tile, key
 * tile) pair as skip/full/partial, compact the non-skipped key tiles of every query
 * tile, transpose to the query tiles of every key tile, order both lists
 * longest-first, and count the allowed pairs of every map head exactly).
 * tile_q, tile_k in {64, 128}.  On success *out receives a new plan (LCA_OK); on any
 * error *out is left NULL.  Synchronises `stream`. */
lca_status lca_mask_build(const lca_mask_desc* desc, int tile_q, int tile_k, void* stream,
                          lca_plan** out);

lca_status lca_plan_get_info(const lca_plan* plan, lca_plan_info* info);

/* Copy a plan's arrays to HOST buffers (any pointer may be NULL to skip it), sizes
 * from lca_plan_info: cls [map_heads*n_qt*n_kt] uint8 tile bytes (class and empty-half
 * flags, see LCA_TILE_CLASS_MASK); rowptr [map_heads*n_qt+1],
 * kt_idx [nnz], kt_cls [nnz] (per (h_m, qt) row, ascending kt); colptr
 * [map_heads*n_kt+1], qt_idx [nnz], qt_cls [nnz] (per (h_m, kt) column, ascending qt);
 * work_q [map_heads*n_qt], work_k [map_heads*n_kt] (row/column indices h_m*n + t,
 * longest list first, ties by index); n_valid [map_heads] int64 (allowed pairs).
 * Synchronises the device. */
lca_status lca_plan_export(const lca_plan* plan, uint8_t* cls, int32_t* rowptr, int32_t* kt_idx,
                           uint8_t* kt_cls, int32_t* colptr, int32_t* qt_idx, uint8_t* qt_cls,
                           int32_t* work_q, int32_t* work_k, int64_t* n_valid);

void lca_plan_destroy(lca_plan* plan);

/* Forward: O (bf16) and LSE (fp32, natural log) for all heads and rows.
 * Requires head_dim 128 or 64, plan tile_q == 128, tile_k == 128, plan seqlen ==
 * shape->seqlen, plan map_heads in {1, h_kv, h_q}; a plan with 64-row or 64-column tiles
 * returns LCA_ERR_UNSUPPORTED (the attention kernels run 128 x 128 tiles only, and
 * leave out the empty 64-row / 64-column halves of a tile instead: see the tile-byte
 * flags above).  Reads q/k/v/o_row_stride only.  softmax_scale <= 0 means
 * 1/sqrt(head_dim).  The launch runs one persistent CTA per SM that takes (query tile,
 * head) units from a counter the plan owns; each call takes the next of the plan's 16
 * counters (and zeroes it first on `stream`), so at most 16 forward calls that share a
 * plan may be in flight on the GPU at once. */
lca_status lca_attn_fwd(const lca_plan* plan, const lca_shape* shape, const void* q,
                        const void* k, const void* v, void* o, float* lse, float softmax_scale,
                        void* stream);

/* ---- block maps from block scores (dynamic block-sparse masks)
 *
 * The benchmark builds a sparse mask by scoring every (query block, key block) pair
 * and keeping, for each query block, the k best key blocks, k following from the
 * sparsity ratio ("Long-Context Attention Benchmark", appendix A.2: Score Calculation,
 * Top-k Selection).  Its dynamic masks score blocks from the data, e.g. from
 * mean-pooled queries and keys (appendix A.3, "VSA").  lca_block_scores computes such
 * scores and lca_block_topk turns any score array into a block map that a
 * LCA_BLOCK_SPARSE_UNIFORM descriptor can pass to lca_mask_build (as a device array). */

/* Bytes of device workspace lca_block_scores needs: the pooled query and key blocks,
 * 2 * map_heads * ceil(seqlen / block) * 128 fp32 (0 for invalid arguments). */
size_t lca_block_scores_workspace(const lca_shape* shape, int block, int map_heads);

/* scores[h_m][r][c] = scale * < mean of Q over the rows of query block r (rows clipped
 * at seqlen) and the query heads of map head h_m,
 *                              mean of K over the rows of key block c and the KV heads
 * of those query heads >.
 * Preconditions: batch 1, head_dim 128, h_q % h_kv == 0, 1 <= block <= seqlen,
 * map_heads 1, h_kv or h_q (query heads h_m*h_q/map_heads .. +h_q/map_heads share a map
 * head), row strides multiples of 8 elements, q/k/scores/workspace 16-byte aligned
 * device pointers.  `scores` is a caller-owned device array of map_heads * n_b * n_b
 * fp32 (n_b = ceil(seqlen / block)); `workspace` holds at least
 * lca_block_scores_workspace() bytes.  softmax_scale <= 0 means 1/sqrt(128).
 * Asynchronous on `stream`; invalid arguments return before any launch. */
lca_status lca_block_scores(const lca_shape* shape, const void* q, const void* k, int block,
                            int map_heads, float softmax_scale, float* scores, void* workspace,
                            size_t ws_bytes, void* stream);

/* Top-k selection per row: block_map[h][r][c] = 1 for the k largest scores[h][r][.]
 * (descending score, ties by ascending c), 0 elsewhere.  scores: fp32 device array
 * [map_heads][n_rows][n_cols] without NaNs; block_map: uint8 device array of the same
 * shape (caller-owned).  Requires 1 <= k <= n_cols.  Asynchronous on `stream`. */
lca_status lca_block_topk(const float* scores, int map_heads, int n_rows, int n_cols, int k,
                          uint8_t* block_map, void* stream);

/* Bytes of device workspace lca_attn_bwd needs: two fp32 rows per (batch, query head),
 * LSE * log2(e) and D = rowsum(dO * O), each padded to seqlen rounded up to 128, i.e.
 * 8 * batch * h_q * round_up(seqlen, 128) bytes (0 for a NULL plan or shape). */
size_t lca_attn_bwd_workspace(const lca_plan* plan, const lca_shape* shape, int flags);

/* Backward: dQ, dK, dV (bf16) from Q, K, V, O, dO and the forward's LSE.
 * Same preconditions as lca_attn_fwd, plus the gradient-side row strides of `shape`
 * (dO read with do_row_stride; dQ, dK, dV written with dq/dk/dv_row_stride; each 0 or
 * >= its heads * head_dim and a multiple of 8, else LCA_ERR_INVALID_ARG).  Every row of
 * dQ, dK and dV below seqlen is written (zero where no pair reaches it); nothing else in
 * their buffers is touched.  `workspace` is a caller-owned device buffer of at least
 * lca_attn_bwd_workspace() bytes (16-byte aligned).  The result is deterministic (no
 * floating-point atomics).  flags: reserved, pass 0. */
lca_status lca_attn_bwd(const lca_plan* plan, const lca_shape* shape, const void* q,
                        const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, void* workspace,
                        size_t ws_bytes, float softmax_scale, int flags, void* stream);

/* Backward pass that allocates nothing, for callers that cannot allocate device memory
 * when they run the backward: code under a caching or pooled allocator that forbids
 * allocations outside its own pool, runtimes that hand an op only its own input and
 * output tensors, and programs that reserve all device memory up front.  The attention
 * method itself has no counterpart of this call: it only changes where the workspace
 * of lca_attn_bwd comes from.
 *
 * Same arguments, preconditions and results as lca_attn_bwd (flags 0), except that
 * the workspace is a fixed 64 MiB buffer compiled into the library (a file-scope
 * device array that every GPU loading the library holds until the process exits),
 * so it serves at most batch * h_q * round_up(seqlen, 128) <= 2^23 rows; larger
 * shapes return
 * LCA_ERR_UNSUPPORTED without launching anything.  No cudaMalloc / cudaFree is made
 * (with lca_profile_enable on, the timing events of the launches come from a pool
 * that grows on first use).
 * The first call on a device looks the buffer's device address up (with that device
 * current; again after the device's context was torn down and re-created, e.g. by
 * cudaDeviceReset).
 * Every call on a device shares the one buffer: each call overwrites every entry it
 * reads, so nothing needs clearing, but calls whose work overlaps on the GPU (other
 * streams, other threads) race on it and must be serialised by the caller. */
lca_status lca_attn_bwd_noalloc(const lca_plan* plan, const lca_shape* shape, const void* q,
                                const void* k, const void* v, const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv,
                                float softmax_scale, void* stream);

/* Synchronise `stream`, read and clear the device error word: LCA_OK, LCA_ERR_TIMEOUT
 * when a bounded device wait ran out since the last call, or LCA_ERR_CUDA when a kernel
 * refused to run (its shared memory came up without the alignment it needs). */
lca_status lca_get_last_device_error(void* stream);

/* Bound, in nanoseconds, of every device-side wait of later launches (default 2 s). */
void lca_set_wait_timeout_ns(uint64_t ns);

/* Self-check of the bounded-wait machinery: launches one CTA that waits on an mbarrier
 * nothing ever arrives on, with the given bound, and returns the resulting device
 * status (LCA_ERR_TIMEOUT when the bound works).  Synchronises `stream`. */
lca_status lca_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/* Self-check of the tensor-core operand layouts: one 128 x 128 x 128 bf16 GEMM with
 * fp32 accumulation on one CTA.  a, b: device bf16 [128][128] row-major; c: device
 * fp32 [128][128] row-major output.  variant 0: c = a b^T (both loaded K-major by TMA);
 * 1: c = a b (b loaded MN-major); 2: c = a b with a written to shared memory by the
 * threads in the 128-byte swizzle; 3: c = a^T b (a loaded MN-major); 4: c = a b with a
 * held in tensor memory (written by the threads with tcgen05.st).  Synchronises
 * `stream`; returns the device status. */
lca_status lca_selftest_umma(int variant, const void* a, const void* b, float* c, void* stream);

/* Per-kernel timing (tracing).  While enabled, every kernel launch of the library is
 * bracketed by two CUDA events recorded on the launch stream (no synchronisation is
 * added).  lca_profile_read synchronises the device, writes up to `max_entries`
 * records (one per kernel that launched since the last read: name, number of
 * launches, summed event time in milliseconds) and clears the records; it returns the
 * number of records written, or -1 on a CUDA error. */
typedef struct {
  char name[32];
  int64_t launches;
  double total_ms;
} lca_kernel_time;

void lca_profile_enable(int on);
int lca_profile_read(lca_kernel_time* out, int max_entries);

const char* lca_status_string(lca_status s);

#ifdef __cplusplus
}
#endif
#endif /* LCA_H_ */
