"""Mask predicates: allowed(i, j) for every mask type, written pair by pair.

The benchmark sorts its 14 mask patterns into 12 static masks (regular and
heterogeneous) and 2 dynamic block-sparse masks [LongCA-bench summary, §2.1.1
"Input Mask Patterns"; reading note, "Key design" 1: FULL, CAUSAL, sliding
window, document variants; shared question, global sliding, causal blockwise,
prefix LM, block causal document; uniform and variable block-sparse].  The
pages give names only.  The readings taken here (0-indexed positions, query i,
key j, sequence length S):

* FULL: every pair.
* CAUSAL: j <= i.
* SLIDING_WINDOW(w): j <= i and i - j < w (w keys including the query's own
  position; causal).  Any w >= S reduces to CAUSAL.
* FULL_DOCUMENT / CAUSAL_DOCUMENT: doc(i) == doc(j) [and j <= i], documents
  given by cu_seqlens [§A.4.1 "FULL/CAUSAL DOCUMENT": variable-length
  sequences packed together].
* SLIDING_WINDOW_DOCUMENT(w): the sliding window inside the query's document,
  doc(i) == doc(j) and j <= i and i - j < w.  The pages count six regular masks
  and name FULL, CAUSAL, sliding window and the document variants; this is the
  plainest sixth (the window's document variant).  Any w >= S reduces to
  CAUSAL_DOCUMENT, one document to SLIDING_WINDOW.
* PREFIX_LM(P): j < P or j <= i (bidirectional over the prefix, causal after).
* SHARED_QUESTION: segment 0 is the question, later segments are answers;
  j <= i and (seg(j) == seg(i) or seg(j) == 0): answers see the question and
  themselves causally, never each other; the question is causal in itself.
* GLOBAL_SLIDING(G, w): global tokens plus a window [§A.4.1 "GLOBAL
  SLIDING"].  Causal reading (base_causal = 1): j <= i and (j < G or i - j <
  w).  Symmetric reading (base_causal = 0): j < G or i < G or |i - j| < w.
* CAUSAL_BLOCKWISE(Bk): j // Bk <= i // Bk (full within a block, causal
  across blocks).
* BLOCK_CAUSAL_DOCUMENT(Bk): doc(i) == doc(j) and (j - st) // Bk <= (i - st)
  // Bk with st the document's start [§A.4.1 "BLOCK CAUSAL DOCUMENT": the
  document mask raised to block level].
* BLOCK_SPARSE_UNIFORM(b, map): map[h][i // b][j // b] [§A.2 "Block
  Partitioning": equal block sizes].
* BLOCK_SPARSE_VARIABLE(offsets, map): map[h][rb(i)][cb(j)] with rb/cb the
  blocks of the head's own row/column partitions [§A.2: grid dimensions follow
  the lengths of the query- and key-block lists].
* Both block-sparse masks are further ANDed with j <= i when base_causal is
  set and with doc(i) == doc(j) when cu_seqlens is given.

Maps are per map head: one map (map_heads = 1), one per KV head (GQA shares a
mask within a KV group [§A.2 "Score Calculation"]) or one per query head.
"""
from __future__ import annotations

import numpy as np

from long_context_masked_gb300 import inputs as _in


def map_head_of(h_q: int, h_q_total: int, h_kv_total: int, map_heads: int) -> int:
    """Map head used by query head ``h_q`` (GQA: the KV head's map)."""
    if map_heads == 1:
        return 0
    if map_heads == h_kv_total:
        return h_q // (h_q_total // h_kv_total)
    if map_heads == h_q_total:
        return h_q
    raise ValueError("map_heads must be 1, H_kv or H_q")


def _segment_of(cu: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Index of the segment [cu[s], cu[s+1]) holding position x."""
    return np.searchsorted(np.asarray(cu, np.int64), x, side="right") - 1


def allowed(desc, h_m: int, i: np.ndarray, j: np.ndarray) -> np.ndarray:
    """Boolean array, True where query i may attend to key j.

    ``i`` and ``j`` are integer arrays that broadcast against each other
    (typically a column of query positions and a row of key positions).
    """
    i = np.asarray(i, np.int64)
    j = np.asarray(j, np.int64)
    t = desc.type
    if t == _in.FULL:
        return np.ones(np.broadcast_shapes(i.shape, j.shape), bool)
    if t == _in.CAUSAL:
        return j <= i
    if t == _in.SLIDING_WINDOW:
        return (j <= i) & (i - j < desc.window)
    if t == _in.FULL_DOCUMENT:
        return _segment_of(desc.cu_seqlens, i) == _segment_of(desc.cu_seqlens, j)
    if t == _in.CAUSAL_DOCUMENT:
        return (_segment_of(desc.cu_seqlens, i) == _segment_of(desc.cu_seqlens, j)) & (j <= i)
    if t == _in.SLIDING_WINDOW_DOCUMENT:
        same = _segment_of(desc.cu_seqlens, i) == _segment_of(desc.cu_seqlens, j)
        return same & (j <= i) & (i - j < desc.window)
    if t == _in.PREFIX_LM:
        return (j < desc.prefix_len) | (j <= i)
    if t == _in.SHARED_QUESTION:
        si = _segment_of(desc.cu_seqlens, i)
        sj = _segment_of(desc.cu_seqlens, j)
        return (j <= i) & ((sj == si) | (sj == 0))
    if t == _in.GLOBAL_SLIDING:
        g, w = desc.num_global, desc.window
        if desc.base_causal:
            return (j <= i) & ((j < g) | (i - j < w))
        return (j < g) | (i < g) | (np.abs(i - j) < w)
    if t == _in.CAUSAL_BLOCKWISE:
        return (j // desc.block) <= (i // desc.block)
    if t == _in.BLOCK_CAUSAL_DOCUMENT:
        cu = np.asarray(desc.cu_seqlens, np.int64)
        di = _segment_of(cu, i)
        dj = _segment_of(cu, j)
        return (di == dj) & ((j - cu[dj]) // desc.block <= (i - cu[di]) // desc.block)
    if t in (_in.BLOCK_SPARSE_UNIFORM, _in.BLOCK_SPARSE_VARIABLE):
        bmap = np.asarray(desc.block_map)[h_m]
        if t == _in.BLOCK_SPARSE_UNIFORM:
            rb = i // desc.block
            cb = j // desc.block
        else:
            rb = _segment_of(np.asarray(desc.row_offsets)[h_m], i)
            cb = _segment_of(np.asarray(desc.col_offsets)[h_m], j)
        ok = bmap[rb, cb] != 0
        if desc.base_causal:
            ok = ok & (j <= i)
        if desc.cu_seqlens is not None:
            ok = ok & (_segment_of(desc.cu_seqlens, i) == _segment_of(desc.cu_seqlens, j))
        return ok
    raise ValueError(f"unknown mask type {t}")


def mask_rows(desc, h_m: int, rows) -> np.ndarray:
    """Rows of the S x S mask: bool [len(rows), S]."""
    rows = np.asarray(rows, np.int64)
    cols = np.arange(desc.seqlen, dtype=np.int64)
    return np.broadcast_to(allowed(desc, h_m, rows[:, None], cols[None, :]),
                           (len(rows), desc.seqlen))


def materialize_mask(desc, h_m: int = 0) -> np.ndarray:
    """The whole S x S mask of map head ``h_m`` (bool)."""
    return mask_rows(desc, h_m, np.arange(desc.seqlen))
