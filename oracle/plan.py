"""Tile plan by brute force over the materialised mask.

The benchmark converts each mask into a unified representation from which
kernel-specific inputs are derived, and its context-parallel framework
precomputes the metadata it needs once [LongCA-bench summary, §2.2 "Attention
Kernel"; reading note, "Key design" 2 and 3].  The representation defined here
is the one the CUDA library consumes:

* the S x S mask is cut into tiles of ``tile_q`` query rows by ``tile_k`` key
  columns; tiles on the last row/column are clipped at S;
* a tile is SKIP (0) when no in-range pair is allowed, FULL (1) when every
  in-range pair is allowed, PARTIAL (2) otherwise;
* the tile byte of a non-skipped tile adds flags for its empty halves (no
  allowed in-range pair): 4 = key columns [0, tile_k/2), 8 = key columns
  [tile_k/2, tile_k), 16 = query rows [0, tile_q/2), 32 = query rows
  [tile_q/2, tile_q).  The benchmark's sparse masks are built on a block grid
  finer than a tile (64-token blocks against 128-token tiles), so a tile can
  hold allowed pairs in one half only and a kernel can leave the other half out;
* per (map head, query tile) row: the non-skipped key tiles in ascending order
  with their class and key-half flags (tile byte & 15; CSR: ``rowptr``,
  ``kt_idx``, ``kt_cls``);
* per (map head, key tile) column: the non-skipped query tiles in ascending
  order with their class and query-half flags moved to bits 2-3 (``colptr``,
  ``qt_idx``, ``qt_cls``);
* work orders: row indices (h_m * nQt + qt) sorted by descending list length,
  ties by ascending index (``work_q``), and likewise for columns
  (``work_k``), i.e. longest-processing-time-first.
"""
from __future__ import annotations

from typing import Dict, Sequence

import numpy as np

from .masks import mask_rows


def tile_rows_ref(desc, tile_q: int, tile_k: int, h_m: int, qts: Sequence[int]) -> np.ndarray:
    """Tile bytes of the given query tiles of map head ``h_m``: uint8 [len(qts), nKt]."""
    assert tile_q % 2 == 0 and tile_k % 2 == 0, "tiles have two halves"
    s_len = desc.seqlen
    n_kt = (s_len + tile_k - 1) // tile_k
    out = np.zeros((len(qts), n_kt), np.uint8)
    pad = n_kt * tile_k - s_len
    for a, qt in enumerate(qts):
        rows = np.arange(qt * tile_q, min(s_len, (qt + 1) * tile_q))
        m = mask_rows(desc, h_m, rows)
        any_m = np.concatenate([m, np.zeros((len(rows), pad), bool)], axis=1)
        all_m = np.concatenate([m, np.ones((len(rows), pad), bool)], axis=1)
        any_t = any_m.reshape(len(rows), n_kt, tile_k).any(axis=(0, 2))
        all_t = all_m.reshape(len(rows), n_kt, tile_k).all(axis=(0, 2))
        cls = np.where(all_t, 1, 2)
        # halves with an allowed pair: key columns of the tile, then query rows
        key_h = any_m.reshape(len(rows), n_kt, 2, tile_k // 2).any(axis=(0, 3))
        top = any_m[:tile_q // 2].reshape(-1, n_kt, tile_k).any(axis=(0, 2))
        bottom = any_m[tile_q // 2:].reshape(-1, n_kt, tile_k).any(axis=(0, 2))
        flags = (4 * ~key_h[:, 0] + 8 * ~key_h[:, 1] + 16 * ~top + 32 * ~bottom)
        out[a] = np.where(any_t, cls + flags, 0).astype(np.uint8)
    return out


def row_list_byte(tile_byte: np.ndarray) -> np.ndarray:
    """Entry of a row list: the class and the key-half flags."""
    return (tile_byte & 15).astype(np.uint8)


def col_list_byte(tile_byte: np.ndarray) -> np.ndarray:
    """Entry of a column list: the class and the query-half flags in bits 2-3."""
    return ((tile_byte & 3) | ((tile_byte >> 2) & 12)).astype(np.uint8)


def _lpt_order(lengths: np.ndarray) -> np.ndarray:
    idx = np.arange(len(lengths))
    return np.lexsort((idx, -lengths.astype(np.int64))).astype(np.int32)


def tile_plan_ref(desc, tile_q: int, tile_k: int) -> Dict[str, np.ndarray]:
    """The whole plan: classes, both CSR lists and both work orders."""
    s_len = desc.seqlen
    n_qt = (s_len + tile_q - 1) // tile_q
    n_kt = (s_len + tile_k - 1) // tile_k
    hm_n = desc.map_heads
    cls = np.zeros((hm_n, n_qt, n_kt), np.uint8)
    for hm in range(hm_n):
        cls[hm] = tile_rows_ref(desc, tile_q, tile_k, hm, range(n_qt))

    rows = cls.reshape(hm_n * n_qt, n_kt)
    row_len = np.count_nonzero(rows, axis=1)
    rowptr = np.zeros(hm_n * n_qt + 1, np.int32)
    rowptr[1:] = np.cumsum(row_len)
    kt_idx = np.concatenate([np.nonzero(r)[0] for r in rows]).astype(np.int32) \
        if rows.size else np.zeros(0, np.int32)
    kt_cls = row_list_byte(rows[rows != 0])

    cols = np.transpose(cls, (0, 2, 1)).reshape(hm_n * n_kt, n_qt)
    col_len = np.count_nonzero(cols, axis=1)
    colptr = np.zeros(hm_n * n_kt + 1, np.int32)
    colptr[1:] = np.cumsum(col_len)
    qt_idx = np.concatenate([np.nonzero(c)[0] for c in cols]).astype(np.int32) \
        if cols.size else np.zeros(0, np.int32)
    qt_cls = col_list_byte(cols[cols != 0])

    return {
        "cls": cls, "rowptr": rowptr, "kt_idx": kt_idx, "kt_cls": kt_cls,
        "colptr": colptr, "qt_idx": qt_idx, "qt_cls": qt_cls,
        "work_q": _lpt_order(row_len), "work_k": _lpt_order(col_len),
    }
