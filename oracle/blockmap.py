"""Block-sparse maps from block scores: mean-pooled Q/K scores and top-k selection.

The benchmark builds its sparse masks in three steps (LongCA-bench summary page,
appendix A.2 "Details of Sparse Data Sampling"):

* Block Partitioning: the attention map is cut into query-block and key-block grids;
* Score Calculation: every (query block, key block) pair gets an importance score,
  per head under MHA and shared by the query heads of a KV group under GQA (the
  benchmark itself draws random scores);
* Top-k Selection: each query block keeps its k best key blocks, k following from
  the sparsity ratio.

The dynamic masks the benchmark covers score blocks from the data: VSA's coarse stage
mean-pools the tokens of each block and scores pooled queries against pooled keys
(appendix A.3 "VSA").

Readings taken here where the pages are silent:

* k = round((1 - sparsity) * n_col_blocks), clipped to [1, n_col_blocks];
* top-k orders a row by descending score and breaks ties by ascending key-block
  index, so the selection is unique;
* the pooled score of map head h_m, query block r and key block c is
  ``scale * <mean Q over block r's rows and h_m's query heads,
               mean K over block c's rows and the KV heads of those query heads>``,
  with rows clipped at S (the last block may be short) and scale = 1/sqrt(d).
"""
from __future__ import annotations

import math

import numpy as np

from .masks import map_head_of


def topk_count(n_col_blocks: int, sparsity: float) -> int:
    """k of a top-k map: the number of key blocks each query block keeps."""
    k = int(round((1.0 - sparsity) * n_col_blocks))
    return min(max(k, 1), n_col_blocks)


def topk_block_map(scores: np.ndarray, k: int) -> np.ndarray:
    """uint8 map [H_m, n_rb, n_cb]: 1 on the k highest-scoring key blocks of each row
    (descending score, ties by ascending index)."""
    scores = np.asarray(scores)
    h_m, n_rb, n_cb = scores.shape
    out = np.zeros((h_m, n_rb, n_cb), np.uint8)
    idx = np.arange(n_cb)
    for h in range(h_m):
        for r in range(n_rb):
            order = np.lexsort((idx, -scores[h, r].astype(np.float64)))
            out[h, r, order[:k]] = 1
    return out


def _heads_of_map_head(h_m: int, map_heads: int, h_q: int, h_kv: int):
    """Query heads using map head h_m and the KV heads they read."""
    qh = [h for h in range(h_q) if map_head_of(h, h_q, h_kv, map_heads) == h_m]
    group = h_q // h_kv
    kvh = sorted({h // group for h in qh})
    return qh, kvh


def pooled_block_scores(q: np.ndarray, k: np.ndarray, block: int, map_heads: int,
                        scale: float | None = None) -> np.ndarray:
    """fp64 scores [H_m, n_rb, n_cb] from mean-pooled query and key blocks.

    ``q`` is [1, S, H_q, d] and ``k`` is [1, S, H_kv, d] (any float dtype; the
    values are taken exactly in fp64).
    """
    q = np.asarray(q, np.float64)[0]
    k = np.asarray(k, np.float64)[0]
    s_len, h_q, d = q.shape
    h_kv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nb = (s_len + block - 1) // block
    out = np.zeros((map_heads, nb, nb))
    for h_m in range(map_heads):
        qh, kvh = _heads_of_map_head(h_m, map_heads, h_q, h_kv)
        qp = np.zeros((nb, d))
        kp = np.zeros((nb, d))
        for b in range(nb):
            r0, r1 = b * block, min(s_len, (b + 1) * block)
            qp[b] = q[r0:r1][:, qh].reshape(-1, d).mean(axis=0)
            kp[b] = k[r0:r1][:, kvh].reshape(-1, d).mean(axis=0)
        out[h_m] = scale * (qp @ kp.T)
    return out
