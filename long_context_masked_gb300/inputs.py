"""Seeded synthetic inputs shared by the CUDA path, its tests and the bench.

This module only draws data: document lengths, block partitions, block maps and
the Q/K/V/dO tensors, plus the plain mask-descriptor container.  It holds none of
the attention arithmetic and no mask evaluation, so both sides (the oracle and
the CUDA library) can take their inputs from it without sharing any of the
method's code.

Workload recipes follow the benchmark described in "Long-Context Attention
Benchmark: From Kernel Efficiency to Distributed Context Parallelism"
(LongCA-bench):

* dense masks over variable-length documents packed to one sequence
  (section 2.1.2, "Input Data Sampling"; appendix A.1).  The corpora the paper
  samples from are not available, so document lengths are drawn from a
  lognormal model (mu = ln 2048, sigma = 1, clipped to [128, S]) instead;
* block-sparse maps built by partitioning the attention map into query/key
  block grids (appendix A.2, "Block Partitioning") with random keep decisions
  at sparsities 0.2/0.5/0.8 (section 2.1.2; appendix A.2, "Top-k Selection");
* Q/K/V/dO drawn as N(0, 1) in fp32 and rounded to bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

# Mask type codes (same values as lca_mask_type in include/lca.h).
FULL = 0
CAUSAL = 1
SLIDING_WINDOW = 2
FULL_DOCUMENT = 3
CAUSAL_DOCUMENT = 4
PREFIX_LM = 5
SHARED_QUESTION = 6
GLOBAL_SLIDING = 7
CAUSAL_BLOCKWISE = 8
BLOCK_CAUSAL_DOCUMENT = 9
BLOCK_SPARSE_UNIFORM = 10
BLOCK_SPARSE_VARIABLE = 11
SLIDING_WINDOW_DOCUMENT = 12

MASK_NAMES = {
    FULL: "FULL",
    CAUSAL: "CAUSAL",
    SLIDING_WINDOW: "SLIDING_WINDOW",
    FULL_DOCUMENT: "FULL_DOCUMENT",
    CAUSAL_DOCUMENT: "CAUSAL_DOCUMENT",
    PREFIX_LM: "PREFIX_LM",
    SHARED_QUESTION: "SHARED_QUESTION",
    GLOBAL_SLIDING: "GLOBAL_SLIDING",
    CAUSAL_BLOCKWISE: "CAUSAL_BLOCKWISE",
    BLOCK_CAUSAL_DOCUMENT: "BLOCK_CAUSAL_DOCUMENT",
    BLOCK_SPARSE_UNIFORM: "BLOCK_SPARSE_UNIFORM",
    BLOCK_SPARSE_VARIABLE: "BLOCK_SPARSE_VARIABLE",
    SLIDING_WINDOW_DOCUMENT: "SLIDING_WINDOW_DOCUMENT",
}

# Tile classes written by the mask builder (lca_tile_class), and the empty-half flags of a
# non-skipped tile's byte (a half without any allowed in-range pair).  Row-list entries
# (kt_cls) carry the class and the key-half flags; column-list entries (qt_cls) carry the
# class and the query-half flags moved down to 4 / 8.
TILE_SKIP = 0
TILE_FULL = 1
TILE_PARTIAL = 2
TILE_CLASS_MASK = 3
TILE_KEY_HALF0_EMPTY = 4
TILE_KEY_HALF1_EMPTY = 8
TILE_QUERY_HALF0_EMPTY = 16
TILE_QUERY_HALF1_EMPTY = 32


@dataclasses.dataclass
class MaskDesc:
    """Plain container mirroring ``lca_mask_desc``; arrays live on the host.

    Fields not used by a mask type keep their defaults.  ``cu_seqlens`` holds
    ``num_segments + 1`` ascending offsets starting at 0 and ending at
    ``seqlen``.  For the variable block-sparse map, ``row_offsets`` and
    ``col_offsets`` are ``[map_heads, n_blocks + 1]`` arrays (each head's
    partition padded at its end by repeating ``seqlen``).
    """

    type: int
    seqlen: int
    window: int = 0
    num_global: int = 0
    prefix_len: int = 0
    block: int = 0
    base_causal: int = 0
    cu_seqlens: Optional[np.ndarray] = None
    map_heads: int = 1
    n_row_blocks: int = 0
    n_col_blocks: int = 0
    row_offsets: Optional[np.ndarray] = None
    col_offsets: Optional[np.ndarray] = None
    block_map: Optional[np.ndarray] = None

    @property
    def name(self) -> str:
        return MASK_NAMES[self.type]

    @property
    def num_segments(self) -> int:
        return 0 if self.cu_seqlens is None else len(self.cu_seqlens) - 1


# ---------------------------------------------------------------- documents

def lognormal_doc_lengths(seqlen: int, seed: int, mu: float = math.log(2048.0),
                          sigma: float = 1.0, lo: int = 128) -> List[int]:
    """Document lengths packed to exactly ``seqlen`` tokens.

    Lengths are floor(lognormal(mu, sigma)) clipped to [lo, seqlen], drawn in
    order until their sum reaches ``seqlen``; the last document is cut to the
    remainder (so it may be shorter than ``lo``).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths: List[int] = []
    total = 0
    while total < seqlen:
        x = int(math.floor(rng.lognormal(mu, sigma)))
        x = min(max(x, lo), seqlen)
        x = min(x, seqlen - total)
        lengths.append(x)
        total += x
    return lengths


def cu_from_lengths(lengths: Sequence[int]) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def shared_question_cu(question: int, answers: Sequence[int]) -> np.ndarray:
    """Segment offsets for a shared question (segment 0) followed by answers."""
    return cu_from_lengths([question] + list(answers))


# ------------------------------------------------------------ block maps

def uniform_block_map(seqlen: int, block: int, map_heads: int, sparsity: float,
                      seed: int) -> np.ndarray:
    """Uniform block grid with Bernoulli keep decisions.

    Each block is kept when u < 1 - sparsity (u uniform in [0, 1), drawn in
    head-major, row-major order); diagonal blocks are then forced kept.
    """
    nb = (seqlen + block - 1) // block
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.random((map_heads, nb, nb))
    m = (u < (1.0 - sparsity)).astype(np.uint8)
    idx = np.arange(nb)
    m[:, idx, idx] = 1
    return m


VARIABLE_BLOCK_SIZES = tuple(range(32, 257, 16))  # 32, 48, ..., 256


def variable_partition(seqlen: int, rng: np.random.Generator) -> np.ndarray:
    """Offsets of one variable block partition of [0, seqlen)."""
    sizes: List[int] = []
    total = 0
    choices = np.asarray(VARIABLE_BLOCK_SIZES)
    while total < seqlen:
        x = int(choices[rng.integers(0, len(choices))])
        x = min(x, seqlen - total)
        sizes.append(x)
        total += x
    return cu_from_lengths(sizes)


def variable_block_map(seqlen: int, map_heads: int, seed: int, keep: float = 0.5):
    """Per-head variable row/column partitions and a map over them.

    Returns ``(row_offsets, col_offsets, block_map)``.  A block is a "causal
    block" when its first column is not after its last row
    (col_start <= row_end - 1).  One uniform u is drawn per block in row-major
    order; causal blocks are kept when u < keep, other blocks are 0.  Blocks
    that contain a diagonal element are forced kept.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    rows, cols = [], []
    for _ in range(map_heads):
        rows.append(variable_partition(seqlen, rng))
        cols.append(variable_partition(seqlen, rng))
    n_rb = max(len(r) - 1 for r in rows)
    n_cb = max(len(c) - 1 for c in cols)
    row_off = np.full((map_heads, n_rb + 1), seqlen, dtype=np.int32)
    col_off = np.full((map_heads, n_cb + 1), seqlen, dtype=np.int32)
    bmap = np.zeros((map_heads, n_rb, n_cb), dtype=np.uint8)
    for h in range(map_heads):
        r, c = rows[h], cols[h]
        row_off[h, :len(r)] = r
        col_off[h, :len(c)] = c
        nr, nc = len(r) - 1, len(c) - 1
        u = rng.random((nr, nc))
        r_start = r[:-1][:, None].astype(np.int64)
        r_end = r[1:][:, None].astype(np.int64)
        c_start = c[:-1][None, :].astype(np.int64)
        c_end = c[1:][None, :].astype(np.int64)
        causal_block = c_start <= r_end - 1
        kept = causal_block & (u < keep)
        has_diag = (r_start < c_end) & (c_start < r_end)
        bmap[h, :nr, :nc] = (kept | has_diag).astype(np.uint8)
    return row_off, col_off, bmap


def random_block_scores(map_heads: int, n_row_blocks: int, n_col_blocks: int,
                        seed: int) -> np.ndarray:
    """Random block importance scores, fp32 uniform in [0, 1), [H_m, n_rb, n_cb].

    The benchmark scores blocks randomly so that only the block-sparse attention
    itself is measured (appendix A.2, "Score Calculation"); a top-k selection over
    these scores gives its top-k maps.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.random((map_heads, n_row_blocks, n_col_blocks), dtype=np.float32)


# ------------------------------------------------------------ descriptors

def make_desc(mask_type: int, seqlen: int, *, window: int = 4096, num_global: int = 256,
              prefix_len: Optional[int] = None, block: int = 2048, doc_seed: int = 0,
              question: int = 2048, answers: Optional[Sequence[int]] = None,
              cu_seqlens: Optional[np.ndarray] = None, base_causal: Optional[int] = None,
              sparse_block: int = 128, sparsity: float = 0.5, map_heads: int = 1,
              map_seed: int = 0, variable_keep: float = 0.5) -> MaskDesc:
    """Descriptor for one mask of the benchmark's workload recipes."""
    t = mask_type
    if t in (FULL, CAUSAL):
        return MaskDesc(t, seqlen)
    if t == SLIDING_WINDOW:
        return MaskDesc(t, seqlen, window=window)
    if t in (FULL_DOCUMENT, CAUSAL_DOCUMENT):
        if cu_seqlens is None:
            cu_seqlens = cu_from_lengths(lognormal_doc_lengths(seqlen, doc_seed))
        return MaskDesc(t, seqlen, cu_seqlens=np.asarray(cu_seqlens, np.int32))
    if t == SLIDING_WINDOW_DOCUMENT:
        if cu_seqlens is None:
            cu_seqlens = cu_from_lengths(lognormal_doc_lengths(seqlen, doc_seed))
        return MaskDesc(t, seqlen, window=window, cu_seqlens=np.asarray(cu_seqlens, np.int32))
    if t == PREFIX_LM:
        return MaskDesc(t, seqlen, prefix_len=seqlen // 4 if prefix_len is None else prefix_len)
    if t == SHARED_QUESTION:
        if cu_seqlens is None:
            if answers is None:
                n = 4
                a = (seqlen - question) // n
                answers = [a] * (n - 1) + [seqlen - question - a * (n - 1)]
            cu_seqlens = shared_question_cu(question, answers)
        return MaskDesc(t, seqlen, cu_seqlens=np.asarray(cu_seqlens, np.int32))
    if t == GLOBAL_SLIDING:
        return MaskDesc(t, seqlen, window=window, num_global=num_global,
                        base_causal=1 if base_causal is None else base_causal)
    if t == CAUSAL_BLOCKWISE:
        return MaskDesc(t, seqlen, block=block)
    if t == BLOCK_CAUSAL_DOCUMENT:
        if cu_seqlens is None:
            cu_seqlens = cu_from_lengths(lognormal_doc_lengths(seqlen, doc_seed))
        return MaskDesc(t, seqlen, block=block, cu_seqlens=np.asarray(cu_seqlens, np.int32))
    if t == BLOCK_SPARSE_UNIFORM:
        bmap = uniform_block_map(seqlen, sparse_block, map_heads, sparsity, map_seed)
        return MaskDesc(t, seqlen, block=sparse_block,
                        base_causal=0 if base_causal is None else base_causal,
                        cu_seqlens=None if cu_seqlens is None else np.asarray(cu_seqlens, np.int32),
                        map_heads=map_heads, n_row_blocks=bmap.shape[1],
                        n_col_blocks=bmap.shape[2], block_map=bmap)
    if t == BLOCK_SPARSE_VARIABLE:
        if cu_seqlens is None:
            cu_seqlens = cu_from_lengths(lognormal_doc_lengths(seqlen, doc_seed))
        ro, co, bmap = variable_block_map(seqlen, map_heads, map_seed, variable_keep)
        return MaskDesc(t, seqlen, base_causal=1 if base_causal is None else base_causal,
                        cu_seqlens=np.asarray(cu_seqlens, np.int32), map_heads=map_heads,
                        n_row_blocks=bmap.shape[1], n_col_blocks=bmap.shape[2],
                        row_offsets=ro, col_offsets=co, block_map=bmap)
    raise ValueError(f"unknown mask type {mask_type}")


# ------------------------------------------------------------ tensors

def qkv_do(batch: int, seqlen: int, h_q: int, h_kv: int, head_dim: int, seed: int):
    """Q, K, V, dO as bf16 CPU tensors drawn N(0, 1) in fp32 from ``seed``.

    Layouts: Q and dO ``[B, S, H_q, d]``; K and V ``[B, S, H_kv, d]``.
    """
    import torch

    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((batch, seqlen, h_q, head_dim), generator=g, dtype=torch.float32)
    k = torch.randn((batch, seqlen, h_kv, head_dim), generator=g, dtype=torch.float32)
    v = torch.randn((batch, seqlen, h_kv, head_dim), generator=g, dtype=torch.float32)
    do = torch.randn((batch, seqlen, h_q, head_dim), generator=g, dtype=torch.float32)
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
            do.to(torch.bfloat16))
