"""Valid-pair counts: by popcount of the materialised mask and by closed forms.

The benchmark reports throughput in FLOPs/s per mask and sequence length
[LongCA-bench summary, §A.4 "Reported metrics", §A.4.1]; the FLOPs credited are
those of the allowed (unmasked) pairs only, so the exact number of allowed
pairs per head is part of the measurement.  ``n_valid_popcount`` counts the
materialised mask; ``n_valid_closed_form`` sums the per-row key counts that
follow from each mask's definition, an independent derivation used to pin the
mask materialisation.
"""
from __future__ import annotations

import numpy as np

from long_context_masked_gb300 import inputs as _in
from .masks import mask_rows


def n_valid_popcount(desc, h_m: int = 0, chunk: int = 1024) -> int:
    s_len = desc.seqlen
    total = 0
    for r0 in range(0, s_len, chunk):
        total += int(np.count_nonzero(mask_rows(desc, h_m, np.arange(r0, min(s_len, r0 + chunk)))))
    return total


def _blockwise_count(length: int, block: int) -> int:
    """Pairs of a block-causal mask over one span of ``length`` tokens."""
    tot = 0
    for b0 in range(0, length, block):
        rows = min(block, length - b0)
        tot += rows * min(b0 + block, length)
    return tot


def n_valid_closed_form(desc, h_m: int = 0) -> int:
    """Number of allowed pairs of map head ``h_m`` from per-row key counts."""
    s = desc.seqlen
    t = desc.type
    if t == _in.FULL:
        return s * s
    if t == _in.CAUSAL:
        return s * (s + 1) // 2
    if t == _in.SLIDING_WINDOW:
        w = desc.window
        if w >= s:
            return s * (s + 1) // 2
        return w * (w + 1) // 2 + (s - w) * w
    lengths = None if desc.cu_seqlens is None else np.diff(np.asarray(desc.cu_seqlens, np.int64))
    if t == _in.FULL_DOCUMENT:
        return int((lengths * lengths).sum())
    if t == _in.CAUSAL_DOCUMENT:
        return int((lengths * (lengths + 1) // 2).sum())
    if t == _in.SLIDING_WINDOW_DOCUMENT:
        w = desc.window
        tot = 0
        for n in lengths.tolist():   # a window of w keys inside every document
            tot += n * (n + 1) // 2 if n <= w else w * (w + 1) // 2 + (n - w) * w
        return tot
    if t == _in.PREFIX_LM:
        p = desc.prefix_len
        return p * p + (s * (s + 1) - p * (p + 1)) // 2
    if t == _in.SHARED_QUESTION:
        q = int(lengths[0])
        tot = q * (q + 1) // 2
        for a in lengths[1:]:
            a = int(a)
            tot += a * q + a * (a + 1) // 2
        return tot
    if t == _in.GLOBAL_SLIDING and desc.base_causal:
        g, w = desc.num_global, desc.window
        i = np.arange(s, dtype=np.int64)
        return int((np.minimum(i + 1, w) + np.maximum(0, np.minimum(g, i - w + 1))).sum())
    if t == _in.CAUSAL_BLOCKWISE:
        return _blockwise_count(s, desc.block)
    if t == _in.BLOCK_CAUSAL_DOCUMENT:
        return sum(_blockwise_count(int(L), desc.block) for L in lengths)
    if t == _in.BLOCK_SPARSE_UNIFORM and not desc.base_causal and desc.cu_seqlens is None:
        b = desc.block
        nb = (s + b - 1) // b
        size = np.minimum(b, s - np.arange(nb) * b).astype(np.int64)
        return int((np.asarray(desc.block_map[h_m], np.int64) * size[:, None] * size[None, :]).sum())
    raise ValueError("no closed form for this mask; use n_valid_popcount")
