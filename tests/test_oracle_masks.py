"""Pins for the oracle's mask definitions and the workload generators (CPU)."""
import numpy as np
import pytest

import oracle
from long_context_masked_gb300 import inputs as I
from tests._golden import load_mask_cases

CASES = load_mask_cases()


@pytest.mark.parametrize("name,desc,expected", CASES, ids=[c[0] for c in CASES])
def test_golden_hand_drawn_masks(name, desc, expected):
    got = oracle.materialize_mask(desc, 0)
    assert got.shape == expected.shape
    assert np.array_equal(got, expected), f"{name}\n{got.astype(int)}"


def _structured_descs(s, seed):
    rng = np.random.default_rng(seed)
    lens = I.lognormal_doc_lengths(s, seed, mu=np.log(max(8, s // 6)), sigma=1.0, lo=3)
    cu = I.cu_from_lengths(lens)
    w = int(rng.integers(1, s + 3))
    out = [
        I.MaskDesc(I.FULL, s),
        I.MaskDesc(I.CAUSAL, s),
        I.MaskDesc(I.SLIDING_WINDOW, s, window=w),
        I.MaskDesc(I.FULL_DOCUMENT, s, cu_seqlens=cu),
        I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=cu),
        I.MaskDesc(I.PREFIX_LM, s, prefix_len=int(rng.integers(0, s + 1))),
        I.MaskDesc(I.GLOBAL_SLIDING, s, num_global=int(rng.integers(0, s // 2 + 1)),
                   window=int(rng.integers(1, s + 1)), base_causal=1),
        I.MaskDesc(I.CAUSAL_BLOCKWISE, s, block=int(rng.integers(1, s + 2))),
        I.MaskDesc(I.BLOCK_CAUSAL_DOCUMENT, s, block=int(rng.integers(1, 40)), cu_seqlens=cu),
        I.MaskDesc(I.SLIDING_WINDOW_DOCUMENT, s, window=max(1, w // 2), cu_seqlens=cu),
    ]
    q = int(rng.integers(1, s // 3 + 2))
    rest = s - q
    n_ans = int(rng.integers(1, 5))
    cuts = np.sort(rng.choice(np.arange(1, rest), size=min(n_ans - 1, rest - 1), replace=False)) \
        if rest > 1 else np.array([], int)
    answers = np.diff(np.concatenate([[0], cuts, [rest]])).tolist()
    out.append(I.MaskDesc(I.SHARED_QUESTION, s, cu_seqlens=I.shared_question_cu(q, answers)))
    b = int(rng.integers(1, 17))
    bm = I.uniform_block_map(s, b, 2, float(rng.random()), seed)
    out.append(I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=b, map_heads=2,
                          n_row_blocks=bm.shape[1], n_col_blocks=bm.shape[2], block_map=bm))
    return out


@pytest.mark.parametrize("s,seed", [(1, 0), (7, 1), (64, 2), (97, 3), (200, 4), (333, 5)])
def test_closed_form_counts_match_popcount(s, seed):
    for d in _structured_descs(s, seed):
        for hm in range(d.map_heads):
            assert oracle.n_valid_popcount(d, hm, chunk=37) == oracle.n_valid_closed_form(d, hm), d.name


def test_closed_form_counts_at_benchmark_sizes():
    # Values worked out from the per-row key counts of each mask.
    s = 8192
    assert oracle.n_valid_closed_form(I.MaskDesc(I.SLIDING_WINDOW, s, window=4096)) == 25_167_872
    assert oracle.n_valid_closed_form(I.MaskDesc(I.CAUSAL, 1024)) == 524_800
    assert oracle.n_valid_closed_form(I.MaskDesc(I.FULL, 1024)) == 1_048_576
    s = 32768
    p = 8192
    assert oracle.n_valid_closed_form(I.MaskDesc(I.PREFIX_LM, s, prefix_len=p)) == \
        p * p + (s * (s + 1) - p * (p + 1)) // 2
    n = s // 2048
    assert oracle.n_valid_closed_form(I.MaskDesc(I.CAUSAL_BLOCKWISE, s, block=2048)) == \
        2048 * 2048 * n * (n + 1) // 2
    q, a = 2048, 7680
    cu = I.shared_question_cu(q, [a] * 4)
    assert cu[-1] == s
    assert oracle.n_valid_closed_form(I.MaskDesc(I.SHARED_QUESTION, s, cu_seqlens=cu)) == \
        q * (q + 1) // 2 + 4 * (a * (a + 1) // 2 + a * q)


def test_popcount_matches_closed_form_at_moderate_size():
    s = 4096
    cu = I.cu_from_lengths(I.lognormal_doc_lengths(s, 3, mu=np.log(512)))
    for d in [I.make_desc(I.GLOBAL_SLIDING, s, num_global=256, window=1024),
              I.make_desc(I.BLOCK_CAUSAL_DOCUMENT, s, block=512, cu_seqlens=cu),
              I.make_desc(I.SHARED_QUESTION, s, question=256, answers=[960] * 4),
              I.make_desc(I.PREFIX_LM, s)]:
        assert oracle.n_valid_popcount(d) == oracle.n_valid_closed_form(d)


def _eq(a, b):
    return np.array_equal(oracle.materialize_mask(a), oracle.materialize_mask(b))


@pytest.mark.parametrize("s", [1, 5, 33, 130])
def test_mask_reductions(s):
    causal = I.MaskDesc(I.CAUSAL, s)
    full = I.MaskDesc(I.FULL, s)
    assert _eq(I.MaskDesc(I.SLIDING_WINDOW, s, window=s), causal)
    assert _eq(I.MaskDesc(I.SLIDING_WINDOW, s, window=s + 7), causal)
    w = max(1, s // 3)
    assert _eq(I.MaskDesc(I.GLOBAL_SLIDING, s, num_global=0, window=w, base_causal=1),
               I.MaskDesc(I.SLIDING_WINDOW, s, window=w))
    assert _eq(I.MaskDesc(I.PREFIX_LM, s, prefix_len=0), causal)
    assert _eq(I.MaskDesc(I.PREFIX_LM, s, prefix_len=1), causal)
    assert _eq(I.MaskDesc(I.PREFIX_LM, s, prefix_len=s), full)
    assert _eq(I.MaskDesc(I.CAUSAL_BLOCKWISE, s, block=1), causal)
    assert _eq(I.MaskDesc(I.CAUSAL_BLOCKWISE, s, block=s), full)
    one_doc = np.array([0, s], np.int32)
    b = max(1, s // 4)
    assert _eq(I.MaskDesc(I.BLOCK_CAUSAL_DOCUMENT, s, block=b, cu_seqlens=one_doc),
               I.MaskDesc(I.CAUSAL_BLOCKWISE, s, block=b))
    cu = I.cu_from_lengths(I.lognormal_doc_lengths(s, 1, mu=np.log(max(2, s // 3)), lo=1))
    assert _eq(I.MaskDesc(I.BLOCK_CAUSAL_DOCUMENT, s, block=1, cu_seqlens=cu),
               I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=cu))
    assert _eq(I.MaskDesc(I.SLIDING_WINDOW_DOCUMENT, s, window=s, cu_seqlens=cu),
               I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=cu))
    assert _eq(I.MaskDesc(I.SLIDING_WINDOW_DOCUMENT, s, window=w, cu_seqlens=one_doc),
               I.MaskDesc(I.SLIDING_WINDOW, s, window=w))
    assert np.array_equal(oracle.materialize_mask(
        I.MaskDesc(I.SLIDING_WINDOW_DOCUMENT, s, window=1, cu_seqlens=cu)), np.eye(s, dtype=bool))
    if s >= 2:
        assert _eq(I.MaskDesc(I.SHARED_QUESTION, s, cu_seqlens=I.shared_question_cu(1, [s - 1])),
                   causal)
    # all-ones block maps reduce to their base masks
    ones = np.ones((1, (s + 3) // 4, (s + 3) // 4), np.uint8)
    assert _eq(I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=4, block_map=ones), full)
    assert _eq(I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=4, block_map=ones, base_causal=1),
               causal)
    ro, co, _ = I.variable_block_map(s, 1, seed=s)
    vones = np.ones((1, ro.shape[1] - 1, co.shape[1] - 1), np.uint8)
    assert _eq(I.MaskDesc(I.BLOCK_SPARSE_VARIABLE, s, base_causal=1, cu_seqlens=cu,
                          row_offsets=ro, col_offsets=co, block_map=vones),
               I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=cu))


def test_diagonal_only_map_is_identity_mask():
    s, b = 12, 1
    eye = np.eye(s, dtype=np.uint8)[None]
    m = oracle.materialize_mask(I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=b, block_map=eye))
    assert np.array_equal(m, np.eye(s, dtype=bool))


def test_doc_lengths_recipe():
    for s, seed in [(8192, 0), (32768, 1), (131072, 2), (300, 3)]:
        lens = I.lognormal_doc_lengths(s, seed)
        assert sum(lens) == s
        assert all(128 <= x <= s for x in lens[:-1])
        assert 1 <= lens[-1] <= s
    assert I.lognormal_doc_lengths(8192, 5) == I.lognormal_doc_lengths(8192, 5)


def test_uniform_map_recipe():
    m = I.uniform_block_map(4096, 64, 3, 0.8, 7)
    assert m.shape == (3, 64, 64)
    assert (m[:, np.arange(64), np.arange(64)] == 1).all()
    off = ~np.eye(64, dtype=bool)
    frac = m[:, off].mean()
    assert abs(frac - 0.2) < 0.03


def test_variable_map_recipe():
    s = 20000
    ro, co, bm = I.variable_block_map(s, 4, seed=11)
    sizes = set(I.VARIABLE_BLOCK_SIZES)
    for h in range(4):
        for off in (ro[h], co[h]):
            valid = off[: np.searchsorted(off, s) + 1]
            assert valid[0] == 0 and valid[-1] == s
            d = np.diff(valid)
            assert all(x in sizes for x in d[:-1]) and 1 <= d[-1] <= 256
        r = ro[h][: np.searchsorted(ro[h], s) + 1]
        c = co[h][: np.searchsorted(co[h], s) + 1]
        nr, nc = len(r) - 1, len(c) - 1
        causal_blk = c[:-1][None, :] <= r[1:][:, None] - 1
        diag = (r[:-1][:, None] < c[1:][None, :]) & (c[:-1][None, :] < r[1:][:, None])
        sub = bm[h, :nr, :nc].astype(bool)
        assert sub[diag].all()
        assert not sub[~causal_blk].any()
        frac = sub[causal_blk & ~diag].mean()
        assert abs(frac - 0.5) < 0.05
