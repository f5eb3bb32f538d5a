"""Pins for the oracle's tile plan (CPU)."""
import numpy as np
import pytest

import oracle
from long_context_masked_gb300 import inputs as I
from tests._golden import load_plan_case


@pytest.mark.parametrize("name", ["plan_small.txt", "plan_halves.txt"])
def test_hand_worked_plan(name):
    desc, tq, tk, exp = load_plan_case(name)
    p = oracle.tile_plan_ref(desc, tq, tk)
    for key, val in exp.items():
        assert np.array_equal(p[key].astype(np.int64), val.astype(np.int64)), key


def _tile_popcounts(m, tq, tk):
    """Allowed pairs and in-range pairs per tile, and allowed pairs per tile half:
    halves[..., 0:2] key columns [0, tk/2) / [tk/2, tk), [..., 2:4] query rows."""
    s = m.shape[0]
    nq, nk = -(-s // tq), -(-s // tk)
    out = np.zeros((nq, nk), np.int64)
    area = np.zeros((nq, nk), np.int64)
    halves = np.zeros((nq, nk, 4), np.int64)
    for a in range(nq):
        for b in range(nk):
            r0, c0 = a * tq, b * tk
            blk = m[r0:r0 + tq, c0:c0 + tk]
            out[a, b] = blk.sum()
            area[a, b] = blk.size
            halves[a, b, 0] = m[r0:r0 + tq, c0:c0 + tk // 2].sum()
            halves[a, b, 1] = m[r0:r0 + tq, c0 + tk // 2:c0 + tk].sum()
            halves[a, b, 2] = m[r0:r0 + tq // 2, c0:c0 + tk].sum()
            halves[a, b, 3] = m[r0 + tq // 2:r0 + tq, c0:c0 + tk].sum()
    return out, area, halves


@pytest.mark.parametrize("seed", range(4))
def test_plan_consistent_with_mask(seed):
    rng = np.random.default_rng(seed)
    s = int(rng.integers(50, 400))
    tq, tk = [(16, 16), (16, 32), (32, 16), (64, 64)][seed]
    cu = I.cu_from_lengths(I.lognormal_doc_lengths(s, seed, mu=np.log(40), lo=5))
    bm = I.uniform_block_map(s, 8, 3, 0.6, seed)
    ro, co, vm = I.variable_block_map(s, 2, seed)
    q = max(1, s // 7)
    rest = s - q
    descs = [
        I.MaskDesc(I.CAUSAL, s), I.MaskDesc(I.FULL, s),
        I.MaskDesc(I.SLIDING_WINDOW, s, window=37),
        I.MaskDesc(I.FULL_DOCUMENT, s, cu_seqlens=cu),
        I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=cu),
        I.MaskDesc(I.SLIDING_WINDOW_DOCUMENT, s, window=23, cu_seqlens=cu),
        I.MaskDesc(I.PREFIX_LM, s, prefix_len=s // 4),
        I.MaskDesc(I.SHARED_QUESTION, s,
                   cu_seqlens=np.array([0, q, q + rest // 2, s], np.int32)),
        I.MaskDesc(I.GLOBAL_SLIDING, s, num_global=5, window=29),
        I.MaskDesc(I.GLOBAL_SLIDING, s, num_global=5, window=29, base_causal=0),
        I.MaskDesc(I.CAUSAL_BLOCKWISE, s, block=19),
        I.MaskDesc(I.BLOCK_CAUSAL_DOCUMENT, s, block=12, cu_seqlens=cu),
        I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=8, map_heads=3, block_map=bm,
                   n_row_blocks=bm.shape[1], n_col_blocks=bm.shape[2]),
        I.MaskDesc(I.BLOCK_SPARSE_VARIABLE, s, base_causal=1, cu_seqlens=cu, map_heads=2,
                   row_offsets=ro, col_offsets=co, block_map=vm,
                   n_row_blocks=vm.shape[1], n_col_blocks=vm.shape[2]),
    ]
    for d in descs:
        p = oracle.tile_plan_ref(d, tq, tk)
        for hm in range(d.map_heads):
            m = oracle.materialize_mask(d, hm)
            pc, area, halves = _tile_popcounts(m, tq, tk)
            cls = p["cls"][hm].astype(np.int64)
            assert ((cls == 0) == (pc == 0)).all()
            assert (((cls & 3) == 1) == (pc == area)).all()
            assert ((cls & 3) != 3).all() and (cls < 64).all()
            for bit, x in ((4, 0), (8, 1), (16, 2), (32, 3)):
                flag = (cls & bit) != 0
                assert (flag == ((pc > 0) & (halves[..., x] == 0))).all(), bit
            assert pc.sum() == oracle.n_valid_popcount(d, hm)
        # CSR rows, CSR columns and the class array describe the same tiles
        hmn, nq, nk = p["cls"].shape
        rows = p["cls"].reshape(hmn * nq, nk)
        for r in range(hmn * nq):
            a, b = p["rowptr"][r], p["rowptr"][r + 1]
            assert np.array_equal(p["kt_idx"][a:b], np.nonzero(rows[r])[0])
            assert np.array_equal(p["kt_cls"][a:b], rows[r][rows[r] != 0] & 15)
        cols = np.transpose(p["cls"], (0, 2, 1)).reshape(hmn * nk, nq)
        for c in range(hmn * nk):
            a, b = p["colptr"][c], p["colptr"][c + 1]
            assert np.array_equal(p["qt_idx"][a:b], np.nonzero(cols[c])[0])
            nz = cols[c][cols[c] != 0]
            assert np.array_equal(p["qt_cls"][a:b], (nz & 3) | ((nz >> 4) << 2))
        # longest first, ties by index, a permutation
        for key, ptr in (("work_q", "rowptr"), ("work_k", "colptr")):
            lens = np.diff(p[ptr])
            w = p[key]
            assert sorted(w.tolist()) == list(range(len(lens)))
            pairs = list(zip(-lens[w], w))
            assert pairs == sorted(pairs)


def test_tile_rows_matches_full_plan():
    s = 300
    desc = I.MaskDesc(I.GLOBAL_SLIDING, s, num_global=20, window=50, base_causal=1)
    p = oracle.tile_plan_ref(desc, 32, 64)
    rows = oracle.tile_rows_ref(desc, 32, 64, 0, [0, 3, 9])
    assert np.array_equal(rows, p["cls"][0, [0, 3, 9]])
