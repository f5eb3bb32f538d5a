"""Bit-exact parity of the GPU mask builder with the oracle's brute-force plan."""
import numpy as np
import pytest

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import inputs as I
from tests._gpu import small_descs

pytestmark = pytest.mark.gpu

KEYS = ("rowptr", "kt_idx", "kt_cls", "colptr", "qt_idx", "qt_cls", "work_q", "work_k")


def _compare(desc, tq, tk):
    plan = lca.mask_build(desc, tq, tk)
    got = plan.export()
    ref = oracle.tile_plan_ref(desc, tq, tk)
    assert np.array_equal(got["cls"], ref["cls"]), f"{desc.name} cls"
    for key in KEYS:
        assert np.array_equal(got[key], ref[key]), f"{desc.name} {key}"
    for hm in range(desc.map_heads):
        assert got["n_valid"][hm] == oracle.n_valid_popcount(desc, hm), f"{desc.name} n_valid"
    info = plan.info
    assert info["nnz"] == len(ref["kt_idx"])
    assert info["n_partial"] == int(((ref["cls"] & 3) == 2).sum())


@pytest.mark.parametrize("s", [1000, 1408])
@pytest.mark.parametrize("tiles", [(128, 128), (128, 64), (64, 128), (64, 64)])
def test_plan_bit_exact_all_masks(s, tiles):
    for desc in small_descs(s, hq=4, hkv=2, seed=s):
        _compare(desc, *tiles)


@pytest.mark.parametrize("s", [1344, 950])
def test_plan_half_flags(s):
    # 64-token blocks against 128 tiles, and ragged tails whose second half is past S
    for seed, sp in ((1, 0.5), (2, 0.8)):
        _compare(I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=sp,
                             map_heads=2, map_seed=seed), 128, 128)
    _compare(I.make_desc(I.CAUSAL, s), 128, 128)
    _compare(I.make_desc(I.FULL, s), 128, 64)
    got = lca.mask_build(I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=0.5,
                                     map_heads=2, map_seed=1), 128, 128).export()
    flags = got["cls"][got["cls"] != 0] >> 2
    for bit in (1, 2, 4, 8):   # every flag occurs
        assert (flags & bit).any(), bit


def test_plan_degenerate_cases():
    # one token; a sequence shorter than a tile; an empty map row; all-zero map
    _compare(I.MaskDesc(I.CAUSAL, 1), 128, 128)
    _compare(I.MaskDesc(I.FULL, 77), 128, 64)
    bm = np.ones((1, 10, 10), np.uint8)
    bm[0, 3, :] = 0
    _compare(I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, 640, block=64, block_map=bm,
                        n_row_blocks=10, n_col_blocks=10), 128, 128)
    z = np.zeros((1, 5, 5), np.uint8)
    _compare(I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, 600, block=128, block_map=z,
                        n_row_blocks=5, n_col_blocks=5), 128, 128)
    _compare(I.MaskDesc(I.SLIDING_WINDOW, 900, window=1), 64, 64)
    _compare(I.MaskDesc(I.CAUSAL_DOCUMENT, 700, cu_seqlens=np.array([0, 1, 2, 300, 300, 700],
                                                                    np.int32)), 128, 128)


def _check_internal(got, n_qt, n_kt, hm_n):
    cls = got["cls"]
    rows = cls.reshape(hm_n * n_qt, n_kt)
    lens = np.count_nonzero(rows, axis=1)
    assert np.array_equal(np.diff(got["rowptr"]), lens)
    cols = np.transpose(cls, (0, 2, 1)).reshape(hm_n * n_kt, n_qt)
    assert np.array_equal(np.diff(got["colptr"]), np.count_nonzero(cols, axis=1))
    nz_r = np.nonzero(rows)
    assert np.array_equal(got["kt_idx"], nz_r[1])
    assert np.array_equal(got["kt_cls"], oracle.row_list_byte(rows[nz_r]))
    nz_c = np.nonzero(cols)
    assert np.array_equal(got["qt_idx"], nz_c[1])
    assert np.array_equal(got["qt_cls"], oracle.col_list_byte(cols[nz_c]))
    for key, ptr in (("work_q", "rowptr"), ("work_k", "colptr")):
        ln = np.diff(got[ptr])
        w = got[key]
        assert np.array_equal(np.sort(w), np.arange(len(ln)))
        assert np.array_equal(w, np.lexsort((np.arange(len(ln)), -ln)))


FULL_SIZE = [
    (I.FULL, dict()), (I.CAUSAL, dict()), (I.SLIDING_WINDOW, dict(window=4096)),
    (I.FULL_DOCUMENT, dict(doc_seed=3)), (I.CAUSAL_DOCUMENT, dict(doc_seed=3)),
]


@pytest.mark.parametrize("s", [8192, 49152])
def test_plan_full_size_dense_regular(s):
    for t, kw in FULL_SIZE:
        desc = I.make_desc(t, s, **kw)
        plan = lca.mask_build(desc, 128, 128)
        got = plan.export()
        n_qt = -(-s // 128)
        _check_internal(got, n_qt, n_qt, 1)
        assert got["n_valid"][0] == oracle.n_valid_closed_form(desc)
        qts = np.random.default_rng(s + t).choice(n_qt, 12, replace=False)
        assert np.array_equal(got["cls"][0, qts], oracle.tile_rows_ref(desc, 128, 128, 0, qts))


def test_plan_full_size_heterogeneous():
    s = 32768
    descs = [I.make_desc(I.PREFIX_LM, s), I.make_desc(I.SHARED_QUESTION, s, question=2048,
                                                      answers=[7680] * 4),
             I.make_desc(I.GLOBAL_SLIDING, s, num_global=256, window=4096),
             I.make_desc(I.CAUSAL_BLOCKWISE, s, block=2048),
             I.make_desc(I.BLOCK_CAUSAL_DOCUMENT, s, block=2048, doc_seed=1),
             I.make_desc(I.BLOCK_CAUSAL_DOCUMENT, s, block=1024, doc_seed=1)]
    for desc in descs:
        got = lca.mask_build(desc, 128, 128).export()
        _check_internal(got, 256, 256, 1)
        assert got["n_valid"][0] == oracle.n_valid_closed_form(desc), desc.name
        qts = np.random.default_rng(desc.type).choice(256, 10, replace=False)
        assert np.array_equal(got["cls"][0, qts], oracle.tile_rows_ref(desc, 128, 128, 0, qts))


@pytest.mark.parametrize("block,heads", [(64, 8), (128, 32)])
def test_plan_full_size_uniform_sparse(block, heads):
    s = 131072
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=block, sparsity=0.5,
                       map_heads=heads, map_seed=block)
    got = lca.mask_build(desc, 128, 128).export()
    _check_internal(got, 1024, 1024, heads)
    for hm in (0, heads - 1):
        assert got["n_valid"][hm] == oracle.n_valid_closed_form(desc, hm)
        qts = np.random.default_rng(hm).choice(1024, 4, replace=False)
        assert np.array_equal(got["cls"][hm, qts], oracle.tile_rows_ref(desc, 128, 128, hm, qts))


def test_plan_full_size_variable_sparse():
    s = 131072
    desc = I.make_desc(I.BLOCK_SPARSE_VARIABLE, s, map_heads=8, map_seed=5, doc_seed=5)
    got = lca.mask_build(desc, 128, 128).export()
    _check_internal(got, 1024, 1024, 8)
    for hm in (0, 7):
        qts = np.random.default_rng(hm).choice(1024, 4, replace=False)
        assert np.array_equal(got["cls"][hm, qts], oracle.tile_rows_ref(desc, 128, 128, hm, qts))
    # exact pair counts on the same recipe at a size the oracle counts quickly
    small = I.make_desc(I.BLOCK_SPARSE_VARIABLE, 16384, map_heads=2, map_seed=5, doc_seed=5)
    g2 = lca.mask_build(small, 128, 128).export()
    for hm in range(2):
        assert g2["n_valid"][hm] == oracle.n_valid_popcount(small, hm)


def test_plan_reports_its_device_memory():
    """lca_plan_info.device_bytes covers at least the arrays lca_plan_export copies out
    and the plan's copy of the block map."""
    s = 2000
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=0.5, map_heads=2,
                       map_seed=1)
    plan = lca.mask_build(desc, 128, 128)
    inf = plan.info
    hm, nq, nk, nnz = inf["map_heads"], inf["n_qt"], inf["n_kt"], inf["nnz"]
    exported = (hm * nq * nk + 4 * (hm * nq + 1) + 5 * nnz + 4 * (hm * nk + 1) + 5 * nnz
                + 4 * hm * (nq + nk) + 8 * hm)
    assert inf["device_bytes"] >= exported + desc.block_map.nbytes
    assert inf["device_bytes"] < 4 * (exported + desc.block_map.nbytes) + (1 << 20)
