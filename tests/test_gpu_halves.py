"""Parity of the half-width tile path: plan entries that flag one half of a tile as
empty (64-token sparse blocks against 128-token tiles, ragged tails past S).  Long
lists with enough flagged entries run the kernels' half-width loops (N = 64 recompute,
half the k-steps of the accumulating MMAs); short lists run the plain loops, which
treat a flagged tile as a partial full-width one.  Every element is compared with the
fp64 oracle, and each 64-row block of every gradient is held to the bar on its own, so
that an error confined to one half of a tile cannot hide in a tensor-wide norm."""
import numpy as np
import pytest

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import inputs as I
from tests._gpu import GRAD_REL_FRO, check_grad, check_lse, check_o, make_inputs, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _empty_rows(desc, hq, hkv, name):
    """[S, H] rows without any allowed pair: query rows (dQ, H = H_q) or key rows
    attended by no query of the heads sharing them (dK / dV, H = H_kv)."""
    masks = [oracle.materialize_mask(desc, hm) for hm in range(desc.map_heads)]
    mh = [oracle.map_head_of(h, hq, hkv, desc.map_heads) for h in range(hq)]
    if name == "dQ":
        return np.stack([~masks[mh[h]].any(axis=1) for h in range(hq)], axis=1)
    g = hq // hkv
    return np.stack([~np.any([masks[mh[hk * g + x]].any(axis=0) for x in range(g)], axis=0)
                     for hk in range(hkv)], axis=1)


def _check_blocks(g, ref, empty, what):
    """Every 64-row block of [B, S, H, d] within the bar on its own; rows without any
    allowed pair exactly 0."""
    assert (g.transpose(1, 2, 0, 3)[empty] == 0).all(), f"{what}: rows without pairs not 0"
    for r0 in range(0, g.shape[1], 64):
        gb, rb = g[:, r0:r0 + 64], ref[:, r0:r0 + 64]
        if np.any(rb != 0):
            e = rel_fro(gb, rb)
            assert e <= GRAD_REL_FRO, f"{what} rows {r0}+64: relative Frobenius {e:.3e}"


def _half_path_lists(ptr, ent, share):
    """Lists the kernels run on the half-width path: at least 64 entries, at least
    1/share of them flagged (share 4 in the forward, 2 in the backward)."""
    n = np.diff(ptr)
    f = np.add.reduceat((ent >> 2) != 0, ptr[:-1]) if len(ent) else np.zeros_like(n)
    f = np.where(n > 0, f, 0)
    return int(((n >= 64) & (share * f >= n)).sum())


def _run(desc, b, s, hq, hkv, seed, head_dim=128, half_path=False):
    host, dev = make_inputs(b, s, hq, hkv, seed=seed, head_dim=head_dim)
    plan = lca.mask_build(desc, 128, 128)
    exp = plan.export()
    assert (exp["cls"] >> 2).any(), "case without a flagged half"
    fwd_rows = _half_path_lists(exp["rowptr"], exp["kt_cls"], 4)
    dq_rows = _half_path_lists(exp["rowptr"], exp["kt_cls"], 2)
    kv_cols = _half_path_lists(exp["colptr"], exp["qt_cls"], 2)
    if half_path:
        assert fwd_rows > 0, fwd_rows
    if half_path == "all":
        assert dq_rows > 0 and kv_cols > 0, (dq_rows, kv_cols)
    q, k, v, do = dev
    o, lse = lca.attn_fwd(plan, q, k, v)
    dq, dk, dv = lca.attn_bwd(plan, q, k, v, o, do, lse)
    assert lca.last_device_error() == 0
    o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc)
    check_o(to_np(o), o_ref, desc.name)
    check_lse(lse.cpu().numpy().astype(np.float64), lse_ref, desc.name)
    ref = oracle.attn_bwd_ref(*host, desc)
    for name, g in zip(("dQ", "dK", "dV"), (dq, dk, dv)):
        g = to_np(g)
        check_grad(g, ref[name], f"{desc.name} {name}")
        _check_blocks(g, ref[name], _empty_rows(desc, hq, hkv, name), f"{desc.name} {name}")


@pytest.mark.parametrize("sparsity", [0.5, 0.8])
def test_sparse_64_blocks_long_lists(sparsity):
    # 128.5 tiles: long lists on the half-width path, and a ragged last half
    s = 16448
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=sparsity,
                       map_heads=1, map_seed=int(10 * sparsity))
    _run(desc, 1, s, 2, 1, seed=s + int(10 * sparsity),
         half_path="all" if sparsity == 0.8 else True)


def test_sparse_64_blocks_long_lists_per_query_head_d64():
    s = 16448
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=0.6, map_heads=2,
                       map_seed=8)
    _run(desc, 1, s, 2, 1, seed=8, head_dim=64, half_path=True)


@pytest.mark.parametrize("s", [1344, 1088])
@pytest.mark.parametrize("sparsity", [0.5, 0.8])
def test_sparse_64_blocks_gqa(s, sparsity):
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=sparsity,
                       map_heads=2, map_seed=s + int(10 * sparsity))
    _run(desc, 1, s, 8, 2, seed=s)


def test_sparse_64_blocks_per_query_head():
    s = 1344
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=0.6, map_heads=4,
                       map_seed=3)
    _run(desc, 1, s, 4, 2, seed=5)


@pytest.mark.parametrize("mask", [I.FULL, I.CAUSAL, I.SLIDING_WINDOW])
def test_ragged_tail_half(mask):
    # S = 10.5 tiles: the last key tile's and query tile's second halves are past S
    s = 1344
    _run(I.make_desc(mask, s, window=200), 1, s, 4, 1, seed=mask)


def test_designed_half_patterns():
    """A map on 64-blocks where query tile 0 keeps only the left key halves, query tile
    1 only the right ones, and key tile 2 is reached only by the lower query halves."""
    s = 768
    nb = s // 64
    bm = np.zeros((1, nb, nb), np.uint8)
    bm[0, 0:2, 0:6:2] = 1          # rows 0-127: left halves of key tiles 0-2
    bm[0, 2:4, 1:6:2] = 1          # rows 128-255: right halves of key tiles 0-2
    bm[0, 5, 4:6] = 1              # key tile 2 from the lower half of query tile 2 only
    bm[0, 6:12, 6:12] = np.tril(np.ones((6, 6), np.uint8))
    desc = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=64, block_map=bm, n_row_blocks=nb,
                      n_col_blocks=nb)
    _run(desc, 1, s, 2, 1, seed=17)


def test_head_dim_64_half_tiles():
    s = 1344
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=0.5, map_heads=2,
                       map_seed=9)
    _run(desc, 1, s, 4, 2, seed=9, head_dim=64)
