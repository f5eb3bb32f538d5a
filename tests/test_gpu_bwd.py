"""Backward parity of the CUDA path with the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import inputs as I
from tests._gpu import (check_grad, make_inputs, oracle_bwd_heads, oracle_dkdv_cols,
                        sampled_cols, small_descs, to_np)

pytestmark = pytest.mark.gpu


def _run(desc, dev, scale=None, tiles=(128, 128)):
    plan = lca.mask_build(desc, *tiles)
    q, k, v, do = dev
    o, lse = lca.attn_fwd(plan, q, k, v, scale=scale)
    dq, dk, dv = lca.attn_bwd(plan, q, k, v, o, do, lse, scale=scale)
    assert lca.last_device_error() == 0
    return plan, (o, lse), (dq, dk, dv)


def _check_all(desc, host, dev, scale=None, what=""):
    _, _, grads = _run(desc, dev, scale=scale)
    ref = oracle.attn_bwd_ref(*host, desc, scale=scale)
    for name, g in zip(("dQ", "dK", "dV"), grads):
        check_grad(to_np(g), ref[name], f"{what}{desc.name} {name}")


@pytest.mark.parametrize("mask", [I.FULL, I.CAUSAL])
def test_tiny_config_in_full(mask):
    host, dev = make_inputs(1, 1024, 4, 4, seed=0)
    _check_all(I.make_desc(mask, 1024), host, dev)


@pytest.mark.parametrize("s", [1000, 1408])
def test_every_mask_type_gqa(s):
    hq, hkv = 8, 2
    host, dev = make_inputs(1, s, hq, hkv, seed=s + 1)
    for desc in small_descs(s, hq, hkv, seed=s):
        _check_all(desc, host, dev)


def test_batched_and_scaled():
    host, dev = make_inputs(2, 300, 4, 2, seed=9)
    for mask in (I.FULL, I.CAUSAL, I.GLOBAL_SLIDING):
        desc = I.make_desc(mask, 300, num_global=20, window=60)
        _check_all(desc, host, dev, scale=0.2)


def test_per_query_head_maps_under_gqa():
    s, hq, hkv = 640, 4, 2
    host, dev = make_inputs(1, s, hq, hkv, seed=21)
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=0.6, map_heads=hq,
                       map_seed=4)
    _check_all(desc, host, dev)


def test_empty_rows_and_tiny_sequences():
    s = 640
    bm = np.ones((1, 10, 10), np.uint8)
    bm[0, 3, :] = 0
    bm[0, :, 7] = 0           # key block 7 is never attended: dK = dV = 0 there
    desc = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=64, block_map=bm, n_row_blocks=10,
                      n_col_blocks=10)
    host, dev = make_inputs(1, s, 2, 2, seed=5)
    _, _, (dq, dk, dv) = _run(desc, dev)
    assert (to_np(dq)[0, 192:256] == 0).all()
    assert (to_np(dk)[0, 448:512] == 0).all() and (to_np(dv)[0, 448:512] == 0).all()
    _check_all(desc, host, dev)
    for s in (1, 7, 130):
        host, dev = make_inputs(1, s, 2, 1, seed=s)
        for mask in (I.FULL, I.CAUSAL):
            _check_all(I.make_desc(mask, s), host, dev)


def test_deterministic():
    s = 2048
    host, dev = make_inputs(1, s, 8, 2, seed=3)
    desc = I.make_desc(I.CAUSAL_DOCUMENT, s, doc_seed=2)
    _, _, g1 = _run(desc, dev)
    _, _, g2 = _run(desc, dev)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("mask,kw", [(I.FULL, {}), (I.CAUSAL, {}),
                                     (I.SLIDING_WINDOW, {"window": 1024}),
                                     (I.FULL_DOCUMENT, {"doc_seed": 4}),
                                     (I.CAUSAL_DOCUMENT, {"doc_seed": 4}),
                                     (I.SHARED_QUESTION, {"question": 512, "answers": [896] * 4}),
                                     (I.BLOCK_CAUSAL_DOCUMENT, {"block": 512, "doc_seed": 4})])
def test_one_kv_group_medium_in_full(mask, kw):
    # one KV group of the 64:8 layout (8 query heads) at S = 4096, all rows
    s = 4096
    host, dev = make_inputs(1, s, 8, 1, seed=50 + mask)
    _check_all(I.make_desc(mask, s, **kw), host, dev)


@pytest.mark.parametrize("s,hq,hkv,mask,kw", [
    (16384, 4, 2, I.CAUSAL, {}),
    (16384, 4, 2, I.FULL_DOCUMENT, {"doc_seed": 11}),
    (32768, 2, 2, I.GLOBAL_SLIDING, {"num_global": 256, "window": 4096}),
    (16384, 16, 2, I.CAUSAL, {}),
    (16384, 4, 2, I.BLOCK_CAUSAL_DOCUMENT, {"block": 1024, "doc_seed": 12}),
    (16384, 4, 2, I.BLOCK_SPARSE_VARIABLE, {"map_heads": 2, "map_seed": 13, "doc_seed": 13}),
])
def test_multi_wave_grids_in_full(s, hq, hkv, mask, kw):
    """dQ, dK and dV compared element by element with the full fp64 backward on grids of
    several waves (256-512 dK/dV CTAs, 512-2048 dQ CTAs): the longest-first launch order,
    the 16-item launch chunks and the group loops of the dK/dV kernel across waves.
    16:2 at 16K runs one KV group of the 64:8 layout twice; BLOCK_CAUSAL_DOCUMENT takes
    the pages' block of 1024; the variable block map over documents is the long-varlen
    workload's mask at a size the full oracle finishes."""
    host, dev = make_inputs(1, s, hq, hkv, seed=700 + hq + mask)
    desc = I.make_desc(mask, s, **kw)
    _, _, grads = _run(desc, dev)
    ref = oracle_bwd_heads(host, desc, range(hq))
    for name, g in zip(("dQ", "dK", "dV"), grads):
        check_grad(to_np(g), ref[name], f"{desc.name} {hq}:{hkv} S={s} {name}")


def _sampled_dkdv(desc, host, grads, kv_heads, ncols, seed):
    """dK/dV rows of sampled keys against the oracle's key-column backward, per KV head."""
    s = host[0].shape[1]
    cols = sampled_cols(s, ncols, seed)
    rk, rv = oracle_dkdv_cols(host, desc, kv_heads, cols)
    for a, hk in enumerate(kv_heads):
        check_grad(to_np(grads[1][0, cols, hk]), rk[a], f"{desc.name} dK cols hk{hk}")
        check_grad(to_np(grads[2][0, cols, hk]), rv[a], f"{desc.name} dV cols hk{hk}")


def _invariants(desc, host, dev, grads, plan):
    """Properties that hold at any size: for every KV head, sum_j dK_j = 0 and
    sum_j dV_j = sum of dO over the group's non-empty rows (rows of P sum to 1)."""
    dq, dk, dv = (to_np(g) for g in grads)
    _, s, hq, d = host[0].shape
    hkv = host[1].shape[2]
    g = hq // hkv
    do = host[3]
    for hk in range(hkv):
        sk = dk[0, :, hk].sum(axis=0)
        scale_k = np.sqrt(s) * np.sqrt((dk[0, :, hk] ** 2).mean()) + 1e-30
        assert np.abs(sk).max() <= 0.05 * scale_k, f"{desc.name} sum dK, hk={hk}"
        sv = dv[0, :, hk].sum(axis=0)
        ref = do[0, :, hk * g:(hk + 1) * g].sum(axis=(0, 1))
        scale_v = np.sqrt(s * g) * np.sqrt((do[0, :, hk * g:(hk + 1) * g] ** 2).mean())
        assert np.abs(sv - ref).max() <= 0.05 * scale_v, f"{desc.name} sum dV, hk={hk}"


def _sampled_dq(desc, host, grads, heads, nrows, seed):
    dq = grads[0]
    s = host[0].shape[1]
    rng = np.random.default_rng(seed)
    rows = np.sort(np.concatenate([rng.choice(s, nrows - 2, replace=False), [0, s - 1]]))
    ref, _, _, _ = oracle.attn_dq_rows_ref(*host, desc, heads=heads, rows=rows)
    for a, h in enumerate(heads):
        check_grad(to_np(dq[0, rows, h]), ref[a], f"{desc.name} dQ rows h{h}")


@pytest.mark.parametrize("mask,kw", [(I.FULL, {}), (I.CAUSAL, {}),
                                     (I.SLIDING_WINDOW, {"window": 4096}),
                                     (I.FULL_DOCUMENT, {"doc_seed": 1}),
                                     (I.CAUSAL_DOCUMENT, {"doc_seed": 1}),
                                     (I.SLIDING_WINDOW_DOCUMENT, {"window": 1024, "doc_seed": 2})])
def test_dense_regular_full_size(mask, kw):
    s = 16384
    host, dev = make_inputs(1, s, 64, 8, seed=300 + mask)
    desc = I.make_desc(mask, s, **kw)
    plan, _, grads = _run(desc, dev)
    _sampled_dq(desc, host, grads, heads=[0, 17, 63], nrows=24, seed=mask)
    _sampled_dkdv(desc, host, grads, kv_heads=[5], ncols=24, seed=mask)
    _invariants(desc, host, dev, grads, plan)


@pytest.mark.parametrize("mask,kw", [(I.PREFIX_LM, {}),
                                     (I.SHARED_QUESTION, {"question": 2048, "answers": [7680] * 4}),
                                     (I.GLOBAL_SLIDING, {"num_global": 256, "window": 4096}),
                                     (I.CAUSAL_BLOCKWISE, {"block": 2048}),
                                     (I.BLOCK_CAUSAL_DOCUMENT, {"block": 2048, "doc_seed": 2}),
                                     # the pages' block of 1024
                                     (I.BLOCK_CAUSAL_DOCUMENT, {"block": 1024, "doc_seed": 3})])
def test_heterogeneous_full_size(mask, kw):
    s = 32768
    host, dev = make_inputs(1, s, 64, 64, seed=400 + mask)
    desc = I.make_desc(mask, s, **kw)
    plan, _, grads = _run(desc, dev)
    _sampled_dq(desc, host, grads, heads=[0, 40], nrows=16, seed=mask)
    _sampled_dkdv(desc, host, grads, kv_heads=[40], ncols=16, seed=mask)
    _invariants(desc, host, dev, grads, plan)


@pytest.mark.parametrize("s,block,hq,hkv,sparsity", [(131072, 64, 64, 8, 0.5), (65536, 128, 32, 32, 0.8),
                                                     (32768, 64, 32, 32, 0.2)])
def test_uniform_block_sparse_full_size(s, block, hq, hkv, sparsity):
    map_heads = hkv if hq != hkv else hq
    host, dev = make_inputs(1, s, hq, hkv, seed=500 + block)
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=block, sparsity=sparsity,
                       map_heads=map_heads, map_seed=block)
    plan, _, grads = _run(desc, dev)
    _sampled_dq(desc, host, grads, heads=[0, hq - 1], nrows=12, seed=block)
    if s <= 32768:    # the key-column oracle evaluates every row that reaches a key
        _sampled_dkdv(desc, host, grads, kv_heads=[hkv - 1], ncols=12, seed=block)
    _invariants(desc, host, dev, grads, plan)


def test_variable_block_sparse_long_varlen():
    s = 131072
    host, dev = make_inputs(1, s, 64, 8, seed=600)
    desc = I.make_desc(I.BLOCK_SPARSE_VARIABLE, s, map_heads=8, map_seed=7, doc_seed=7)
    plan, _, grads = _run(desc, dev)
    _sampled_dq(desc, host, grads, heads=[0, 37], nrows=12, seed=7)
    _invariants(desc, host, dev, grads, plan)


@pytest.mark.parametrize("hq,hkv,b", [(8, 2, 1), (4, 4, 1), (4, 2, 2)])
def test_head_dim_64(hq, hkv, b):
    """head_dim 64: every mask type (one sequence), or the batched dense masks."""
    s = 1000
    host, dev = make_inputs(b, s, hq, hkv, seed=640 + hq, head_dim=64)
    descs = small_descs(s, hq, hkv, seed=7) if b == 1 else \
        [I.make_desc(m, s, window=120) for m in (I.FULL, I.CAUSAL, I.SLIDING_WINDOW)]
    for desc in descs:
        _check_all(desc, host, dev, what="d64 ")


def test_head_dim_64_medium_full_rows():
    s = 4096
    host, dev = make_inputs(1, s, 8, 1, seed=65, head_dim=64)
    for mask, kw in ((I.CAUSAL, {}), (I.CAUSAL_DOCUMENT, {"doc_seed": 3})):
        _check_all(I.make_desc(mask, s, **kw), host, dev, what="d64 ")
