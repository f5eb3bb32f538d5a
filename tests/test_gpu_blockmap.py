"""Block maps from block scores on the GPU (lca_block_scores, lca_block_topk) against
the fp64 oracle, and the resulting block-sparse attention end to end."""
import math

import numpy as np
import pytest
import torch

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import inputs as I
from tests._gpu import check_grad, check_lse, check_o, make_inputs, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hm,nr,nc,sparsity,quant", [
    (8, 37, 300, 0.2, None), (8, 37, 300, 0.5, None), (8, 37, 300, 0.8, None),
    (2, 5, 7, 0.5, 3), (4, 16, 1024, 0.5, 5), (1, 3, 2048, 0.8, None), (3, 9, 256, 0.0, None),
    (2, 4, 257, 0.99, 2)])
def test_topk_bit_exact(hm, nr, nc, sparsity, quant):
    """Random scores (the benchmark's own sampling), with many ties when quantised."""
    s = I.random_block_scores(hm, nr, nc, seed=nc + hm)
    if quant:
        s = np.floor(s * quant).astype(np.float32) - 1.0      # a few distinct values, negatives
    k = oracle.topk_count(nc, sparsity)
    got = lca.block_topk(torch.from_numpy(s).cuda(), k)
    assert lca.last_device_error() == 0
    assert np.array_equal(to_np(got), oracle.topk_block_map(s, k))


def _score_tol(ref):
    """fp32 pooling (sums of up to a few thousand bf16 values) and a 128-term fp32 dot
    product: errors of order 1e-6 relative to the largest score of the map head."""
    return np.broadcast_to(1e-4 * np.abs(ref).max(axis=(1, 2), keepdims=True) + 1e-9, ref.shape)


@pytest.mark.parametrize("s,hq,hkv,block,map_heads", [
    (1000, 8, 2, 64, 1), (1000, 8, 2, 64, 2), (1000, 8, 2, 128, 8), (777, 4, 4, 100, 4),
    (2048, 8, 1, 128, 1)])
def test_pooled_scores(s, hq, hkv, block, map_heads):
    host, dev = make_inputs(1, s, hq, hkv, seed=s + block)
    got = to_np(lca.block_scores(dev[0], dev[1], block, map_heads))
    ref = oracle.pooled_block_scores(host[0], host[1], block, map_heads)
    tol = _score_tol(ref)
    assert lca.last_device_error() == 0
    assert got.shape == ref.shape
    assert (np.abs(got - ref) <= tol).all(), np.abs(got - ref).max()


def _check_map_from_scores(got_map, ref_scores, tol, k):
    """Exact where the k-th / (k+1)-th oracle scores are further apart than the score
    error; elsewhere the selection must be valid within that error."""
    hm, nr, nc = ref_scores.shape
    ref_map = oracle.topk_block_map(ref_scores, k)
    assert (got_map.sum(axis=2) == k).all()
    for h in range(hm):
        for r in range(nr):
            row = ref_scores[h, r]
            srt = np.sort(row)[::-1]
            margin = srt[k - 1] - srt[k] if k < nc else np.inf
            if margin > 2 * tol[h, r].max():
                assert np.array_equal(got_map[h, r], ref_map[h, r]), (h, r)
            else:
                sel, rest = row[got_map[h, r] == 1], row[got_map[h, r] == 0]
                if rest.size:
                    assert sel.min() >= rest.max() - 2 * tol[h, r].max()


@pytest.mark.parametrize("sparsity", [0.2, 0.5, 0.8])
def test_dynamic_map_from_pooled_scores(sparsity):
    s, hq, hkv, block = 2048, 8, 2, 64
    host, dev = make_inputs(1, s, hq, hkv, seed=77)
    scores = lca.block_scores(dev[0], dev[1], block, hkv)
    nb = scores.shape[1]
    k = oracle.topk_count(nb, sparsity)
    got = to_np(lca.block_topk(scores, k))
    ref = oracle.pooled_block_scores(host[0], host[1], block, hkv)
    _check_map_from_scores(got, ref, _score_tol(ref), k)


@pytest.mark.parametrize("block", [64, 128])
def test_topk_map_drives_sparse_attention(block):
    """Random-score top-k map built on the device, passed to lca_mask_build as a device
    array; the attention matches the oracle run on the oracle's own top-k map."""
    s, hq, hkv = 1000, 8, 2
    nb = (s + block - 1) // block
    scores = I.random_block_scores(hkv, nb, nb, seed=block)
    k = oracle.topk_count(nb, 0.5)
    dmap = lca.block_topk(torch.from_numpy(scores).cuda(), k)
    ref_map = oracle.topk_block_map(scores, k)
    assert np.array_equal(to_np(dmap), ref_map)
    mk = dict(block=block, map_heads=hkv, n_row_blocks=nb, n_col_blocks=nb)
    desc_gpu = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block_map=dmap, **mk)
    desc_ref = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block_map=ref_map, **mk)
    host, dev = make_inputs(1, s, hq, hkv, seed=block + 1)
    plan = lca.mask_build(desc_gpu, 128, 128)
    q, kk, v, do = dev
    o, lse = lca.attn_fwd(plan, q, kk, v)
    dq, dk, dv = lca.attn_bwd(plan, q, kk, v, o, do, lse)
    assert lca.last_device_error() == 0
    ref_o, ref_lse = oracle.attn_fwd_ref(*host[:3], desc_ref)
    check_o(to_np(o), ref_o, "topk O")
    check_lse(to_np(lse), ref_lse, "topk LSE")
    ref = oracle.attn_bwd_ref(*host, desc_ref)
    for name, g in zip(("dQ", "dK", "dV"), (dq, dk, dv)):
        check_grad(to_np(g), ref[name], f"topk {name}")


def test_full_size_dynamic_scores_sampled():
    """S = 32K, GQA 64:8, one map per KV head, 128-blocks: pooled scores of sampled
    map heads and query blocks against the oracle, and their top-k rows."""
    s, hq, hkv, block = 32768, 64, 8, 128
    q, k, _, _ = I.qkv_do(1, s, hq, hkv, 128, seed=11)
    scores = lca.block_scores(q.cuda(), k.cuda(), block, hkv)
    kk = oracle.topk_count(s // block, 0.5)
    dmap = to_np(lca.block_topk(scores, kk))
    scores = to_np(scores)
    assert lca.last_device_error() == 0
    for hm in (0, 5):
        qn = q[:, :, hm * 8:(hm + 1) * 8].float().numpy()
        kn = k[:, :, hm:hm + 1].float().numpy()
        ref = oracle.pooled_block_scores(qn, kn, block, 1)[0]
        tol = _score_tol(ref[None])[0]
        assert (np.abs(scores[hm] - ref) <= tol).all()
        _check_map_from_scores(dmap[hm][None], ref[None], tol[None], kk)
