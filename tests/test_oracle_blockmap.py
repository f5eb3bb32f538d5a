"""Pins of oracle.blockmap (top-k block maps and mean-pooled block scores) against
hand-worked values, brute force, closed forms and invariants."""
import math

import numpy as np
import pytest

import oracle.blockmap as BM
from tests._golden import float_matrix, load_blockmap_cases


CASES = load_blockmap_cases()


@pytest.mark.parametrize("name", ["topk k2", "topk k4"])
def test_topk_hand_worked(name):
    c = CASES[name]
    scores = float_matrix(c["scores"])[None]
    got = BM.topk_block_map(scores, int(c["k"]))
    assert np.array_equal(got[0], float_matrix(c["map"]).astype(np.uint8))


def test_pooled_scores_hand_worked():
    c = CASES["pooled S3 block2"]
    q = float_matrix(c["q"]).reshape(1, 3, 2, 2)
    k = float_matrix(c["k"]).reshape(1, 3, 1, 2)
    got = BM.pooled_block_scores(q, k, block=2, map_heads=1)
    assert np.allclose(got[0] * math.sqrt(2.0), float_matrix(c["scores_times_sqrt2"]), atol=1e-12)


@pytest.mark.parametrize("n,s,k", [(10, 0.2, 8), (10, 0.5, 5), (10, 0.8, 2), (3, 0.9, 1),
                                   (7, 0.0, 7), (256, 0.5, 128), (1, 0.8, 1)])
def test_topk_count(n, s, k):
    assert BM.topk_count(n, s) == k


def test_topk_properties_random():
    rng = np.random.default_rng(3)
    scores = rng.integers(0, 6, size=(3, 9, 17)).astype(np.float64)   # many ties
    for k in (1, 5, 17):
        m = BM.topk_block_map(scores, k)
        assert (m.sum(axis=2) == k).all()
        for h in range(3):
            for r in range(9):
                sel, rest = scores[h, r][m[h, r] == 1], scores[h, r][m[h, r] == 0]
                if rest.size:
                    assert sel.min() >= rest.max()
                    # on the boundary value, the kept entries are the lowest indices
                    t = sel.min()
                    eq = np.flatnonzero(scores[h, r] == t)
                    kept = np.flatnonzero((scores[h, r] == t) & (m[h, r] == 1))
                    assert np.array_equal(kept, eq[:kept.size])


def test_topk_all_equal_keeps_first_k():
    m = BM.topk_block_map(np.zeros((1, 4, 6)), 3)
    assert (m[0, :, :3] == 1).all() and (m[0, :, 3:] == 0).all()


def _brute_scores(q, k, block, map_heads):
    """Scalar loops over rows, heads and dimensions."""
    _, s, hq, d = q.shape
    hkv = k.shape[2]
    g = hq // hkv
    nb = (s + block - 1) // block
    out = np.zeros((map_heads, nb, nb))
    for hm in range(map_heads):
        if map_heads == 1:
            qh = list(range(hq))
        elif map_heads == hkv:
            qh = [h for h in range(hq) if h // g == hm]
        else:
            qh = [hm]
        kvh = sorted({h // g for h in qh})
        for r in range(nb):
            for c in range(nb):
                acc = 0.0
                for x in range(d):
                    qs, qn = 0.0, 0
                    for i in range(r * block, min(s, (r + 1) * block)):
                        for h in qh:
                            qs += float(q[0, i, h, x])
                            qn += 1
                    ks, kn = 0.0, 0
                    for j in range(c * block, min(s, (c + 1) * block)):
                        for h in kvh:
                            ks += float(k[0, j, h, x])
                            kn += 1
                    acc += (qs / qn) * (ks / kn)
                out[hm, r, c] = acc / math.sqrt(d)
    return out


@pytest.mark.parametrize("hq,hkv,map_heads", [(4, 2, 1), (4, 2, 2), (4, 2, 4), (2, 2, 2)])
def test_pooled_scores_brute_force(hq, hkv, map_heads):
    rng = np.random.default_rng(hq * 10 + map_heads)
    s, d, block = 11, 4, 4                       # three blocks, the last one short
    q = rng.standard_normal((1, s, hq, d))
    k = rng.standard_normal((1, s, hkv, d))
    got = BM.pooled_block_scores(q, k, block, map_heads)
    assert np.allclose(got, _brute_scores(q, k, block, map_heads), rtol=1e-12, atol=1e-12)


def test_pooled_scores_constant_inputs_and_invariances():
    s, d, block = 20, 8, 6
    a = np.arange(1, d + 1, dtype=np.float64)
    bvec = np.linspace(-1, 1, d)
    q = np.broadcast_to(a, (1, s, 4, d)).copy()
    k = np.broadcast_to(bvec, (1, s, 2, d)).copy()
    got = BM.pooled_block_scores(q, k, block, 2)
    assert np.allclose(got, a @ bvec / math.sqrt(d))
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, s, 4, d))
    k = rng.standard_normal((1, s, 2, d))
    base = BM.pooled_block_scores(q, k, block, 2)
    perm = np.arange(s)
    perm[:block] = perm[:block][::-1]            # permute rows inside block 0
    assert np.allclose(BM.pooled_block_scores(q[:, perm], k[:, perm], block, 2), base)
    assert np.allclose(BM.pooled_block_scores(3.0 * q, k, block, 2), 3.0 * base)
