"""Pins for the oracle's attention forward/backward (CPU, fp64)."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_masked_gb300 import inputs as I
from tests._golden import load_attention_closed_form


def _rand(shape, rng):
    return rng.standard_normal(shape)


def test_closed_form_cases():
    exp = load_attention_closed_form()
    # two_keys
    q = np.array([[[[math.log(3.0)]]]])
    k = np.array([[[[1.0]], [[0.0]]]]).reshape(1, 2, 1, 1)
    v = np.array([4.0, 8.0]).reshape(1, 2, 1, 1)
    kq = np.zeros((1, 2, 1, 1))
    kq[0, 0] = q[0, 0]
    desc = I.MaskDesc(I.FULL, 2)
    # query row 0 only matters; row 1 is a second query we ignore
    do = np.ones((1, 2, 1, 1))
    r = oracle.attn_bwd_ref(kq, k, v, do, desc, scale=1.0)
    got = {"O": r["O"][0, 0, 0, 0], "LSE": r["LSE"][0, 0, 0], "dQ": r["dQ"][0, 0, 0, 0]}
    # row 1 has q = 0 -> p = [1/2, 1/2]; its dS = p*(dP - D) with D = 6 -> [-1, 1]
    # and q = 0 adds nothing to dK, but adds p to dV: remove it.
    dk = r["dK"][0, :, 0, 0]
    dv = r["dV"][0, :, 0, 0] - np.array([0.5, 0.5])
    for case, qty, idx, val in exp:
        if case != "two_keys":
            continue
        if qty in got:
            assert got[qty] == pytest.approx(val, abs=1e-12)
        elif qty == "dK":
            assert dk[idx] == pytest.approx(val, abs=1e-12)
        elif qty == "dV":
            assert dv[idx] == pytest.approx(val, abs=1e-12)
    # causal_first_row
    q = np.array([2.0, 5.0]).reshape(1, 2, 1, 1)
    k = np.array([7.0, 1.0]).reshape(1, 2, 1, 1)
    v = np.array([3.0, 9.0]).reshape(1, 2, 1, 1)
    o, lse = oracle.attn_fwd_ref(q, k, v, I.MaskDesc(I.CAUSAL, 2), scale=1.0)
    for case, qty, idx, val in exp:
        if case != "causal_first_row":
            continue
        g = o[0, idx, 0, 0] if qty == "O" else lse[0, 0, idx]
        assert g == pytest.approx(val, rel=1e-14, abs=1e-13)


def _brute_force(q, k, v, do, desc, scale):
    """Scalar loops straight from the definition (no vectorisation)."""
    b_n, s, hq, d = q.shape
    hkv = k.shape[2]
    g = hq // hkv
    m_full = {hm: oracle.materialize_mask(desc, hm) for hm in range(desc.map_heads)}
    o = np.zeros_like(q)
    lse = np.full((b_n, hq, s), -np.inf)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(b_n):
        for h in range(hq):
            hk = h // g
            hm = oracle.map_head_of(h, hq, hkv, desc.map_heads)
            m = m_full[hm]
            for i in range(s):
                keys = [j for j in range(s) if m[i, j]]
                if not keys:
                    continue
                sc = {j: scale * sum(q[b, i, h, t] * k[b, j, hk, t] for t in range(d)) for j in keys}
                mx = max(sc.values())
                z = sum(math.exp(sc[j] - mx) for j in keys)
                lse[b, h, i] = mx + math.log(z)
                p = {j: math.exp(sc[j] - lse[b, h, i]) for j in keys}
                for t in range(d):
                    o[b, i, h, t] = sum(p[j] * v[b, j, hk, t] for j in keys)
                dp = {j: sum(do[b, i, h, t] * v[b, j, hk, t] for t in range(d)) for j in keys}
                dd = sum(p[j] * dp[j] for j in keys)
                for j in keys:
                    ds = p[j] * (dp[j] - dd)
                    for t in range(d):
                        dq[b, i, h, t] += scale * ds * k[b, j, hk, t]
                        dk[b, j, hk, t] += scale * ds * q[b, i, h, t]
                        dv[b, j, hk, t] += p[j] * do[b, i, h, t]
    return o, lse, dq, dk, dv


def _small_descs(s):
    cu = np.array([0, 5, 6, s], np.int32)
    bm = np.array([[[1, 0, 1, 0], [0, 0, 0, 0], [1, 1, 0, 1], [0, 1, 1, 1]],
                   [[0, 1, 0, 0], [1, 1, 1, 1], [0, 0, 1, 0], [1, 0, 0, 1]]], np.uint8)
    return [
        I.MaskDesc(I.FULL, s),
        I.MaskDesc(I.CAUSAL, s),
        I.MaskDesc(I.SLIDING_WINDOW, s, window=3),
        I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=cu),
        I.MaskDesc(I.FULL_DOCUMENT, s, cu_seqlens=cu),
        I.MaskDesc(I.GLOBAL_SLIDING, s, num_global=2, window=3, base_causal=1),
        # map head 0 has an all-zero block row -> empty query rows 4..7
        I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=4, map_heads=2, n_row_blocks=4,
                   n_col_blocks=4, block_map=bm),
    ]


@pytest.mark.parametrize("idx", range(7))
def test_brute_force_loops(idx):
    rng = np.random.default_rng(idx)
    s, d = 14, 4
    desc = _small_descs(s)[idx]
    hq, hkv = 4, 2
    q, do = _rand((1, s, hq, d), rng), _rand((1, s, hq, d), rng)
    k, v = _rand((1, s, hkv, d), rng), _rand((1, s, hkv, d), rng)
    sc = 0.7
    o, lse, dq, dk, dv = _brute_force(q, k, v, do, desc, sc)
    r = oracle.attn_bwd_ref(q, k, v, do, desc, scale=sc, chunk=5)
    np.testing.assert_allclose(r["O"], o, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(r["LSE"]), np.isinf(lse))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(r["LSE"][fin], lse[fin], atol=1e-12)
    np.testing.assert_allclose(r["dQ"], dq, atol=1e-12)
    np.testing.assert_allclose(r["dK"], dk, atol=1e-12)
    np.testing.assert_allclose(r["dV"], dv, atol=1e-12)
    o2, lse2 = oracle.attn_fwd_ref(q, k, v, desc, scale=sc, chunk=3)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    if idx == 6:
        assert np.isinf(lse[0, 0, 4:8]).all() and (o[0, 4:8, 0] == 0).all()


def test_finite_differences():
    rng = np.random.default_rng(42)
    s, d, hq, hkv = 10, 3, 4, 2
    desc = I.MaskDesc(I.GLOBAL_SLIDING, s, num_global=2, window=3, base_causal=1)
    q, do = _rand((1, s, hq, d), rng), _rand((1, s, hq, d), rng)
    k, v = _rand((1, s, hkv, d), rng), _rand((1, s, hkv, d), rng)
    sc = 0.9

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd_ref(q_, k_, v_, desc, scale=sc)
        return float((o * do).sum())

    r = oracle.attn_bwd_ref(q, k, v, do, desc, scale=sc)
    eps = 1e-6
    for name, x in (("dQ", q), ("dK", k), ("dV", v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy()
            xm = x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"dQ": (xp, k, v), "dK": (q, xp, v), "dV": (q, k, xp)}[name]
            args_m = {"dQ": (xm, k, v), "dK": (q, xm, v), "dV": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(r[name], num, atol=1e-7, rtol=1e-6)


def test_rows_sum_to_one_and_d_equals_do_dot_o():
    rng = np.random.default_rng(3)
    s, d = 40, 8
    for desc in _small_descs(16)[:6]:
        desc = I.MaskDesc(desc.type, s, window=desc.window, num_global=desc.num_global,
                          base_causal=desc.base_causal,
                          cu_seqlens=None if desc.cu_seqlens is None else np.array([0, 9, 10, 31, s], np.int32))
        q, k = _rand((1, s, 2, d), rng), _rand((1, s, 2, d), rng)
        ones = np.ones((1, s, 2, d))
        o, _ = oracle.attn_fwd_ref(q, k, ones, desc)
        np.testing.assert_allclose(o, 1.0, atol=1e-13)
        v, do = _rand((1, s, 2, d), rng), _rand((1, s, 2, d), rng)
        r = oracle.attn_bwd_ref(q, k, v, do, desc)
        np.testing.assert_allclose(r["D"], np.einsum("bshd,bshd->bhs", do, r["O"]), atol=1e-12)


def test_documents_are_independent_attentions():
    rng = np.random.default_rng(5)
    cu = np.array([0, 7, 8, 20, 33], np.int32)
    s, d = 33, 6
    q, k, v, do = (_rand((1, s, 2, d), rng) for _ in range(4))
    for packed_type, piece_type in ((I.FULL_DOCUMENT, I.FULL), (I.CAUSAL_DOCUMENT, I.CAUSAL)):
        r = oracle.attn_bwd_ref(q, k, v, do, I.MaskDesc(packed_type, s, cu_seqlens=cu))
        for a, b in zip(cu[:-1], cu[1:]):
            sl = slice(a, b)
            rp = oracle.attn_bwd_ref(q[:, sl], k[:, sl], v[:, sl], do[:, sl],
                                     I.MaskDesc(piece_type, int(b - a)))
            for key in ("O", "dQ", "dK", "dV"):
                np.testing.assert_allclose(r[key][:, sl], rp[key], atol=1e-12)
            np.testing.assert_allclose(r["LSE"][:, :, sl], rp["LSE"], atol=1e-12)


def test_library_sdpa_witness():
    rng = np.random.default_rng(9)
    s, d, hq = 48, 16, 2
    cu = np.array([0, 20, 21, 48], np.int32)
    for desc in [I.MaskDesc(I.FULL, s), I.MaskDesc(I.CAUSAL, s),
                 I.MaskDesc(I.PREFIX_LM, s, prefix_len=12),
                 I.MaskDesc(I.SHARED_QUESTION, s, cu_seqlens=cu),
                 I.MaskDesc(I.CAUSAL_BLOCKWISE, s, block=10),
                 I.MaskDesc(I.BLOCK_CAUSAL_DOCUMENT, s, block=6, cu_seqlens=cu)]:
        q, k, v = (_rand((1, s, hq, d), rng) for _ in range(3))
        o, _ = oracle.attn_fwd_ref(q, k, v, desc)
        m = torch.from_numpy(np.array(oracle.materialize_mask(desc)))
        tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m)
        np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)
        if desc.type == I.CAUSAL:
            ref2 = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
            np.testing.assert_allclose(o, ref2.permute(0, 2, 1, 3).numpy(), atol=1e-12)


def test_gqa_equals_replicated_mha():
    rng = np.random.default_rng(11)
    s, d, hq, hkv = 20, 4, 6, 2
    g = hq // hkv
    desc = I.MaskDesc(I.SLIDING_WINDOW, s, window=5)
    q, do = _rand((1, s, hq, d), rng), _rand((1, s, hq, d), rng)
    k, v = _rand((1, s, hkv, d), rng), _rand((1, s, hkv, d), rng)
    r = oracle.attn_bwd_ref(q, k, v, do, desc)
    kr, vr = np.repeat(k, g, axis=2), np.repeat(v, g, axis=2)
    rm = oracle.attn_bwd_ref(q, kr, vr, do, desc)
    np.testing.assert_allclose(r["O"], rm["O"], atol=1e-13)
    np.testing.assert_allclose(r["dQ"], rm["dQ"], atol=1e-13)
    np.testing.assert_allclose(r["dK"], rm["dK"].reshape(1, s, hkv, g, d).sum(3), atol=1e-12)
    np.testing.assert_allclose(r["dV"], rm["dV"].reshape(1, s, hkv, g, d).sum(3), atol=1e-12)


def test_row_functions_match_full():
    rng = np.random.default_rng(13)
    s, d, hq, hkv = 50, 8, 4, 2
    bm = I.uniform_block_map(s, 8, hkv, 0.5, 1)
    desc = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=8, map_heads=hkv, n_row_blocks=bm.shape[1],
                      n_col_blocks=bm.shape[2], block_map=bm)
    q, do = _rand((2, s, hq, d), rng), _rand((2, s, hq, d), rng)
    k, v = _rand((2, s, hkv, d), rng), _rand((2, s, hkv, d), rng)
    r = oracle.attn_bwd_ref(q, k, v, do, desc)
    rows = [0, 7, 8, 31, 49]
    heads = [1, 3]
    dq, o, lse, dd = oracle.attn_dq_rows_ref(q, k, v, do, desc, heads=heads, rows=rows, batch=1)
    o2, lse2 = oracle.attn_fwd_rows_ref(q, k, v, desc, heads=heads, rows=rows, batch=1)
    for a, h in enumerate(heads):
        np.testing.assert_allclose(dq[a], r["dQ"][1, rows, h], atol=1e-13)
        np.testing.assert_allclose(o[a], r["O"][1, rows, h], atol=1e-13)
        np.testing.assert_allclose(o2[a], r["O"][1, rows, h], atol=1e-13)
        np.testing.assert_allclose(lse2[a], r["LSE"][1, h, rows], atol=1e-13)
        np.testing.assert_allclose(dd[a], r["D"][1, h, rows], atol=1e-13)


def test_row_range_restriction_is_a_slice_of_the_full_result():
    rng = np.random.default_rng(17)
    s, d = 40, 4
    desc = I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=np.array([0, 13, 40], np.int32))
    q, k, v, do = (_rand((1, s, 2, d), rng) for _ in range(4))
    full = oracle.attn_bwd_ref(q, k, v, do, desc, chunk=7)
    parts = [oracle.attn_bwd_ref(q, k, v, do, desc, chunk=7, row_range=r) for r in ((0, 17), (17, 40))]
    np.testing.assert_allclose(parts[0]["dQ"][:, :17] + parts[1]["dQ"][:, :17], full["dQ"][:, :17],
                               atol=1e-13)
    np.testing.assert_allclose(parts[0]["dK"] + parts[1]["dK"], full["dK"], atol=1e-13)
    np.testing.assert_allclose(parts[0]["dV"] + parts[1]["dV"], full["dV"], atol=1e-13)


def test_key_column_function_matches_finite_differences():
    """dK/dV at selected keys equal the numerical gradient of L = sum(O * dO) with
    respect to those key and value rows (independent of attn_bwd_ref)."""
    rng = np.random.default_rng(23)
    s, d, hq, hkv = 12, 3, 4, 2
    desc = I.MaskDesc(I.CAUSAL_DOCUMENT, s, cu_seqlens=np.array([0, 5, 12], np.int32))
    q, do = _rand((1, s, hq, d), rng), _rand((1, s, hq, d), rng)
    k, v = _rand((1, s, hkv, d), rng), _rand((1, s, hkv, d), rng)
    sc = 0.7
    cols, kv_heads = [0, 4, 5, 11], [1, 0]
    dk, dv = oracle.attn_dkdv_cols_ref(q, k, v, do, desc, kv_heads=kv_heads, cols=cols, scale=sc)

    def loss(k_, v_):
        o, _ = oracle.attn_fwd_ref(q, k_, v_, desc, scale=sc)
        return float((o * do).sum())

    eps = 1e-6
    for a, hk in enumerate(kv_heads):
        for c, j in enumerate(cols):
            for x in range(d):
                for name, got in (("k", dk), ("v", dv)):
                    kp, km, vp, vm = k.copy(), k.copy(), v.copy(), v.copy()
                    if name == "k":
                        kp[0, j, hk, x] += eps
                        km[0, j, hk, x] -= eps
                    else:
                        vp[0, j, hk, x] += eps
                        vm[0, j, hk, x] -= eps
                    num = (loss(kp, vp) - loss(km, vm)) / (2 * eps)
                    assert abs(got[a, c, x] - num) <= 1e-7 + 1e-6 * abs(num), (name, hk, j, x)


@pytest.mark.parametrize("mask", [I.FULL, I.SLIDING_WINDOW, I.SHARED_QUESTION,
                                  I.BLOCK_SPARSE_UNIFORM, I.BLOCK_SPARSE_VARIABLE])
def test_key_column_function_matches_full_backward(mask):
    """Restricting the backward to the rows that reach the selected keys changes
    nothing: every mask type, GQA with per-query-head maps, unreachable keys give 0."""
    rng = np.random.default_rng(29 + mask)
    s, d, hq, hkv = 90, 5, 4, 2
    if mask == I.BLOCK_SPARSE_UNIFORM:
        bm = I.uniform_block_map(s, 16, hq, 0.5, 3)
        bm[:, :, 2] = 0                      # key block 2 is never attended
        desc = I.MaskDesc(mask, s, block=16, map_heads=hq, n_row_blocks=bm.shape[1],
                          n_col_blocks=bm.shape[2], block_map=bm)
    elif mask == I.SHARED_QUESTION:
        desc = I.make_desc(mask, s, question=20, answers=[30, 40])
    else:
        desc = I.make_desc(mask, s, window=17, map_heads=hkv, map_seed=5, doc_seed=5)
    q, do = _rand((1, s, hq, d), rng), _rand((1, s, hq, d), rng)
    k, v = _rand((1, s, hkv, d), rng), _rand((1, s, hkv, d), rng)
    full = oracle.attn_bwd_ref(q, k, v, do, desc, chunk=31)
    cols = [0, 1, 33, 34, 35, 60, 89]
    dk, dv = oracle.attn_dkdv_cols_ref(q, k, v, do, desc, kv_heads=[0, 1], cols=cols, chunk=13)
    for a in range(2):
        np.testing.assert_allclose(dk[a], full["dK"][0, cols, a], atol=1e-12)
        np.testing.assert_allclose(dv[a], full["dV"][0, cols, a], atol=1e-12)
    if mask == I.BLOCK_SPARSE_UNIFORM:
        assert (dk[:, 2:5] == 0).all() and (dv[:, 2:5] == 0).all()
    # restricted to one query head at a time, the contributions add up to the group's
    parts = [oracle.attn_dkdv_cols_ref(q, k, v, do, desc, kv_heads=[0, 1], cols=cols, heads=[h])
             for h in range(hq)]
    np.testing.assert_allclose(sum(p[0] for p in parts), dk, atol=1e-12)
    np.testing.assert_allclose(sum(p[1] for p in parts), dv, atol=1e-12)
