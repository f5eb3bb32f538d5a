"""Exact masked softmax attention, forward and backward, in fp64 on the host.

Definition (the computation every kernel in the benchmark performs: standard
softmax attention with a mask [LongCA-bench summary, abstract and §4 "Attention
kernels"; reading note, "Key design" 2: the naive stepwise attention baseline]).
For batch b, query head h (KV head h // g, g = H_q / H_kv) and the mask M of
the head's map head:

    s_ij   = scale * <q_i, k_j>                 (scale defaults to 1/sqrt(d))
    LSE_i  = ln sum_{j: M_ij} exp(s_ij)         (natural log)
    P_ij   = M_ij * exp(s_ij - LSE_i)
    O_i    = sum_j P_ij v_j

and, given dO, the gradients of L = sum(O * dO):

    dV_j   = sum_i P_ij dO_i
    dP_ij  = <dO_i, v_j>
    D_i    = sum_j P_ij dP_ij
    dS_ij  = P_ij (dP_ij - D_i)
    dQ_i   = scale * sum_j dS_ij k_j
    dK_j   = scale * sum_i dS_ij q_i

dK and dV of a KV head sum over its g query heads.  A row with no allowed key
has O = 0, LSE = -inf, dQ = 0 and adds nothing to dK/dV (reading taken here:
the pages do not discuss empty rows).

Inputs are numpy arrays in the library's layouts, Q/O/dO ``[B, S, H_q, d]`` and
K/V ``[B, S, H_kv, d]``; they are upcast to fp64 (bf16 values are exact in
fp64).  Rows are processed in chunks of whole rows, which changes nothing in the
arithmetic of a row.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

from .masks import allowed, mask_rows, map_head_of


def _default_scale(d: int, scale: Optional[float]) -> float:
    return 1.0 / math.sqrt(d) if (scale is None or scale <= 0) else float(scale)


def _row_softmax(s: np.ndarray, m: np.ndarray):
    """LSE and P for a block of whole rows (s: scores, m: mask)."""
    masked = np.where(m, s, -np.inf)
    mx = masked.max(axis=1, keepdims=True)
    empty = ~np.isfinite(mx)
    mx_safe = np.where(empty, 0.0, mx)
    e = np.where(m, np.exp(masked - mx_safe), 0.0)
    tot = e.sum(axis=1, keepdims=True)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, mx_safe + np.log(np.where(empty, 1.0, tot)))
    p = np.where(m, np.exp(np.where(m, s, 0.0) - np.where(empty, 0.0, lse)), 0.0)
    return lse[:, 0], p


def attn_fwd_rows_ref(q, k, v, desc, *, heads: Sequence[int], rows: Sequence[int],
                      batch: int = 0, scale: Optional[float] = None):
    """O and LSE for selected query heads and rows of one batch entry.

    Returns ``(O [len(heads), len(rows), d], LSE [len(heads), len(rows)])``.
    """
    _, s_len, h_q, d = q.shape
    h_kv = k.shape[2]
    g = h_q // h_kv
    sc = _default_scale(d, scale)
    rows = np.asarray(rows, np.int64)
    o = np.zeros((len(heads), len(rows), d))
    lse = np.zeros((len(heads), len(rows)))
    for a, h in enumerate(heads):
        hm = map_head_of(h, h_q, h_kv, desc.map_heads)
        kk = np.asarray(k[batch, :, h // g, :], np.float64)
        vv = np.asarray(v[batch, :, h // g, :], np.float64)
        qq = np.asarray(q[batch, rows, h, :], np.float64)
        m = mask_rows(desc, hm, rows)
        s = sc * (qq @ kk.T)
        lse[a], p = _row_softmax(s, m)
        o[a] = p @ vv
    return o, lse


def attn_fwd_ref(q, k, v, desc, *, scale: Optional[float] = None, chunk: int = 2048):
    """Full forward: ``(O [B, S, H_q, d], LSE [B, H_q, S])`` in fp64."""
    b_n, s_len, h_q, d = q.shape
    o = np.zeros((b_n, s_len, h_q, d))
    lse = np.zeros((b_n, h_q, s_len))
    for b in range(b_n):
        for r0 in range(0, s_len, chunk):
            rows = np.arange(r0, min(s_len, r0 + chunk))
            oo, ll = attn_fwd_rows_ref(q, k, v, desc, heads=range(h_q), rows=rows,
                                       batch=b, scale=scale)
            o[b, rows] = np.transpose(oo, (1, 0, 2))
            lse[b, :, rows] = ll.T
    return o, lse


def attn_bwd_ref(q, k, v, do, desc, *, scale: Optional[float] = None, chunk: int = 2048,
                 heads: Optional[Sequence[int]] = None, row_range=None):
    """Forward plus analytic backward, fp64.

    Returns a dict with O, LSE, D, dQ, dK, dV in the library's layouts.  When
    ``heads`` is given only those query heads are processed (their dK/dV
    contributions still land on their KV heads); when ``row_range = (r0, r1)`` is
    given only those query rows are processed, so dK/dV hold just their
    contributions (used to time bounded samples).
    """
    b_n, s_len, h_q, d = q.shape
    h_kv = k.shape[2]
    g = h_q // h_kv
    sc = _default_scale(d, scale)
    heads = list(range(h_q)) if heads is None else list(heads)
    o = np.zeros((b_n, s_len, h_q, d))
    lse = np.zeros((b_n, h_q, s_len))
    dd = np.zeros((b_n, h_q, s_len))
    dq = np.zeros((b_n, s_len, h_q, d))
    dk = np.zeros((b_n, s_len, h_kv, d))
    dv = np.zeros((b_n, s_len, h_kv, d))
    for b in range(b_n):
        for h in heads:
            hk = h // g
            hm = map_head_of(h, h_q, h_kv, desc.map_heads)
            kk = np.asarray(k[b, :, hk, :], np.float64)
            vv = np.asarray(v[b, :, hk, :], np.float64)
            lo, hi = (0, s_len) if row_range is None else row_range
            for r0 in range(lo, hi, chunk):
                rows = np.arange(r0, min(hi, r0 + chunk))
                qq = np.asarray(q[b, rows, h, :], np.float64)
                gg = np.asarray(do[b, rows, h, :], np.float64)
                m = mask_rows(desc, hm, rows)
                s = sc * (qq @ kk.T)
                l_rows, p = _row_softmax(s, m)
                lse[b, h, rows] = l_rows
                o[b, rows, h] = p @ vv
                dp = gg @ vv.T
                d_rows = (p * dp).sum(axis=1)
                dd[b, h, rows] = d_rows
                ds = p * (dp - d_rows[:, None])
                dq[b, rows, h] = sc * (ds @ kk)
                dk[b, :, hk] += sc * (ds.T @ qq)
                dv[b, :, hk] += p.T @ gg
    return {"O": o, "LSE": lse, "D": dd, "dQ": dq, "dK": dk, "dV": dv}


def attn_dq_rows_ref(q, k, v, do, desc, *, heads: Sequence[int], rows: Sequence[int],
                     batch: int = 0, scale: Optional[float] = None):
    """dQ (and O, LSE, D) for selected heads and rows; every row is local.

    Returns ``(dQ [nh, nr, d], O [nh, nr, d], LSE [nh, nr], D [nh, nr])``.
    """
    _, s_len, h_q, d = q.shape
    h_kv = k.shape[2]
    g = h_q // h_kv
    sc = _default_scale(d, scale)
    rows = np.asarray(rows, np.int64)
    nh, nr = len(heads), len(rows)
    dq = np.zeros((nh, nr, d))
    o = np.zeros((nh, nr, d))
    lse = np.zeros((nh, nr))
    dd = np.zeros((nh, nr))
    for a, h in enumerate(heads):
        hm = map_head_of(h, h_q, h_kv, desc.map_heads)
        kk = np.asarray(k[batch, :, h // g, :], np.float64)
        vv = np.asarray(v[batch, :, h // g, :], np.float64)
        qq = np.asarray(q[batch, rows, h, :], np.float64)
        gg = np.asarray(do[batch, rows, h, :], np.float64)
        m = mask_rows(desc, hm, rows)
        s = sc * (qq @ kk.T)
        lse[a], p = _row_softmax(s, m)
        o[a] = p @ vv
        dp = gg @ vv.T
        dd[a] = (p * dp).sum(axis=1)
        dq[a] = sc * ((p * (dp - dd[a][:, None])) @ kk)
    return dq, o, lse, dd


def attn_dkdv_cols_ref(q, k, v, do, desc, *, kv_heads: Sequence[int], cols: Sequence[int],
                       batch: int = 0, scale: Optional[float] = None, chunk: int = 2048,
                       heads: Optional[Sequence[int]] = None):
    """dK and dV at selected key positions of selected KV heads, fp64.

    For key j of KV head hk, summed over the query heads h of its group:
    dV_j = sum_i P_ij dO_i and dK_j = scale * sum_i dS_ij q_i with
    dS_ij = P_ij (dP_ij - D_i).  P_ij and dS_ij vanish unless M_ij, so only the
    query rows that may attend at least one selected key are evaluated; each of
    those rows is evaluated over all keys (which gives its LSE_i and D_i).  This
    is the attn_bwd_ref arithmetic restricted to the rows and columns that reach
    the selected keys, for checks at sizes where the full backward is too slow.
    When ``heads`` is given, only those query heads contribute (each KV head then sums
    the given heads of its group).

    Returns ``(dK [len(kv_heads), len(cols), d], dV [len(kv_heads), len(cols), d])``.
    """
    _, s_len, h_q, d = q.shape
    h_kv = k.shape[2]
    g = h_q // h_kv
    sc = _default_scale(d, scale)
    cols = np.asarray(cols, np.int64)
    all_rows = np.arange(s_len, dtype=np.int64)
    dk = np.zeros((len(kv_heads), len(cols), d))
    dv = np.zeros((len(kv_heads), len(cols), d))
    for a, hk in enumerate(kv_heads):
        kk = np.asarray(k[batch, :, hk, :], np.float64)
        vv = np.asarray(v[batch, :, hk, :], np.float64)
        for h in range(hk * g, (hk + 1) * g):
            if heads is not None and h not in heads:
                continue
            hm = map_head_of(h, h_q, h_kv, desc.map_heads)
            reach = np.broadcast_to(allowed(desc, hm, all_rows[:, None], cols[None, :]),
                                    (s_len, len(cols)))
            rows = np.nonzero(reach.any(axis=1))[0]
            for r0 in range(0, len(rows), chunk):
                rr = rows[r0:r0 + chunk]
                qq = np.asarray(q[batch, rr, h, :], np.float64)
                gg = np.asarray(do[batch, rr, h, :], np.float64)
                m = mask_rows(desc, hm, rr)
                _, p = _row_softmax(sc * (qq @ kk.T), m)
                dp = gg @ vv.T
                d_rows = (p * dp).sum(axis=1)
                p_c = p[:, cols]
                ds_c = p_c * (dp[:, cols] - d_rows[:, None])
                dv[a] += p_c.T @ gg
                dk[a] += sc * (ds_c.T @ qq)
    return dk, dv
