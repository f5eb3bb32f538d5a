"""Shared helpers of the GPU parity tests (inputs, tolerance checks)."""
import numpy as np
import torch

from long_context_masked_gb300 import inputs as I

# Tolerances of the parity bar (bf16 inputs, fp32 accumulation):
O_MAX_ABS = 1e-2         # forward output, max-abs
LSE_MAX_ABS = 1e-3       # logsumexp (natural log), max-abs over finite rows
GRAD_REL_FRO = 1e-2      # dQ / dK / dV, relative Frobenius error per tensor


def bf16_half_ulp(x):
    """Half a bf16 ulp of |x| (the rounding error bound of one bf16 output)."""
    ax = np.maximum(np.abs(x), 1e-30)
    e = np.floor(np.log2(ax))
    return 0.5 * np.exp2(e - 7)


def check_o(o_gpu, o_ref, what=""):
    """Strict max-abs 1e-2; violations are tolerated only where |O_ref| >= 2, where
    one bf16 rounding of the output alone exceeds 1e-2 (then error - half ulp <= 1e-2)."""
    o_gpu = np.asarray(o_gpu, np.float64)
    err = np.abs(o_gpu - o_ref)
    bad = err > O_MAX_ABS
    if bad.any():
        assert (np.abs(o_ref[bad]) >= 2).all(), f"{what}: O max-abs {err.max():.3e}"
        excess = (err - bf16_half_ulp(o_ref))[bad].max()
        assert excess <= O_MAX_ABS, f"{what}: O excess over half ulp {excess:.3e}"
    return float(err.max())


def check_lse(l_gpu, l_ref, what=""):
    l_gpu = np.asarray(l_gpu, np.float64)
    inf_ref = ~np.isfinite(l_ref)
    assert np.array_equal(~np.isfinite(l_gpu), inf_ref), f"{what}: empty-row pattern differs"
    if inf_ref.any():
        assert (l_gpu[inf_ref] < 0).all()
    fin = ~inf_ref
    err = np.abs(l_gpu[fin] - l_ref[fin]).max() if fin.any() else 0.0
    assert err <= LSE_MAX_ABS, f"{what}: LSE max-abs {err:.3e}"
    return float(err)


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def check_grad(g_gpu, g_ref, what=""):
    e = rel_fro(g_gpu, g_ref)
    assert e <= GRAD_REL_FRO, f"{what}: relative Frobenius {e:.3e}"
    return e


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def make_inputs(b, s, hq, hkv, seed, device="cuda", head_dim=128):
    q, k, v, do = I.qkv_do(b, s, hq, hkv, head_dim, seed)
    host = [to_np(x) for x in (q, k, v, do)]
    dev = [x.to(device) for x in (q, k, v, do)]
    return host, dev


def small_descs(s, hq, hkv, seed=0):
    """One descriptor of every mask type at sequence length s."""
    lens = I.lognormal_doc_lengths(s, seed, mu=np.log(max(64, s // 5)), lo=16)
    cu = I.cu_from_lengths(lens)
    q_len = max(1, s // 8)
    rest = s - q_len
    answers = [rest // 3, rest // 3, rest - 2 * (rest // 3)]
    out = [
        I.make_desc(I.FULL, s),
        I.make_desc(I.CAUSAL, s),
        I.make_desc(I.SLIDING_WINDOW, s, window=max(1, s // 5)),
        I.make_desc(I.FULL_DOCUMENT, s, cu_seqlens=cu),
        I.make_desc(I.CAUSAL_DOCUMENT, s, cu_seqlens=cu),
        I.make_desc(I.SLIDING_WINDOW_DOCUMENT, s, window=max(1, s // 9), cu_seqlens=cu),
        I.make_desc(I.PREFIX_LM, s),
        I.make_desc(I.SHARED_QUESTION, s, question=q_len, answers=answers),
        I.make_desc(I.GLOBAL_SLIDING, s, num_global=max(1, s // 20), window=max(1, s // 6)),
        I.make_desc(I.GLOBAL_SLIDING, s, num_global=max(1, s // 20), window=max(1, s // 6),
                    base_causal=0),
        I.make_desc(I.CAUSAL_BLOCKWISE, s, block=max(1, s // 6)),
        I.make_desc(I.BLOCK_CAUSAL_DOCUMENT, s, block=100, cu_seqlens=cu),
        I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64, sparsity=0.5, map_heads=hkv,
                    map_seed=seed),
        I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=128, sparsity=0.8, map_heads=hq,
                    map_seed=seed + 1),
        I.make_desc(I.BLOCK_SPARSE_VARIABLE, s, map_heads=hkv, map_seed=seed, cu_seqlens=cu),
    ]
    return out


def oracle_bwd_heads(host, desc, heads, scale=None, workers=8):
    """oracle.attn_bwd_ref over the given query heads, one head per worker thread (the
    NumPy work releases the GIL), with dK/dV summed over the heads.  Returns the same
    dict as attn_bwd_ref: dQ is filled for the given heads only, and dK/dV of a KV head
    are complete when all of its query heads are given."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    heads = list(heads)

    def one(h):
        return oracle.attn_bwd_ref(*host, desc, scale=scale, heads=[h])

    with ThreadPoolExecutor(max(1, min(workers, len(heads)))) as ex:
        parts = list(ex.map(one, heads))
    out = parts[0]
    for h, p in zip(heads[1:], parts[1:]):
        out["dQ"][:, :, h] = p["dQ"][:, :, h]
        out["O"][:, :, h] = p["O"][:, :, h]
        out["LSE"][:, h] = p["LSE"][:, h]
        out["D"][:, h] = p["D"][:, h]
        out["dK"] += p["dK"]
        out["dV"] += p["dV"]
    return out


def oracle_dkdv_cols(host, desc, kv_heads, cols, scale=None, workers=8):
    """oracle.attn_dkdv_cols_ref with one query head per worker thread; the heads'
    contributions are summed per KV head."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    g = host[0].shape[2] // host[1].shape[2]
    jobs = [(a, hk, h) for a, hk in enumerate(kv_heads) for h in range(hk * g, (hk + 1) * g)]

    def one(job):
        _, hk, h = job
        return oracle.attn_dkdv_cols_ref(*host, desc, kv_heads=[hk], cols=cols, scale=scale,
                                         heads=[h])

    with ThreadPoolExecutor(max(1, min(workers, len(jobs)))) as ex:
        parts = list(ex.map(one, jobs))
    d = host[1].shape[3]
    dk = np.zeros((len(kv_heads), len(cols), d))
    dv = np.zeros((len(kv_heads), len(cols), d))
    for (a, _, _), (pk, pv) in zip(jobs, parts):
        dk[a] += pk[0]
        dv[a] += pv[0]
    return dk, dv


def sampled_cols(s, n, seed):
    """n sorted key positions: the first and last, the rest drawn without repetition."""
    rng = np.random.default_rng(seed)
    return np.sort(np.concatenate([rng.choice(np.arange(1, s - 1), n - 2, replace=False),
                                   [0, s - 1]]))
