"""Forward parity of the CUDA path with the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import inputs as I
from tests._gpu import check_lse, check_o, make_inputs, small_descs, to_np

pytestmark = pytest.mark.gpu


def _fwd(desc, dev, scale=None):
    plan = lca.mask_build(desc, 128, 128)
    q, k, v, _ = dev
    o, lse = lca.attn_fwd(plan, q, k, v, scale=scale)
    assert lca.last_device_error() == 0
    return to_np(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("mask", [I.FULL, I.CAUSAL])
def test_tiny_config_in_full(mask):
    # B=1, S=1024, H_q=H_kv=4, d=128, seed 0
    host, dev = make_inputs(1, 1024, 4, 4, seed=0)
    desc = I.make_desc(mask, 1024)
    o, lse = _fwd(desc, dev)
    o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc)
    check_o(o, o_ref, desc.name)
    check_lse(lse, lse_ref, desc.name)


@pytest.mark.parametrize("s", [1000, 1408])
def test_every_mask_type_gqa(s):
    hq, hkv = 8, 2
    host, dev = make_inputs(1, s, hq, hkv, seed=s)
    for desc in small_descs(s, hq, hkv, seed=s):
        o, lse = _fwd(desc, dev)
        o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc)
        check_o(o, o_ref, desc.name)
        check_lse(lse, lse_ref, desc.name)


def test_batched_and_scaled():
    host, dev = make_inputs(3, 300, 4, 1, seed=7)
    for mask in (I.FULL, I.CAUSAL, I.SLIDING_WINDOW, I.PREFIX_LM):
        desc = I.make_desc(mask, 300, window=50)
        o, lse = _fwd(desc, dev, scale=0.05)
        o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc, scale=0.05)
        check_o(o, o_ref, desc.name)
        check_lse(lse, lse_ref, desc.name)


def test_empty_rows_and_tiny_sequences():
    s = 640
    bm = np.ones((1, 10, 10), np.uint8)
    bm[0, 3, :] = 0          # query rows 192..255 see nothing
    desc = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=64, block_map=bm, n_row_blocks=10,
                      n_col_blocks=10)
    host, dev = make_inputs(1, s, 2, 2, seed=3)
    o, lse = _fwd(desc, dev)
    o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc)
    assert (o[0, 192:256] == 0).all() and np.isinf(lse[0, :, 192:256]).all()
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    for s in (1, 5, 129):
        host, dev = make_inputs(1, s, 2, 1, seed=s)
        for mask in (I.FULL, I.CAUSAL):
            desc = I.make_desc(mask, s)
            o, lse = _fwd(desc, dev)
            o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc)
            check_o(o, o_ref)
            check_lse(lse, lse_ref)


def test_large_logits_rescale_path():
    # scores with a large spread force the running-max rescale of the accumulator
    s = 1024
    host, dev = make_inputs(1, s, 2, 2, seed=11)
    q, k, v, do = dev
    ramp = torch.linspace(0.2, 6.0, s, device="cuda").view(1, s, 1, 1)
    k2 = (k.float() * ramp).to(torch.bfloat16)
    host2 = [host[0], to_np(k2), host[2]]
    desc = I.make_desc(I.CAUSAL, s)
    plan = lca.mask_build(desc, 128, 128)
    o, lse = lca.attn_fwd(plan, q, k2, v)
    o_ref, lse_ref = oracle.attn_fwd_ref(*host2, desc)
    check_o(to_np(o), o_ref)
    check_lse(lse.cpu().numpy(), lse_ref)


def _sampled(desc, b, s, hq, hkv, heads, nrows, seed):
    host, dev = make_inputs(b, s, hq, hkv, seed=seed)
    o, lse = _fwd(desc, dev)
    rng = np.random.default_rng(seed)
    rows = np.sort(np.concatenate([rng.choice(s, nrows - 2, replace=False), [0, s - 1]]))
    o_ref, lse_ref = oracle.attn_fwd_rows_ref(*host[:3], desc, heads=heads, rows=rows)
    for a, h in enumerate(heads):
        check_o(o[0, rows, h], o_ref[a], f"{desc.name} h{h}")
        check_lse(lse[0, h, rows], lse_ref[a], f"{desc.name} h{h}")


@pytest.mark.parametrize("mask,kw", [(I.FULL, {}), (I.CAUSAL, {}),
                                     (I.SLIDING_WINDOW, {"window": 4096}),
                                     (I.FULL_DOCUMENT, {"doc_seed": 1}),
                                     (I.CAUSAL_DOCUMENT, {"doc_seed": 1}),
                                     (I.SLIDING_WINDOW_DOCUMENT, {"window": 1024, "doc_seed": 2})])
def test_dense_regular_full_size_sampled(mask, kw):
    s = 16384
    desc = I.make_desc(mask, s, **kw)
    _sampled(desc, 1, s, 64, 8, heads=[0, 9, 63], nrows=48, seed=100 + mask)


@pytest.mark.parametrize("mask,kw", [(I.PREFIX_LM, {}),
                                     (I.SHARED_QUESTION, {"question": 2048, "answers": [7680] * 4}),
                                     (I.GLOBAL_SLIDING, {"num_global": 256, "window": 4096}),
                                     (I.CAUSAL_BLOCKWISE, {"block": 2048}),
                                     (I.BLOCK_CAUSAL_DOCUMENT, {"block": 2048, "doc_seed": 2}),
                                     # the pages' block of 1024
                                     (I.BLOCK_CAUSAL_DOCUMENT, {"block": 1024, "doc_seed": 3})])
def test_heterogeneous_full_size_sampled(mask, kw):
    s = 32768
    desc = I.make_desc(mask, s, **kw)
    _sampled(desc, 1, s, 64, 64, heads=[0, 31, 63], nrows=40, seed=200 + mask)


@pytest.mark.parametrize("s,block,hq,hkv,sparsity", [(131072, 64, 64, 8, 0.5), (65536, 128, 32, 32, 0.8),
                                                     (32768, 64, 32, 32, 0.2)])
def test_uniform_block_sparse_full_size_sampled(s, block, hq, hkv, sparsity):
    map_heads = hkv if hq != hkv else hq
    desc = I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=block, sparsity=sparsity,
                       map_heads=map_heads, map_seed=block)
    _sampled(desc, 1, s, hq, hkv, heads=[0, hq - 1], nrows=24, seed=s + block)


def test_variable_block_sparse_long_varlen_sampled():
    s = 131072
    desc = I.make_desc(I.BLOCK_SPARSE_VARIABLE, s, map_heads=8, map_seed=7, doc_seed=7)
    _sampled(desc, 1, s, 64, 8, heads=[0, 37], nrows=24, seed=99)


@pytest.mark.parametrize("hq,hkv,b", [(8, 2, 1), (4, 4, 1), (4, 2, 2)])
def test_head_dim_64(hq, hkv, b):
    """head_dim 64: every mask type (one sequence), or the batched dense masks."""
    s = 1000
    host, dev = make_inputs(b, s, hq, hkv, seed=64 + hq, head_dim=64)
    descs = small_descs(s, hq, hkv, seed=6) if b == 1 else \
        [I.make_desc(m, s, window=120) for m in (I.FULL, I.CAUSAL, I.SLIDING_WINDOW)]
    for desc in descs:
        o, lse = _fwd(desc, dev)
        o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc)
        check_o(o, o_ref, f"d64 {desc.name}")
        check_lse(lse, lse_ref, f"d64 {desc.name}")


def test_concurrent_forwards_share_a_plan():
    """The persistent forward takes its units from a counter of the plan; calls on two
    streams that share one plan each get their own counter and give the results of the
    calls run one after the other (bit-identical: a unit is computed by one CTA)."""
    s, hq, hkv = 4096, 16, 2
    host, dev = make_inputs(1, s, hq, hkv, seed=88)
    q, k, v, _ = dev
    plan = lca.mask_build(I.make_desc(I.CAUSAL_DOCUMENT, s, doc_seed=8))
    ref = [lca.attn_fwd(plan, q, k, v) for _ in range(2)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = []
    for st in streams:
        with torch.cuda.stream(st):
            outs.append(lca.attn_fwd(plan, q, k, v, stream=st))
    torch.cuda.synchronize()
    assert lca.last_device_error() == 0
    for (o, l), (o_ref, l_ref) in zip(outs, ref):
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
    o_ref_host, lse_ref_host = oracle.attn_fwd_ref(*host[:3], plan.desc)
    check_o(to_np(outs[1][0]), o_ref_host, "concurrent")
    check_lse(to_np(outs[1][1]), lse_ref_host, "concurrent")
