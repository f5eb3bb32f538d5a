"""Whole query tiles and key tiles without any allowed pair, among more units than the GPU
has SMs: the persistent forward hands each CTA several units of different lengths, empty
ones included, and the backward's dQ and dK/dV CTAs meet empty lists too.  Results must
match the fp64 oracle, with exact zeros where nothing is attended."""
import numpy as np
import pytest

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import inputs as I
from tests._gpu import check_grad, check_lse, check_o, make_inputs, to_np

pytestmark = pytest.mark.gpu


def test_empty_tiles_among_many_units():
    # block maps take batch 1 (documents and maps are per sequence); 10 query tiles x 64
    # query heads = 640 units
    s, blk, b, hq, hkv = 1280, 64, 1, 64, 8
    nb = s // blk
    rng = np.random.default_rng(17)
    bm = (rng.random((1, nb, nb)) < 0.55).astype(np.uint8)   # lists of varying length
    bm[0, 4:6, :] = 0        # query tile 2 (rows 256..383): no allowed key
    bm[0, 14:16, :] = 0      # query tile 7 (rows 896..1023)
    bm[0, :, 10:12] = 0      # key tile 5 (keys 640..767): never attended
    desc = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=blk, block_map=bm, n_row_blocks=nb,
                      n_col_blocks=nb)
    host, dev = make_inputs(b, s, hq, hkv, seed=23)
    plan = lca.mask_build(desc, 128, 128)
    q, k, v, do = dev
    o, lse = lca.attn_fwd(plan, q, k, v)
    dq, dk, dv = lca.attn_bwd(plan, q, k, v, o, do, lse)
    assert lca.last_device_error() == 0

    o_np, lse_np = to_np(o), to_np(lse)
    for r0 in (256, 896):
        assert (o_np[:, r0:r0 + 128] == 0).all()
        assert np.isneginf(lse_np[:, :, r0:r0 + 128]).all()
        assert (to_np(dq)[:, r0:r0 + 128] == 0).all()
    assert (to_np(dk)[:, 640:768] == 0).all() and (to_np(dv)[:, 640:768] == 0).all()

    o_ref, lse_ref = oracle.attn_fwd_ref(*host[:3], desc)
    check_o(o_np, o_ref)
    check_lse(lse_np, lse_ref)
    ref = oracle.attn_bwd_ref(*host, desc)
    for name, g in zip(("dQ", "dK", "dV"), (dq, dk, dv)):
        check_grad(to_np(g), ref[name], name)
