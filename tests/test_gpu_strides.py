"""Row strides of every tensor (packed QKV inputs, strided gradient buffers) through the
C ABI: results against the fp64 oracle, and host-side rejection of bad strides."""
import ctypes

import numpy as np
import pytest
import torch

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import binding
from long_context_masked_gb300 import inputs as I
from tests._gpu import check_grad, check_lse, check_o, make_inputs, to_np

pytestmark = pytest.mark.gpu


def _packed(parts, dim=2):
    """One contiguous [B, S, sum(heads), d] tensor holding `parts` side by side, and
    the views of it at the parts' places (row stride = sum(heads) * d)."""
    big = torch.cat(parts, dim=dim).contiguous()
    views, h0 = [], 0
    for p in parts:
        views.append(big[:, :, h0:h0 + p.shape[2]])
        h0 += p.shape[2]
    return big, views


@pytest.mark.parametrize("mask", [I.CAUSAL, I.SLIDING_WINDOW_DOCUMENT])
def test_packed_qkv_inputs_and_gradients(mask):
    s, hq, hkv = 700, 8, 2
    host, dev = make_inputs(1, s, hq, hkv, seed=90 + mask)
    q, k, v, do = dev
    _, (qp, kp, vp) = _packed([q, k, v])                 # row stride (hq + 2 hkv) * d
    _, (dop, _) = _packed([do, torch.zeros_like(do)])    # dO with row stride 2 hq d
    desc = I.make_desc(mask, s, window=150, doc_seed=5)
    plan = lca.mask_build(desc)
    o, lse = lca.attn_fwd(plan, qp, kp, vp)
    ref = oracle.attn_bwd_ref(*host, desc)
    check_o(to_np(o), ref["O"], "packed O")
    check_lse(to_np(lse), ref["LSE"], "packed LSE")
    # gradients into a packed dQKV buffer (sentinels around every slice) ...
    sentinel = 7.0
    big = torch.full((1, s, hq + 2 * hkv + 1, 128), sentinel, dtype=torch.bfloat16,
                     device="cuda")
    dq, dk, dv = big[:, :, :hq], big[:, :, hq:hq + hkv], big[:, :, hq + hkv:hq + 2 * hkv]
    lca.attn_bwd(plan, qp, kp, vp, o, dop, lse, dq=dq, dk=dk, dv=dv)
    # ... and into separate contiguous buffers from the same strided inputs
    g2 = lca.attn_bwd(plan, qp, kp, vp, o, dop, lse)
    assert lca.last_device_error() == 0
    assert (to_np(big[:, :, -1]) == sentinel).all()       # the head past dV untouched
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), g2):
        check_grad(to_np(a), ref[name], f"packed {name}")
        assert torch.equal(a, b), name


def test_backward_rejects_bad_gradient_strides():
    s, hq, hkv = 256, 4, 2
    _, dev = make_inputs(1, s, hq, hkv, seed=3)
    q, k, v, do = dev
    plan = lca.mask_build(I.make_desc(I.CAUSAL, s))
    o, lse = lca.attn_fwd(plan, q, k, v)
    lib = binding.load_library()
    ws = torch.empty(2 * hq * 256, dtype=torch.float32, device="cuda")
    out = [torch.empty_like(x) for x in (q, k, v)]
    base = binding._shape(q, k, v, o, do, *out)
    for field, bad in (("do_row_stride", hq * 128 - 8), ("dq_row_stride", hq * 128 + 4),
                       ("dk_row_stride", hkv * 128 - 8), ("dv_row_stride", 12)):
        sh = binding.ShapeC.from_buffer_copy(base)
        setattr(sh, field, bad)
        st = lib.lca_attn_bwd(plan.handle, ctypes.byref(sh), q.data_ptr(), k.data_ptr(),
                              v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                              out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(),
                              ws.data_ptr(), ws.numel() * 4, 0.0, 0, None)
        assert st == 1, field                              # LCA_ERR_INVALID_ARG, no launch
    assert lca.last_device_error() == 0
