"""lca_attn_bwd_noalloc, the backward for callers that cannot allocate device memory
while it runs (pooled allocators that forbid side allocations, runtimes that only hand
out the op's own tensors, programs that reserve all device memory up front).  Through the C ABI it must give the results
of lca_attn_bwd and of the fp64 oracle, on consecutive calls that share its built-in
workspace.

This file is collected last so that a failure here never hides another test."""
import ctypes

import pytest
import torch

import long_context_masked_gb300 as lca
import oracle
from long_context_masked_gb300 import binding
from long_context_masked_gb300 import inputs as I
from tests._gpu import GRAD_REL_FRO, check_grad, make_inputs, rel_fro, to_np

pytestmark = pytest.mark.gpu


def test_noalloc_backward_matches_allocating_backward_and_oracle_twice():
    # two calls in a row on the shared built-in buffer: the larger shape first, so stale
    # workspace rows from the first call would show in the second
    cases = [(1408, 8, 2, I.CAUSAL_DOCUMENT, 77), (600, 4, 1, I.SLIDING_WINDOW, 78)]
    runs = []
    for s, hq, hkv, mask, seed in cases:
        host, dev = make_inputs(1, s, hq, hkv, seed=seed)
        q, k, v, do = dev
        desc = I.make_desc(mask, s, window=200, doc_seed=3)
        plan = lca.mask_build(desc, 128, 128)
        o, lse = lca.attn_fwd(plan, q, k, v)
        ref = lca.attn_bwd(plan, q, k, v, o, do, lse)
        torch.cuda.synchronize()
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        runs.append((host, desc, plan, (q, k, v, o, do, lse), ref, out))
    for _, _, plan, (q, k, v, o, do, lse), _, (dq, dk, dv) in runs:
        lca.attn_bwd_noalloc(plan, q, k, v, o, do, lse, dq=dq, dk=dk, dv=dv)
    assert lca.last_device_error() == 0
    for host, desc, _, _, ref, got in runs:
        full = oracle.attn_bwd_ref(*host, desc)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert rel_fro(to_np(g), to_np(r)) <= GRAD_REL_FRO, name
            check_grad(to_np(g), full[name], f"noalloc {desc.name} {name}")


def test_noalloc_backward_rejects_shapes_beyond_its_buffer():
    lib = binding.load_library()
    s = 131073                      # 64 heads x 131200 padded rows > 2^23
    plan = lca.mask_build(I.make_desc(I.FULL, s), 128, 128)
    sh = binding.ShapeC(1, s, 64, 8, 128, 64 * 128, 8 * 128, 8 * 128, 64 * 128)
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    st = lib.lca_attn_bwd_noalloc(plan.handle, ctypes.byref(sh), p, p, p, p, p, p, p, p, p,
                                  0.0, None)
    assert st == 2                  # LCA_ERR_UNSUPPORTED, nothing launched
    assert lca.last_device_error() == 0
