"""Tensor-core operand layouts and the bounded device wait, through the C ABI."""
import numpy as np
import pytest
import torch

import long_context_masked_gb300 as lca

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_umma_operand_layouts(variant):
    g = torch.Generator().manual_seed(variant)
    a = torch.randn((128, 128), generator=g).to(torch.bfloat16)
    b = torch.randn((128, 128), generator=g).to(torch.bfloat16)
    c = lca.selftest_umma(variant, a.cuda(), b.cuda()).cpu().double().numpy()
    a64, b64 = a.double().numpy(), b.double().numpy()
    ref = {0: a64 @ b64.T, 1: a64 @ b64, 2: a64 @ b64, 3: a64.T @ b64, 4: a64 @ b64}[variant]
    assert np.abs(c - ref).max() < 1e-3


def test_bounded_wait_gives_up_and_reports_timeout():
    assert lca.selftest_wait_timeout(2_000_000) == 5      # LCA_ERR_TIMEOUT
    assert lca.last_device_error() == 0                   # the word was cleared
    torch.cuda.synchronize()                              # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
