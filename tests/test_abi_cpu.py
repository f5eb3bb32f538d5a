"""The C-ABI library loads, exports every declared entry point and validates
arguments on the host before touching the GPU (runs without a GPU)."""
import ctypes
import os
import re

import pytest

from long_context_masked_gb300 import binding
from long_context_masked_gb300 import inputs as I
from long_context_masked_gb300 import build as lca_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.library_path()):
        lca_build.build()
    return binding.load_library()


def _declared():
    with open(os.path.join(ROOT, "include", "lca.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lca_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "lca_mask_build" in names and "lca_attn_fwd" in names and "lca_attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(7):
        assert lib.lca_status_string(code)
    assert lib.lca_status_string(99) == b"unknown status"


def _desc(**kw):
    c = binding.MaskDescC()
    c.type, c.seqlen = 1, 1024
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,tiles,expected", [
    ({}, (32, 128), 2),                                  # unsupported tile
    ({}, (128, 96), 2),
    ({"seqlen": 0}, (128, 128), 1),
    ({"seqlen": (1 << 20) + 1}, (128, 128), 2),
    ({"type": 13}, (128, 128), 1),
    ({"type": 12, "window": 0}, (128, 128), 1),         # window inside documents needs w >= 1
    ({"type": 12, "window": 8, "num_segments": 0}, (128, 128), 1),   # ... and documents
    ({"type": -1}, (128, 128), 1),
    ({"type": 2, "window": 0}, (128, 128), 1),          # sliding window needs w >= 1
    ({"type": 7, "window": 4, "num_global": -1}, (128, 128), 1),
    ({"type": 5, "prefix_len": 1025}, (128, 128), 1),
    ({"type": 8, "block": 0}, (128, 128), 1),
    ({"type": 3, "num_segments": 0}, (128, 128), 1),    # documents need cu_seqlens
    ({"type": 6, "num_segments": 2}, (128, 128), 1),    # ... and a pointer
    ({"type": 10, "block": 64, "map_heads": 1, "n_row_blocks": 16, "n_col_blocks": 16,
      "block_map": 0}, (128, 128), 1),                   # map pointer missing
    ({"type": 10, "block": 64, "map_heads": 1, "n_row_blocks": 15, "n_col_blocks": 16,
      "block_map": 16}, (128, 128), 1),                  # map size does not match S / block
    ({"type": 11, "map_heads": 1, "n_row_blocks": 4, "n_col_blocks": 4, "block_map": 16},
     (128, 128), 1),                                     # variable map without offsets
])
def test_mask_build_rejects_bad_descriptors(lib, kw, tiles, expected):
    out = ctypes.c_void_p(123)
    st = lib.lca_mask_build(ctypes.byref(_desc(**kw)), tiles[0], tiles[1], None, ctypes.byref(out))
    assert st == expected
    assert out.value is None


def test_null_arguments(lib):
    assert lib.lca_mask_build(None, 128, 128, None, ctypes.byref(ctypes.c_void_p())) == 1
    assert lib.lca_mask_build(ctypes.byref(_desc()), 128, 128, None, None) == 1
    sh = binding.ShapeC(1, 1024, 4, 4, 128, 512, 512, 512, 512)
    assert lib.lca_attn_fwd(None, ctypes.byref(sh), 16, 16, 16, 16, 16, 0.0, None) == 1
    assert lib.lca_attn_bwd(None, ctypes.byref(sh), *([16] * 10), 1 << 20, 0.0, 0, None) == 1
    assert lib.lca_attn_bwd_workspace(None, ctypes.byref(sh), 0) == 0
    info = binding.PlanInfoC()
    assert lib.lca_plan_get_info(None, ctypes.byref(info)) == 1
    lib.lca_plan_destroy(None)


def test_block_map_entry_points_validate_before_launch(lib):
    """Invalid shapes, sizes and pointers are rejected on the host (no GPU needed)."""
    sh = binding.ShapeC(1, 1000, 8, 2, 128, 8 * 128, 2 * 128, 2 * 128, 8 * 128)
    assert lib.lca_block_scores_workspace(ctypes.byref(sh), 64, 2) == 2 * 2 * 16 * 128 * 4
    assert lib.lca_block_scores_workspace(ctypes.byref(sh), 0, 2) == 0
    p, ws = 256, 1 << 20
    ok = (ctypes.byref(sh), p, p, 64, 2, 0.0, p, p, ws, None)
    for i, bad in [(3, 0), (3, 1001), (4, 3), (6, 0), (7, 0), (8, 16)]:
        args = list(ok)
        args[i] = bad
        assert lib.lca_block_scores(*args) == 1, (i, bad)
    sh2 = binding.ShapeC(2, 1000, 8, 2, 128, 8 * 128, 2 * 128, 2 * 128, 8 * 128)   # batch 2
    assert lib.lca_block_scores(ctypes.byref(sh2), *ok[1:]) == 1
    sh3 = binding.ShapeC(1, 1000, 8, 2, 64, 8 * 64, 2 * 64, 2 * 64, 8 * 64)        # head_dim 64
    assert lib.lca_block_scores(ctypes.byref(sh3), *ok[1:]) == 1
    assert lib.lca_block_topk(p, 2, 3, 10, 0, p, None) == 1
    assert lib.lca_block_topk(p, 2, 3, 10, 11, p, None) == 1
    assert lib.lca_block_topk(None, 2, 3, 10, 4, p, None) == 1
    assert lib.lca_block_topk(p, 0, 3, 10, 4, p, None) == 1


def test_python_constants_match_the_header():
    """The binding's enum values are the header's (tile classes and empty-half flags,
    mask types)."""
    with open(os.path.join(ROOT, "include", "lca.h")) as f:
        hdr = f.read()
    vals = {m.group(1): int(m.group(2)) for m in re.finditer(r"\bLCA_([A-Z0-9_]+)\s*=\s*(\d+)", hdr)}
    for name in ("TILE_SKIP", "TILE_FULL", "TILE_PARTIAL", "TILE_CLASS_MASK",
                 "TILE_KEY_HALF0_EMPTY", "TILE_KEY_HALF1_EMPTY", "TILE_QUERY_HALF0_EMPTY",
                 "TILE_QUERY_HALF1_EMPTY"):
        assert getattr(I, name) == vals[name], name
    for t, name in I.MASK_NAMES.items():
        assert vals[name] == t, name


def test_shape_marshals_every_row_stride():
    """The binding passes each tensor's own row stride: slices of a packed QKV tensor for
    the inputs, separate buffers for the gradients (CPU tensors; no library call)."""
    import torch

    b, s, hq, hkv, d = 1, 10, 4, 2, 128
    qkv = torch.zeros((b, s, hq + 2 * hkv, d), dtype=torch.bfloat16)
    q, k, v = qkv[:, :, :hq], qkv[:, :, hq:hq + hkv], qkv[:, :, hq + hkv:]
    o = torch.zeros((b, s, hq, d), dtype=torch.bfloat16)
    do = torch.zeros((b, s, 2 * hq, d), dtype=torch.bfloat16)[:, :, hq:]
    dq, dk, dv = torch.zeros_like(o), torch.zeros((b, s, hkv, d)).bfloat16(), \
        torch.zeros((b, s, 3 * hkv, d), dtype=torch.bfloat16)[:, :, :hkv]
    sh = binding._shape(q, k, v, o, do, dq, dk, dv)
    packed = (hq + 2 * hkv) * d
    assert (sh.q_row_stride, sh.k_row_stride, sh.v_row_stride) == (packed,) * 3
    assert sh.o_row_stride == hq * d and sh.do_row_stride == 2 * hq * d
    assert (sh.dq_row_stride, sh.dk_row_stride, sh.dv_row_stride) == (hq * d, hkv * d, 3 * hkv * d)
    fwd = binding._shape(q, k, v, o)          # the forward leaves the gradient strides 0
    assert (fwd.do_row_stride, fwd.dq_row_stride, fwd.dk_row_stride, fwd.dv_row_stride) == (0,) * 4
    with pytest.raises(binding.LcaError):     # heads not packed at stride d
        binding._shape(q, k, v, o, do, dq, dk, torch.zeros((b, s, hkv, 2 * d))[..., ::2])
    with pytest.raises(binding.LcaError):     # wrong head count
        binding._shape(q, k, v, o, do, dq, dk, torch.zeros((b, s, hkv + 1, d)))
