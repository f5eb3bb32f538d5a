"""Parsers for the text fixtures under tests/golden/."""
import os

import numpy as np

from long_context_masked_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

_TYPES = {v: k for k, v in I.MASK_NAMES.items()}


def _ints(text):
    return np.array([int(x) for x in text.split(",")], dtype=np.int64)


def _matrix(text):
    return np.array([[int(x) for x in row.split(",")] for row in text.split(";")])


def load_mask_cases():
    """List of (name, MaskDesc, expected bool mask) from masks_small.txt."""
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, "masks_small.txt")) as f:
        lines = [ln.rstrip("\n") for ln in f]
    k = 0
    while k < len(lines):
        ln = lines[k].strip()
        k += 1
        if not ln or ln.startswith("#"):
            continue
        if ln.startswith("["):
            cur = {"name": ln.strip("[]")}
            continue
        key, _, val = [x.strip() for x in ln.partition("=")]
        if key == "mask":
            s = int(cur["seqlen"])
            rows = [lines[k + r].strip() for r in range(s)]
            k += s
            m = np.array([[c == "1" for c in row] for row in rows], dtype=bool)
            cases.append((cur["name"], _desc_from(cur), m))
        else:
            cur[key] = val
    return cases


def _desc_from(kv):
    t = _TYPES[kv["type"]]
    d = I.MaskDesc(t, int(kv["seqlen"]))
    for key in ("window", "num_global", "prefix_len", "block", "base_causal"):
        if key in kv:
            setattr(d, key, int(kv[key]))
    if "cu_seqlens" in kv:
        d.cu_seqlens = _ints(kv["cu_seqlens"]).astype(np.int32)
    if "block_map" in kv:
        bm = _matrix(kv["block_map"]).astype(np.uint8)
        d.block_map = bm[None]
        d.map_heads = 1
        d.n_row_blocks, d.n_col_blocks = bm.shape
    if "row_offsets" in kv:
        d.row_offsets = _ints(kv["row_offsets"]).astype(np.int32)[None]
        d.col_offsets = _ints(kv["col_offsets"]).astype(np.int32)[None]
    return d


def load_plan_case(name="plan_small.txt"):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if not ln or ln.startswith("#"):
                continue
            key, _, val = [x.strip() for x in ln.partition("=")]
            kv[key] = val
    desc = _desc_from(kv)
    exp = {k: _ints(kv[k]) for k in ("rowptr", "kt_idx", "kt_cls", "colptr", "qt_idx",
                                      "qt_cls", "work_q", "work_k")}
    exp["cls"] = _matrix(kv["cls"])[None]
    return desc, int(kv["tile_q"]), int(kv["tile_k"]), exp


def load_attention_closed_form():
    import math  # noqa: F401  (used by eval of the fixture's expressions)
    out = []
    with open(os.path.join(GOLDEN, "attention_closed_form.txt")) as f:
        for ln in f:
            ln = ln.strip()
            if not ln or ln.startswith("#"):
                continue
            case, qty, idx, expr = ln.split(None, 3)
            out.append((case, qty, int(idx), float(eval(expr, {"math": math}))))
    return out


def load_blockmap_cases():
    """Sections of blockmap_small.txt as {name: {key: value text}}."""
    out, cur = {}, None
    with open(os.path.join(GOLDEN, "blockmap_small.txt")) as f:
        for ln in f:
            ln = ln.strip()
            if not ln or ln.startswith("#"):
                continue
            if ln.startswith("["):
                cur = out.setdefault(ln.strip("[]"), {})
                continue
            key, _, val = [x.strip() for x in ln.partition("=")]
            cur[key] = val
    return out


def float_matrix(text):
    return np.array([[float(x) for x in row.split(",")] for row in text.split(";")])
