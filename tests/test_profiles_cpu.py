"""The ncu summaries under profiles/ describe the kernels as they are in the tree: every
source hash a summary records matches the current file, and the default workload's
roofline traffic is found for the current backward source (runs without a GPU)."""
import hashlib
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "long_context_masked_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


def _sha(name):
    with open(os.path.join(CSRC, name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def _summaries():
    return sorted(n for n in os.listdir(PROFILES) if n.endswith((".md", ".txt")))


def test_summaries_are_text_only():
    for n in os.listdir(PROFILES):
        assert n.endswith((".md", ".txt")), n


@pytest.mark.parametrize("name", _summaries())
def test_recorded_source_hashes_are_current(name):
    with open(os.path.join(PROFILES, name)) as f:
        text = f.read()
    # "`attn_fwd.cu` sha256 6c7e…" and the machine-readable "source_sha256=…" records
    found = re.findall(r"`(\w+\.cu)`\s+(?:sha256\s+)?([0-9a-f]{16,64})", text)
    for src, prefix in found:
        assert _sha(src).startswith(prefix), f"{name}: {src} changed since it was profiled"
    for prefix in re.findall(r"source_sha256=([0-9a-f]+)", text):
        assert _sha("attn_bwd.cu").startswith(prefix), f"{name}: attn_bwd.cu changed"


def test_default_roofline_traffic_is_found():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    t = bench.traffic_from_profiles("bwd", "bench_default")
    assert t is not None and t > 0
