#!/usr/bin/env python
"""Throughput of mask-aware exact softmax attention (mask build + forward + backward).

Metric: TFLOP/s on unmasked FLOPs - 4*d*H_q per allowed (i, j) pair forward and
2.5x that backward - per mask and sequence length, plus the fraction of the GB300
bf16 dense tensor peak.  The default workload is the benchmark's dense regular masks
(LongCA-bench, sections 2.1 and A.4: FULL, CAUSAL, sliding window, full/causal
document over lognormal-length documents) on GQA 64:8, d = 128, at S = 8K, 16K, 32K
and 48K.  One step runs, for every (S, mask): the tile plan build, the forward and the
backward, on synthetic N(0, 1) bf16 inputs resident on the GPU.  Document masks
re-draw their lengths every step (seed = step mod 30; the pages sample 30 runs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--suite dense|heterogeneous|sparse|varlen|dynamic] [--case S:MASK]
                    [--protocol steps|pages] [--no-memory]

``--suite`` selects another of the benchmark's workloads: the heterogeneous static
masks at S = 32K on MHA 64:64; uniform block-sparse maps (blocks 64/128, sparsity
0.2/0.5/0.8, S = 32K-128K, GQA 64:8 and MHA 32:32), reported per case with the
fraction of non-skipped tiles and the time per tile; or S = 128K documents with
variable block-sparse maps.  ``--impl reference`` times the fp64 CPU oracle (the only
reference available here) on a bounded row sample of the selected workload.  After the
timed steps every case's peak device memory is measured, forward and backward apart
(the pages' second metric), and ``--protocol pages`` adds the pages' run protocol
(2 or 30 runs of 5 warm-ups + 20 steps per case, median/min/max).  Prints one JSON
line (rank 0).
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from long_context_masked_gb300 import inputs as I  # noqa: E402

METRIC = "attn fwd/bwd TFLOPs/s on unmasked FLOPs per mask & seqlen; % of bf16 peak"
UNIT = "TFLOP/s"
D = 128
DOC_RUNS = 30
FLUSH_BYTES = 256 << 20
FWD_PER_PAIR, BWD_PER_PAIR = 4.0 * D, 10.0 * D
KERNEL_SOURCES = {"attn_fwd": "attn_fwd.cu", "bwd": "attn_bwd.cu", "bwd_preprocess": "attn_bwd.cu"}
SUITES = ("dense", "heterogeneous", "sparse", "varlen", "dynamic")


# ------------------------------------------------------------------ workloads
#
# A workload is a list of groups (S, H_q, H_kv, cases).  Every group shares one set of
# resident tensors; a case is (name, make, per_step) where make(seed) returns the mask
# descriptor and per_step says whether the descriptor is re-drawn every step.

class Case:
    def __init__(self, name, make, per_step=False, dynamic=None):
        self.name, self.make, self.per_step = name, make, per_step
        # dynamic = (block, sparsity, map_heads): the block map is computed on the GPU
        # inside the step (pooled block scores, then top-k); `make` then only gives the
        # host descriptor the CPU oracle sample uses (a random-score top-k map)
        self.dynamic = dynamic


def dense_cases(s):
    return [Case("FULL", lambda st: I.make_desc(I.FULL, s)),
            Case("CAUSAL", lambda st: I.make_desc(I.CAUSAL, s)),
            Case("SLIDING_WINDOW", lambda st: I.make_desc(I.SLIDING_WINDOW, s, window=4096)),
            Case("FULL_DOCUMENT", lambda st: I.make_desc(I.FULL_DOCUMENT, s, doc_seed=st), True),
            Case("CAUSAL_DOCUMENT", lambda st: I.make_desc(I.CAUSAL_DOCUMENT, s, doc_seed=st),
                 True)]


def heterogeneous_cases(s):
    return [Case("PREFIX_LM", lambda st: I.make_desc(I.PREFIX_LM, s, prefix_len=s // 4)),
            Case("SHARED_QUESTION",
                 lambda st: I.make_desc(I.SHARED_QUESTION, s, question=2048,
                                        answers=[(s - 2048) // 4] * 4)),
            Case("GLOBAL_SLIDING",
                 lambda st: I.make_desc(I.GLOBAL_SLIDING, s, num_global=256, window=4096)),
            Case("CAUSAL_BLOCKWISE", lambda st: I.make_desc(I.CAUSAL_BLOCKWISE, s, block=2048)),
            Case("BLOCK_CAUSAL_DOCUMENT",
                 lambda st: I.make_desc(I.BLOCK_CAUSAL_DOCUMENT, s, block=2048, doc_seed=st),
                 True),
            # the block size the pages' own measurement section gives for this mask
            Case("BLOCK_CAUSAL_DOCUMENT_Bk1024",
                 lambda st: I.make_desc(I.BLOCK_CAUSAL_DOCUMENT, s, block=1024, doc_seed=st),
                 True),
            Case("SLIDING_WINDOW_DOCUMENT",
                 lambda st: I.make_desc(I.SLIDING_WINDOW_DOCUMENT, s, window=1024, doc_seed=st),
                 True)]


def sparse_cases(s, map_heads):
    out = []
    for b in (64, 128):
        for sp in (0.2, 0.5, 0.8):
            out.append(Case(f"UNIFORM_b{b}_s{sp}",
                            lambda st, b=b, sp=sp: I.make_desc(
                                I.BLOCK_SPARSE_UNIFORM, s, sparse_block=b, sparsity=sp,
                                map_heads=map_heads, map_seed=1000 * b + int(10 * sp))))
    return out


def dynamic_cases(s, map_heads, block=128, sparsity=0.5):
    import oracle

    nb = (s + block - 1) // block

    def make(st):
        k = oracle.topk_count(nb, sparsity)
        bmap = oracle.topk_block_map(I.random_block_scores(1, nb, nb, seed=st), k)
        return I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=block, map_heads=1,
                          n_row_blocks=nb, n_col_blocks=nb, block_map=bmap)
    return [Case(f"POOLED_TOPK_b{block}_s{sparsity}", make, dynamic=(block, sparsity, map_heads))]


def workload(suite, case=None):
    """(groups, description) of a named workload, or of one S:MASK dense case."""
    groups, text = _workload(suite, case)
    return groups, text.replace("d=128", f"d={D}")


def _workload(suite, case=None):
    if case is not None:
        s_txt, m_txt = case.split(":")
        s = int(s_txt)
        cases = [c for c in dense_cases(s) if c.name == m_txt]
        if not cases:
            raise SystemExit(f"unknown mask {m_txt}")
        return [(s, 64, 8, cases)], f"single case {case} (GQA 64:8, d=128)"
    if suite == "dense":
        return ([(s, 64, 8, dense_cases(s)) for s in (8192, 16384, 32768, 49152)],
                "dense regular masks (FULL, CAUSAL, SLIDING_WINDOW w=4096, FULL_DOCUMENT, "
                "CAUSAL_DOCUMENT with lognormal(ln 2048, 1) documents clipped to [128, S]), "
                "GQA 64:8, d=128, B=1 per GPU, S in {8K, 16K, 32K, 48K}")
    if suite == "heterogeneous":
        return ([(32768, 64, 64, heterogeneous_cases(32768))],
                "heterogeneous static masks, S=32K, MHA 64:64, d=128: PREFIX_LM (prefix 8K), "
                "SHARED_QUESTION (2K question + 4 x 7.5K answers), GLOBAL_SLIDING (256 global, "
                "w=4096), CAUSAL_BLOCKWISE (2K blocks), BLOCK_CAUSAL_DOCUMENT (2K and 1K "
                "blocks in lognormal documents); plus the sliding window (w=1024) inside "
                "lognormal documents")
    if suite == "sparse":
        groups = []
        for s in (32768, 65536, 131072):
            groups.append((s, 64, 8, sparse_cases(s, 8)))
            groups.append((s, 32, 32, sparse_cases(s, 32)))
        return (groups, "uniform block-sparse maps (Bernoulli keep, diagonal blocks kept), "
                        "blocks 64/128, sparsity 0.2/0.5/0.8, S in {32K, 64K, 128K}, GQA 64:8 "
                        "(one map per KV head) and MHA 32:32 (one map per head), d=128")
    if suite == "varlen":
        return ([(131072, 64, 8, [Case("CAUSAL_DOCUMENT+VARIABLE_BLOCKS",
                                       lambda st: I.make_desc(I.BLOCK_SPARSE_VARIABLE, 131072,
                                                              map_heads=8, map_seed=st,
                                                              doc_seed=st), True)])],
                "S=128K, GQA 64:8, d=128: CAUSAL_DOCUMENT (lognormal documents) AND one "
                "variable block partition per KV head (block sizes 32..256, multiples of 16) "
                "with 50% of the causal blocks kept")
    if suite == "dynamic":
        return ([(s, 64, 8, dynamic_cases(s, 8)) for s in (32768, 65536, 131072)],
                "dynamic block-sparse masks: per step, block scores from mean-pooled Q/K "
                "(128-blocks, one map per KV head), top-k per query block at sparsity 0.5, "
                "plan build from the device map, then forward + backward; S in {32K, 64K, "
                "128K}, GQA 64:8, d=128")
    raise ValueError(suite)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p["bf16_tflops_sustained"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle sample

_ORACLE_INPUTS = {}


def first_map_head(desc):
    """The descriptor restricted to its first map head (query head 0 uses it)."""
    if desc.map_heads == 1:
        return desc
    cut = {"map_heads": 1, "block_map": desc.block_map[:1]}
    for name in ("row_offsets", "col_offsets"):
        if getattr(desc, name) is not None:
            cut[name] = getattr(desc, name)[:1]
    return I.MaskDesc(**{**desc.__dict__, **cut})


def oracle_sample(groups, rows_per_case, seed=0, budget_s=None):
    """Time the fp64 oracle on a bounded sample of the workload.

    Sample: for every case of the workload, query head 0 (with its KV head and map)
    and ``rows_per_case`` whole query rows from the middle of the sequence (all keys),
    forward and backward.  Credited FLOPs: 14*d per allowed pair of the sampled rows.
    Stops starting new cases once ``budget_s`` seconds are spent.
    Returns (TFLOP/s, seconds, description).
    """
    import oracle

    flops = 0.0
    secs = 0.0
    done = total = 0
    for s, hq, hkv, cases in groups:
        key = (s, hq // hkv)
        if key not in _ORACLE_INPUTS:
            _ORACLE_INPUTS[key] = tuple(x.float().numpy()
                                        for x in I.qkv_do(1, s, hq // hkv, 1, D, s))
        q, k, v, do = _ORACLE_INPUTS[key]
        for c in cases:
            total += 1
            if budget_s is not None and secs > budget_s:
                continue
            desc = first_map_head(c.make(seed % DOC_RUNS))
            r0 = s // 2
            r1 = min(s, r0 + rows_per_case)
            t0 = time.perf_counter()
            oracle.attn_bwd_ref(q, k, v, do, desc, heads=[0], row_range=(r0, r1))
            secs += time.perf_counter() - t0
            n_pairs = int(np.count_nonzero(oracle.mask_rows(desc, 0, np.arange(r0, r1))))
            flops += 14.0 * D * n_pairs
            done += 1
    what = (f"fp64 NumPy oracle fwd+bwd, query head 0, {rows_per_case} middle rows x all keys, "
            f"{done} of {total} cases")
    return flops / secs / 1e12, secs, what


def run_reference(args, rank):
    if rank != 0:
        return
    groups, text = workload(args.suite, args.case)
    for _ in range(args.warmup):
        oracle_sample(groups, 64, seed=0)
    vals, secs = [], []
    for step in range(args.steps):
        v, s, what = oracle_sample(groups, 64, seed=step)
        vals.append(v)
        secs.append(s)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 inputs; lognormal documents)",
            "config": {"workload": text, "suite": args.suite, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": what},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def traffic_from_profiles(kernel, tag):
    """DRAM bytes per launch of `kernel` recorded under profiles/ for workload `tag`, if
    the recording matches the kernel's current source (sha256 prefix), else None."""
    src = os.path.join(ROOT, "long_context_masked_gb300", "csrc", KERNEL_SOURCES.get(kernel, ""))
    try:
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    pat = re.compile(r"traffic_bytes_per_launch\s+(\w+)\s+(\d+)\s+source_sha256=([0-9a-f]+)"
                     r"\s+workload=(\S+)")
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for m in pat.finditer(f.read()):
                if m.group(1) == kernel and m.group(3) == sha and m.group(4) == tag:
                    return int(m.group(2))
    return None


def aggregate(flops, ms, dist=None, device=None):
    """Whole-job totals under weak scaling: FLOPs summed over ranks, time the maximum
    over ranks (every rank runs its own batch entry; there is no data-path collective,
    only this reduction of the measurements)."""
    if dist is None or not dist.is_initialized():
        return float(flops), float(ms)
    import torch

    t = torch.tensor([float(flops)], dtype=torch.float64, device=device)
    m = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(t.item()), float(m.item())


def tflops(flops, ms):
    return flops / (ms * 1e-3) / 1e12


def memory_row(d, info, s, hq):
    """Device memory of one (S, mask) case: the attention tensors this path holds (Q, K,
    V, O, dO, dQ, dK, dV, LSE and the backward workspace, from the allocated tensors),
    the plan (as the library reports it), and the activation memory of a standard
    attention module by the pages' model 11bshd + 5bhs^2 + 2bshd, read as bytes with
    hidden size h*d (LongCA-bench summary, appendix A.4.2)."""
    tensors = sum(t.numel() * t.element_size()
                  for t in list(d["dev"]) + [d[x] for x in ("o", "lse", "dq", "dk", "dv", "ws")])
    model = (13 * s * hq * D + 5 * hq * s * s)
    return {"attention_tensors_gb": round(tensors / 1e9, 3),
            "plan_mb": round(info.get("device_bytes", 0) / 1e6, 2),
            "standard_attention_model_gb": round(model / 1e9, 2)}


def measured_memory(lca, torch, dev, s, hq, hkv, desc, seed):
    """Peak device memory of one (S, mask) case, forward and backward separately (the
    pages' second metric, LongCA-bench summary appendix A.4.2): the torch allocator's
    peak while the pass runs, with its inputs resident and its outputs and workspace
    allocated by the call, plus the plan's device bytes (allocated by the library, so
    not seen by torch).  Forward: Q, K, V, O, LSE.  Backward: Q, K, V, O, LSE, dO,
    dQ, dK, dV and the workspace."""
    hq_, hk_, hv_, hdo = I.qkv_do(1, s, hq, hkv, D, seed)
    q, k, v = (x.to(dev) for x in (hq_, hk_, hv_))
    plan = lca.mask_build(desc, 128, 128)
    plan_bytes = plan.info["device_bytes"]
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    o, lse = lca.attn_fwd(plan, q, k, v)
    torch.cuda.synchronize(dev)
    fwd = torch.cuda.max_memory_allocated(dev) + plan_bytes
    do = hdo.to(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    grads = lca.attn_bwd(plan, q, k, v, o, do, lse)
    torch.cuda.synchronize(dev)
    bwd = torch.cuda.max_memory_allocated(dev) + plan_bytes
    del q, k, v, do, o, lse, grads, plan
    torch.cuda.empty_cache()
    return fwd, bwd


def case_label(suite, s, hq, hkv, name):
    return f"S={s}/{name}" if suite == "dense" else f"S={s}/{hq}:{hkv}/{name}"


def pages_protocol(args, groups, data, lca, torch, stream, flush, pk):
    """Per case: n runs (2 for single-sequence masks, 30 for multi-sequence ones: the
    document masks, SHARED_QUESTION and BLOCK_CAUSAL_DOCUMENT; LongCA-bench summary,
    appendix A.4 "Measurement procedure"), each with its own descriptor draw (seed =
    run), 5 warm-up steps and 20 timed steps (L2 flushed before each); a run's value is
    its median step, and the case reports the median, minimum and maximum over runs.
    SHARED_QUESTION's layout is fixed, so its runs repeat one descriptor on the same
    inputs."""
    out = {}
    for gi, (s, hq, hkv, cases) in enumerate(groups):
        d = data[gi]
        q, k, v, do = d["dev"]
        for c in cases:
            if c.dynamic:
                continue
            multi = c.per_step or c.name == "SHARED_QUESTION"
            runs = DOC_RUNS if multi else 2
            fwd_runs, bwd_runs = [], []
            for r in range(runs):
                desc = c.make(r)
                plan = lca.mask_build(desc, 128, 128)
                pairs = int(plan.n_valid().sum()) * (hq // plan.info["map_heads"])
                f_t, b_t = [], []
                for st in range(5 + 20):
                    flush.zero_()
                    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                    ev[0].record(stream)
                    lca.attn_fwd(plan, q, k, v, out=d["o"], lse=d["lse"])
                    ev[1].record(stream)
                    lca.attn_bwd(plan, q, k, v, d["o"], do, d["lse"], dq=d["dq"], dk=d["dk"],
                                 dv=d["dv"], workspace=d["ws"])
                    ev[2].record(stream)
                    torch.cuda.synchronize()
                    if st >= 5:
                        f_t.append(tflops(FWD_PER_PAIR * pairs, ev[0].elapsed_time(ev[1])))
                        b_t.append(tflops(BWD_PER_PAIR * pairs, ev[1].elapsed_time(ev[2])))
                fwd_runs.append(statistics.median(f_t))
                bwd_runs.append(statistics.median(b_t))
                del plan
            out[case_label(args.suite, s, hq, hkv, c.name)] = {
                "runs": runs,
                "fwd_tflops": [round(statistics.median(fwd_runs), 1), round(min(fwd_runs), 1),
                               round(max(fwd_runs), 1)],
                "bwd_tflops": [round(statistics.median(bwd_runs), 1), round(min(bwd_runs), 1),
                               round(max(bwd_runs), 1)],
                "fwd_pct_peak_median": round(100 * statistics.median(fwd_runs) / pk["bf16"], 1),
                "bwd_pct_peak_median": round(100 * statistics.median(bwd_runs) / pk["bf16"], 1)}
    return {"order": "[median, min, max] over runs of the per-run median step",
            "cases": out}


def run_gpu(args, rank, world):
    import torch

    import long_context_masked_gb300 as lca

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lca.load_library()
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        dist.init_process_group("nccl", device_id=dev)

    groups, text = workload(args.suite, args.case)
    default = args.suite == "dense" and not args.case
    tag = "bench_default" if default else (f"case_{args.case}" if args.case else args.suite)
    if D != 128:
        tag += f"_d{D}"     # profiles/ record traffic per head dimension

    # resident inputs (one batch entry per GPU, seeded by rank) and output buffers
    data = []
    for s, hq, hkv, _ in groups:
        q, k, v, do = I.qkv_do(1, s, hq, hkv, D, seed=1000 * rank + s + (hq != 64) * hq)
        data.append({"host": (q, k, v, do) if default else None,
                     "dev": tuple(x.to(dev) for x in (q, k, v, do)),
                     "o": torch.empty((1, s, hq, D), dtype=torch.bfloat16, device=dev),
                     "lse": torch.empty((1, hq, s), dtype=torch.float32, device=dev),
                     "dq": torch.empty((1, s, hq, D), dtype=torch.bfloat16, device=dev),
                     "dk": torch.empty((1, s, hkv, D), dtype=torch.bfloat16, device=dev),
                     "dv": torch.empty((1, s, hkv, D), dtype=torch.bfloat16, device=dev),
                     # lca_attn_bwd_workspace: LSE2 and D rows padded to 128
                     "ws": torch.empty((2 * hq * ((s + 127) // 128 * 128),),
                                       dtype=torch.float32, device=dev)})
        del q, k, v, do
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    # descriptors are drawn on the host before any timing
    descs = {}
    n_draws = min(DOC_RUNS, args.warmup + args.steps)
    for gi, (_, _, _, cases) in enumerate(groups):
        for ci, c in enumerate(cases):
            if c.dynamic:
                continue
            for st in (range(n_draws) if c.per_step else (0,)):
                descs[(gi, ci, st)] = c.make(st)

    def desc_of(gi, ci, st):
        return descs[(gi, ci, st % DOC_RUNS if groups[gi][3][ci].per_step else 0)]

    def step(st, timers=None, e2e=None):
        plans = []
        for gi, (s, hq, hkv, cases) in enumerate(groups):
            d = data[gi]
            if e2e is not None:
                for src, dst in zip(e2e["h2d"][gi], d["dev"]):
                    dst.copy_(src, non_blocking=True)
            q, k, v, do = d["dev"]
            for ci, c in enumerate(cases):
                ev = None
                if timers is not None:
                    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                    ev[0].record(stream)
                if c.dynamic:
                    blk, sparsity, hmaps = c.dynamic
                    scores = lca.block_scores(q, k, blk, hmaps)
                    nb = scores.shape[1]
                    dmap = lca.block_topk(scores, max(1, min(nb, round((1 - sparsity) * nb))))
                    desc = I.MaskDesc(I.BLOCK_SPARSE_UNIFORM, s, block=blk, map_heads=hmaps,
                                      n_row_blocks=nb, n_col_blocks=nb, block_map=dmap)
                else:
                    desc = desc_of(gi, ci, st)
                plan = lca.mask_build(desc, 128, 128)
                if ev is not None:
                    ev[1].record(stream)
                lca.attn_fwd(plan, q, k, v, out=d["o"], lse=d["lse"])
                if ev is not None:
                    ev[2].record(stream)
                lca.attn_bwd(plan, q, k, v, d["o"], do, d["lse"], dq=d["dq"], dk=d["dk"],
                             dv=d["dv"], workspace=d["ws"])
                if ev is not None:
                    ev[3].record(stream)
                    timers.append((gi, c.name, ev))
                plans.append((gi, c.name, plan))
            if e2e is not None:
                for src, dst in zip((d["o"], d["lse"], d["dq"], d["dk"], d["dv"]), e2e["d2h"][gi]):
                    dst.copy_(src, non_blocking=True)
        return plans

    def sync_all():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def pair_counts(plans):
        """(gi, name, query-head pairs, plan info) per plan; drops the plans."""
        return [(gi, name, int(p.n_valid().sum()) * (groups[gi][1] // p.info["map_heads"]),
                 dict(p.info)) for gi, name, p in plans]

    for w in range(args.warmup):
        step(w)
    sync_all()

    # ---- device-resident timed steps
    torch.cuda.reset_peak_memory_stats(dev)
    lca.profile_enable(True)
    lca.profile_read()
    step_ms, counts, timers = [], [], []
    with ClockSampler(local) as clk:
        for st in range(args.steps):
            flush.zero_()
            sync_all()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plans = step(st, timers)
            e1.record(stream)
            sync_all()
            step_ms.append(e0.elapsed_time(e1))
            counts.append(pair_counts(plans))
            del plans
    prof = lca.profile_read()
    lca.profile_enable(False)
    clocks = clk.summary()
    peak_mem = torch.cuda.max_memory_allocated(dev)

    # credited FLOPs from the plans' exact pair counts
    total_pairs = sum(c[2] for st_counts in counts for c in st_counts)
    job_flops, total_ms = aggregate(total_pairs * (FWD_PER_PAIR + BWD_PER_PAIR), sum(step_ms),
                                    dist, dev)
    value = tflops(job_flops, total_ms)
    pk = peaks()

    per_cfg = {}
    flat = [c for st_counts in counts for c in st_counts]
    for (gi, name, ev), (gi2, name2, hp, info) in zip(timers, flat):
        assert (gi, name) == (gi2, name2)
        s, hq, hkv, _ = groups[gi]
        b_ms = ev[0].elapsed_time(ev[1])
        f_ms = ev[1].elapsed_time(ev[2])
        w_ms = ev[2].elapsed_time(ev[3])
        acc = per_cfg.setdefault(case_label(args.suite, s, hq, hkv, name),
                                 {"fwd": [], "bwd": [], "build_ms": [], "fwd_ms": [],
                                  "bwd_ms": [], "pairs": [], "eff": [], "f_tile_us": [],
                                  "b_tile_us": [], "nonskip": [], "info": info, "hq": hq,
                                  "gi": gi, "s": s})
        acc["fwd"].append(tflops(FWD_PER_PAIR * hp, f_ms))
        acc["bwd"].append(tflops(BWD_PER_PAIR * hp, w_ms))
        acc["build_ms"].append(b_ms)
        acc["fwd_ms"].append(f_ms)
        acc["bwd_ms"].append(w_ms)
        acc["pairs"].append(hp)
        # allowed pairs per pair of this step's non-skipped head-tiles (re-drawn masks
        # change both from step to step)
        head_tiles = info["nnz"] * (hq // info["map_heads"])
        acc["eff"].append(hp / (head_tiles * 128 * 128))
        acc["f_tile_us"].append(1e3 * f_ms / head_tiles)
        acc["nonskip"].append(info["nnz"] / (info["map_heads"] * info["n_qt"] * info["n_kt"]))
        acc["b_tile_us"].append(1e3 * w_ms / head_tiles)
    per_config = {}
    for label, v in per_cfg.items():
        fwd, bwd = statistics.median(v["fwd"]), statistics.median(v["bwd"])
        row = {"fwd_tflops": round(fwd, 1), "bwd_tflops": round(bwd, 1),
               "fwd_pct_peak": round(100 * fwd / pk["bf16"], 1),
               "bwd_pct_peak": round(100 * bwd / pk["bf16"], 1),
               "fwd_tflops_min_max": [round(min(v["fwd"]), 1), round(max(v["fwd"]), 1)],
               "bwd_tflops_min_max": [round(min(v["bwd"]), 1), round(max(v["bwd"]), 1)],
               "build_ms": round(statistics.median(v["build_ms"]), 3),
               "memory": memory_row(data[v["gi"]], v["info"], v["s"], v["hq"])}
        if not default:
            f_ms, w_ms = statistics.median(v["fwd_ms"]), statistics.median(v["bwd_ms"])
            row.update({"fwd_ms": round(f_ms, 3), "bwd_ms": round(w_ms, 3),
                        "nonskipped_tile_fraction": round(statistics.median(v["nonskip"]), 4),
                        # allowed pairs per pair of the non-skipped tiles (partial-tile waste)
                        "tile_efficiency": round(statistics.median(v["eff"]), 4),
                        "fwd_us_per_head_tile": round(statistics.median(v["f_tile_us"]), 4),
                        "bwd_us_per_head_tile": round(statistics.median(v["b_tile_us"]), 4)})
        per_config[label] = row

    # roofline of the dominant kernel (largest share of the timed region)
    # algorithmic FLOPs per allowed pair and query head: the forward 4d; the backward
    # launch (dK/dV and dQ passes) 10d, the method's S, dP, dV, dK and dQ products (its
    # recomputation of S and dP in the dQ pass is not credited)
    algo = {"attn_fwd": FWD_PER_PAIR, "bwd": BWD_PER_PAIR}
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0] if prof else None
    roofline = None
    if dom in algo:
        launches, ms = prof[dom]
        achieved = tflops(algo[dom] * total_pairs, ms)
        roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                    "frac": round(achieved / pk["bf16_sustained"], 4),
                    "frac_of_burst": round(achieved / pk["bf16"], 4),
                    "peak_note": f"{pk['source']} bf16 dense (sustained; burst {pk['bf16']})",
                    "traffic": traffic_from_profiles(dom, tag),
                    "launches": launches, "avg_launch_ms": round(ms / launches, 3),
                    "algorithmic_flops_per_pair": algo[dom]}
    kernel_share = {k: round(v[1] / sum(x[1] for x in prof.values()), 4) for k, v in prof.items()}
    gpu_launches = int(sum(v[0] for v in prof.values()))

    # ---- end to end through the public API with host buffers (default workload)
    e2e_steps = max(1, min(args.steps, 5)) if default else 0
    e2e_value, h2d_bytes, d2h_bytes = None, 0, 0
    if e2e_steps:
        h2d = [[x.pin_memory() for x in d["host"]] for d in data]
        d2h = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for t in (d["o"], d["lse"], d["dq"], d["dk"], d["dv"])] for d in data]
        h2d_bytes = sum(x.numel() * x.element_size() for g in h2d for x in g)
        d2h_bytes = sum(x.numel() * x.element_size() for g in d2h for x in g)
        e2e_ms, e2e_pairs = [], 0
        for st in range(e2e_steps):
            flush.zero_()
            sync_all()
            t0 = time.perf_counter()
            plans = step(st, e2e={"h2d": h2d, "d2h": d2h})
            sync_all()
            e2e_ms.append(1e3 * (time.perf_counter() - t0))
            e2e_pairs += sum(c[2] for c in pair_counts(plans))
            del plans
        e2e_flops, e2e_total_ms = aggregate(e2e_pairs * (FWD_PER_PAIR + BWD_PER_PAIR),
                                            sum(e2e_ms), dist, dev)
        e2e_value = tflops(e2e_flops, e2e_total_ms)

    # ---- the pages' run protocol (optional): per case 2 runs (single-sequence masks) or
    # 30 independently drawn runs (multi-sequence masks), each 5 warm-ups + 20 steps
    pages = pages_protocol(args, groups, data, lca, torch, stream, flush, pk) \
        if args.protocol == "pages" else None

    # ---- measured peak memory per case, forward and backward (resident buffers freed)
    if not args.no_memory:
        del data, flush
        torch.cuda.empty_cache()
        for gi, (s, hq, hkv, cases) in enumerate(groups):
            for ci, c in enumerate(cases):
                seeds = range(3) if c.per_step else (0,)
                meas = [measured_memory(lca, torch, dev, s, hq, hkv, c.make(sd), 1000 * rank + s)
                        for sd in seeds]
                row = per_config[case_label(args.suite, s, hq, hkv, c.name)]["memory"]
                row["fwd_peak_gb"] = round(statistics.median(m[0] for m in meas) / 1e9, 3)
                row["bwd_peak_gb"] = round(statistics.median(m[1] for m in meas) / 1e9, 3)
                row["peak_note"] = ("torch allocator peak during the pass + plan bytes; median "
                                    f"over {len(meas)} draw(s)")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, secs, what = oracle_sample(groups, 2048, seed=0, budget_s=30.0)
        cpu = {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": what + f" ({secs:.1f} s)"}

    full_causal = [v for k, v in per_config.items()
                   if k.split("/")[-1] in ("FULL", "CAUSAL") and int(k[2:].split("/")[0]) >= 16384]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 Q/K/V/dO; lognormal document lengths (the "
                "pages' corpora are not available)",
        "config": {"workload": text, "suite": "case" if args.case else args.suite,
                   "head_dim": D, "batch_per_gpu": 1, "tiles": "128x128",
                   "step": "per (S, mask): mask build (for dynamic masks: block scores + top-k + plan) + forward + backward",
                   "l2": "flushed before every timed step (256 MB write)",
                   "parallelism": f"replicas x{world} (independent batch entries, no collective)"},
        "headline": {
            "fwd_pct_peak_full_causal_S>=16K_min":
                min(x["fwd_pct_peak"] for x in full_causal) if full_causal else None,
            "bwd_pct_peak_full_causal_S>=16K_min":
                min(x["bwd_pct_peak"] for x in full_causal) if full_causal else None},
        "per_config": per_config,
        "pages_protocol": pages,
        "roofline": roofline,
        "kernel_time_share": kernel_share,
        "peak_memory_gb": round(peak_mem / 2**30, 3),
        "cpu_baseline": cpu,
        "e2e": {"value": None if e2e_value is None else round(e2e_value, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "steps": e2e_steps},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--suite", choices=SUITES, default="dense",
                    help="workload to time (default: the dense regular masks)")
    ap.add_argument("--head-dim", type=int, choices=(64, 128), default=128,
                    help="head dimension of the synthetic Q/K/V (the benchmark's configs use 128)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed oracle sample in the GPU arm")
    ap.add_argument("--protocol", choices=("steps", "pages"), default="steps",
                    help="'pages' adds the pages' run protocol per case (2 or 30 runs of 5 "
                         "warm-ups + 20 steps; median/min/max over runs) after the timed steps")
    ap.add_argument("--no-memory", action="store_true",
                    help="skip the per-case peak-memory measurement (after the timed steps)")
    ap.add_argument("--case", default=None,
                    help="run a single S:MASK case of the dense workload (e.g. 16384:FULL) "
                         "for profiler captures; skips the end-to-end and CPU legs")
    args = ap.parse_args()
    global D, FWD_PER_PAIR, BWD_PER_PAIR
    D = args.head_dim
    FWD_PER_PAIR, BWD_PER_PAIR = 4.0 * D, 10.0 * D
    if args.suite == "dynamic" and D != 128:
        ap.error("the dynamic suite's block scores are implemented for head_dim 128")
    if args.case:
        args.no_cpu_baseline = True
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_gpu(args, rank, world)


if __name__ == "__main__":
    main()
