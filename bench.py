#!/usr/bin/env python
"""Throughput of mask-aware exact softmax attention (mask build + forward + backward).

Metric: TFLOP/s on unmasked FLOPs - 4*d*H_q per allowed (i, j) pair forward and
2.5x that backward - per mask and sequence length, plus the fraction of the GB300
bf16 dense tensor peak.  The workload is the benchmark's dense regular masks
(LongCA-bench, sections 2.1 and A.4: FULL, CAUSAL, sliding window, full/causal
document over lognormal-length documents) on GQA 64:8, d = 128, at S = 8K, 16K, 32K
and 48K.  One step runs, for every (S, mask): the tile plan build, the forward and the
backward, on synthetic N(0, 1) bf16 inputs resident on the GPU.  Document masks
re-draw their lengths every step (seed = step mod 30; the pages sample 30 runs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the only reference available here)
on a bounded row sample of the same workload.  Prints one JSON line (rank 0).
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
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
HQ, HKV, D = 64, 8, 128
SEQLENS = (8192, 16384, 32768, 49152)
MASKS = (("FULL", I.FULL, {}), ("CAUSAL", I.CAUSAL, {}),
         ("SLIDING_WINDOW", I.SLIDING_WINDOW, {"window": 4096}),
         ("FULL_DOCUMENT", I.FULL_DOCUMENT, {}), ("CAUSAL_DOCUMENT", I.CAUSAL_DOCUMENT, {}))
DOC_RUNS = 30
WORKLOAD = ("dense regular masks (FULL, CAUSAL, SLIDING_WINDOW w=4096, FULL_DOCUMENT, "
            "CAUSAL_DOCUMENT with lognormal(ln 2048, 1) documents clipped to [128, S]), "
            "GQA 64:8, d=128, B=1 per GPU, S in {8K, 16K, 32K, 48K}")
FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = {"attn_fwd": "attn_fwd.cu", "bwd_dkdv": "attn_bwd.cu", "bwd_dq": "attn_bwd.cu",
                  "bwd_preprocess": "attn_bwd.cu"}


def desc_for(mask_type, s, kw, step):
    seed = step % DOC_RUNS
    return I.make_desc(mask_type, s, doc_seed=seed, **kw)


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
        self.out = ""
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


def oracle_sample(rows_per_combo, seed=0, budget_s=None):
    """Time the fp64 oracle on a bounded sample of the workload.

    Sample: for every (S, mask) of the workload, query head 0 and ``rows_per_combo``
    whole query rows from the middle of the sequence (all keys), forward and
    backward.  Credited FLOPs: 14*d per allowed pair of the sampled rows.
    Returns (TFLOP/s, seconds, description).
    """
    import oracle

    flops = 0.0
    secs = 0.0
    done = 0
    for s in SEQLENS:
        if s not in _ORACLE_INPUTS:
            _ORACLE_INPUTS[s] = tuple(x.float().numpy() for x in I.qkv_do(1, s, 8, 1, D, s))
        q, k, v, do = _ORACLE_INPUTS[s]
        for _, t, kw in MASKS:
            desc = desc_for(t, s, kw, seed)
            r0 = s // 2
            r1 = min(s, r0 + rows_per_combo)
            t0 = time.perf_counter()
            oracle.attn_bwd_ref(q, k, v, do, desc, heads=[0], row_range=(r0, r1))
            secs += time.perf_counter() - t0
            n_pairs = int(np.count_nonzero(oracle.mask_rows(desc, 0, np.arange(r0, r1))))
            flops += 14.0 * D * n_pairs
            done += 1
            if budget_s is not None and secs > budget_s:
                break
        if budget_s is not None and secs > budget_s:
            break
    what = (f"fp64 NumPy oracle fwd+bwd, query head 0, {rows_per_combo} middle rows x all keys, "
            f"{done} of {len(SEQLENS) * len(MASKS)} (S, mask) combos")
    return flops / secs / 1e12, secs, what


def run_reference(args, rank):
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(64, seed=0)
    vals, secs = [], []
    for step in range(args.steps):
        v, s, what = oracle_sample(64, seed=step)
        vals.append(v)
        secs.append(s)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 inputs; lognormal documents)",
            "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": what},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def traffic_from_profiles(kernel):
    """DRAM bytes per launch of `kernel` recorded under profiles/, if the recording
    matches the kernel's current source (sha256 prefix), else None."""
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
                if m.group(1) == kernel and m.group(3) == sha and m.group(4) == "bench_default":
                    return int(m.group(2))
    return None


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

    # resident inputs (one batch entry per GPU, seeded by rank) and output buffers
    data = {}
    for s in SEQLENS:
        q, k, v, do = I.qkv_do(1, s, HQ, HKV, D, seed=1000 * rank + s)
        data[s] = {"host": (q, k, v, do),
                   "dev": tuple(x.to(dev) for x in (q, k, v, do)),
                   "o": torch.empty((1, s, HQ, D), dtype=torch.bfloat16, device=dev),
                   "lse": torch.empty((1, HQ, s), dtype=torch.float32, device=dev),
                   "dq": torch.empty((1, s, HQ, D), dtype=torch.bfloat16, device=dev),
                   "dk": torch.empty((1, s, HKV, D), dtype=torch.bfloat16, device=dev),
                   "dv": torch.empty((1, s, HKV, D), dtype=torch.bfloat16, device=dev),
                   "ws": torch.empty((HQ * s,), dtype=torch.float32, device=dev)}
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    descs = {(s, name, st): desc_for(t, s, kw, st)
             for s in SEQLENS for name, t, kw in MASKS for st in range(DOC_RUNS)}

    def step(st, timers=None, e2e=None):
        plans = []
        for s in SEQLENS:
            d = data[s]
            if e2e is not None:
                for src, dst in zip(e2e["h2d"][s], d["dev"]):
                    dst.copy_(src, non_blocking=True)
            q, k, v, do = d["dev"]
            for name, _, _ in MASKS:
                ev = None
                if timers is not None:
                    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                    ev[0].record(stream)
                plan = lca.mask_build(descs[(s, name, st % DOC_RUNS)], 128, 128)
                lca.attn_fwd(plan, q, k, v, out=d["o"], lse=d["lse"])
                if ev is not None:
                    ev[1].record(stream)
                lca.attn_bwd(plan, q, k, v, d["o"], do, d["lse"], dq=d["dq"], dk=d["dk"],
                             dv=d["dv"], workspace=d["ws"])
                if ev is not None:
                    ev[2].record(stream)
                    timers.append((s, name, ev))
                plans.append((s, name, plan))
            if e2e is not None:
                for src, dst in zip((d["o"], d["lse"], d["dq"], d["dk"], d["dv"]), e2e["d2h"][s]):
                    dst.copy_(src, non_blocking=True)
        return plans

    def sync_all():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        if dist is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    for w in range(args.warmup):
        step(w)
    sync_all()

    # ---- device-resident timed steps
    lca.profile_enable(True)
    lca.profile_read()
    step_ms, timers, plans = [], [], []
    with ClockSampler(local) as clk:
        for st in range(args.steps):
            flush.zero_()
            sync_all()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plans.append(step(st, timers))
            e1.record(stream)
            sync_all()
            step_ms.append(e0.elapsed_time(e1))
    prof = lca.profile_read()
    lca.profile_enable(False)
    clocks = clk.summary()

    # credited FLOPs from the plans' exact pair counts
    pairs = {}
    total_pairs = 0
    for st_plans in plans:
        for s, name, plan in st_plans:
            nv = plan.export()["n_valid"]
            hsum = int(nv.sum()) * (HQ // plan.info["map_heads"])
            pairs.setdefault((s, name), []).append(hsum)
            total_pairs += hsum
    fwd_per_pair, bwd_per_pair = 4.0 * D, 10.0 * D
    total_flops = total_pairs * (fwd_per_pair + bwd_per_pair)
    total_ms = max_over_ranks(sum(step_ms))
    value = world * total_flops / (total_ms * 1e-3) / 1e12
    pk = peaks()

    per_cfg = {}
    for idx, (s, name, ev) in enumerate(timers):
        st = idx // (len(SEQLENS) * len(MASKS))
        hp = pairs[(s, name)][st]
        f_ms, b_ms = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])
        acc = per_cfg.setdefault(f"S={s}/{name}", {"fwd": [], "bwd": []})
        acc["fwd"].append(fwd_per_pair * hp / (f_ms * 1e-3) / 1e12)
        acc["bwd"].append(bwd_per_pair * hp / (b_ms * 1e-3) / 1e12)
    per_config = {k: {"fwd_tflops": round(statistics.median(v["fwd"]), 1),
                      "bwd_tflops": round(statistics.median(v["bwd"]), 1),
                      "fwd_pct_peak": round(100 * statistics.median(v["fwd"]) / pk["bf16"], 1),
                      "bwd_pct_peak": round(100 * statistics.median(v["bwd"]) / pk["bf16"], 1)}
                  for k, v in per_cfg.items()}

    # roofline of the dominant kernel (largest share of the timed region)
    algo = {"attn_fwd": fwd_per_pair, "bwd_dkdv": 8.0 * D, "bwd_dq": 2.0 * D}
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0] if prof else None
    roofline = None
    if dom in algo:
        launches, ms = prof[dom]
        achieved = algo[dom] * total_pairs / (ms * 1e-3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": pk["bf16_sustained"], "unit": "TFLOP/s",
                    "frac": round(achieved / pk["bf16_sustained"], 4),
                    "frac_of_burst": round(achieved / pk["bf16"], 4),
                    "peak_note": f"{pk['source']} bf16 dense (sustained; burst {pk['bf16']})",
                    "traffic": traffic_from_profiles(dom),
                    "launches": launches, "avg_launch_ms": round(ms / launches, 3),
                    "algorithmic_flops_per_pair": algo[dom]}
    kernel_share = {k: round(v[1] / sum(x[1] for x in prof.values()), 4) for k, v in prof.items()}
    gpu_launches = int(sum(v[0] for v in prof.values()))

    # ---- end to end through the public API with host buffers
    e2e_steps = 0 if args.case else max(1, min(args.steps, 3))
    h2d = {s: [x.pin_memory() for x in data[s]["host"]] for s in SEQLENS}
    d2h = {s: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
               for t in (data[s]["o"], data[s]["lse"], data[s]["dq"], data[s]["dk"], data[s]["dv"])]
           for s in SEQLENS}
    h2d_bytes = sum(x.numel() * x.element_size() for s in SEQLENS for x in h2d[s])
    d2h_bytes = sum(x.numel() * x.element_size() for s in SEQLENS for x in d2h[s])
    e2e_ms, e2e_pairs = [], 0
    for st in range(e2e_steps):
        flush.zero_()
        sync_all()
        t0 = time.perf_counter()
        pl = step(st, e2e={"h2d": h2d, "d2h": d2h})
        sync_all()
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
        e2e_pairs += sum(int(p.export()["n_valid"].sum()) * (HQ // p.info["map_heads"])
                         for _, _, p in pl)
    e2e_value = (world * e2e_pairs * (fwd_per_pair + bwd_per_pair) /
                 (max_over_ranks(sum(e2e_ms)) * 1e-3) / 1e12) if e2e_steps else None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, secs, what = oracle_sample(256, seed=0, budget_s=30.0)
        cpu = {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": what + f" ({secs:.1f} s)"}

    full_causal = [per_config[k] for k in per_config
                   if k.split("/")[1] in ("FULL", "CAUSAL") and int(k[2:].split("/")[0]) >= 16384]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 Q/K/V/dO; lognormal document lengths (the "
                "pages' corpora are not available)",
        "config": {"workload": WORKLOAD if not args.case else f"single case {args.case}",
                   "seqlens": list(SEQLENS),
                   "masks": [m[0] for m in MASKS], "h_q": HQ, "h_kv": HKV, "head_dim": D,
                   "batch_per_gpu": 1, "tiles": "128x128",
                   "step": "per (S, mask): mask build + forward + backward",
                   "l2": "flushed before every timed step (256 MB write)",
                   "parallelism": f"replicas x{world} (independent batch entries, no collective)"},
        "headline": {
            "fwd_pct_peak_full_causal_S>=16K_min":
                min(x["fwd_pct_peak"] for x in full_causal) if full_causal else None,
            "bwd_pct_peak_full_causal_S>=16K_min":
                min(x["bwd_pct_peak"] for x in full_causal) if full_causal else None},
        "per_config": per_config,
        "roofline": roofline,
        "kernel_time_share": kernel_share,
        "cpu_baseline": cpu,
        "e2e": {"value": None if e2e_value is None else round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes, "steps": e2e_steps},
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
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed oracle sample in the GPU arm")
    ap.add_argument("--case", default=None,
                    help="run a single S:MASK case (e.g. 16384:FULL) for profiler captures; "
                         "skips the end-to-end and CPU legs")
    args = ap.parse_args()
    if args.case:
        global SEQLENS, MASKS
        s_txt, m_txt = args.case.split(":")
        SEQLENS = (int(s_txt),)
        MASKS = tuple(m for m in MASKS if m[0] == m_txt)
        if not MASKS:
            ap.error(f"unknown mask {m_txt}")
        args.no_cpu_baseline = True
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_gpu(args, rank, world)


if __name__ == "__main__":
    main()
