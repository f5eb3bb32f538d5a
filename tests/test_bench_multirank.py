"""The multi-rank measurement logic of bench.py on CPU (gloo, world size 2): whole-job
FLOPs are summed over ranks and the time is the maximum over ranks; the reference arm
runs on rank 0 only."""
import io
import os
import socket
import contextlib

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        flops = [3.0e12, 5.0e12][rank]
        ms = [20.0, 35.0][rank]
        out[rank] = bench.aggregate(flops, ms, dist, "cpu")
    finally:
        dist.destroy_process_group()


def test_aggregate_sums_flops_and_takes_max_time():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        assert res[rank] == (8.0e12, 35.0)
    assert bench.tflops(*res[0]) == pytest.approx(8.0e12 / 0.035 / 1e12)


def test_aggregate_single_process_is_identity():
    assert bench.aggregate(2.0e12, 10.0) == (2.0e12, 10.0)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        steps, warmup, gpus = 1, 0, 2
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args(), rank=1)
    assert buf.getvalue() == ""


def test_workloads_are_well_formed():
    """Every suite names its groups with H_q divisible by H_kv and unique case labels;
    the cheap descriptors of each suite build with the group's sequence length."""
    for suite in bench.SUITES:
        groups, text = bench.workload(suite)
        assert groups and text
        labels = set()
        for s, hq, hkv, cases in groups:
            assert hq % hkv == 0 and cases
            for c in cases:
                label = bench.case_label(suite, s, hq, hkv, c.name)
                assert label not in labels
                labels.add(label)
        s, hq, hkv, cases = min(groups, key=lambda g: g[0])
        if s <= 32768 and suite != "varlen":
            for c in cases:
                d = c.make(0)
                assert d.seqlen == s
                assert d.map_heads in (1, hkv, hq)
    groups, _ = bench.workload("dense", case="16384:CAUSAL")
    assert [(g[0], [c.name for c in g[3]]) for g in groups] == [(16384, ["CAUSAL"])]


def test_oracle_sample_with_per_head_maps():
    """The CPU baseline sample takes query head 0 with the first map head's block map."""
    from long_context_masked_gb300 import inputs as I

    s = 512
    case = bench.Case("UNIFORM", lambda st: I.make_desc(I.BLOCK_SPARSE_UNIFORM, s, sparse_block=64,
                                                       sparsity=0.5, map_heads=4, map_seed=3))
    d1 = bench.first_map_head(case.make(0))
    assert d1.map_heads == 1 and d1.block_map.shape == (1, 8, 8)
    v, secs, what = bench.oracle_sample([(s, 8, 4, [case])], 16)
    assert v > 0 and secs > 0 and "1 of 1 cases" in what
