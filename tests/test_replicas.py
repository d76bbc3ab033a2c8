"""The multi-rank host logic of bench.py, on the CPU with the gloo backend.

With N > 1 every rank runs an independent replica of the workload (no
collective on the data path); after timing, one all-reduce takes the slowest
rank's times and rank 0 reports the FLOPs of all ranks over that time.  These
tests run two gloo ranks as spawned processes and check the reduction, the
reported value and that the other ranks of the reference arm do no work.
"""
import argparse
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_times(rank):
    # rank 1 is slower in the step and the main kernel, rank 0 in e2e
    return {"ms_per_step": 0.030 + 0.010 * rank, "main_ms": 0.020 + 0.005 * rank,
            "e2e_s": 300e-6 - 50e-6 * rank}


def _fake_result(rank):
    from conv2d_backward_implicit_dgrad_gb300.workloads import WORKLOADS
    wl = WORKLOADS["resnet_stage"]
    flops = 2.0 * wl.N * wl.Co * wl.oH * wl.oW * wl.Ci * wl.kH * wl.kW
    nbytes = 4.0 * (wl.N * wl.Co * wl.oH * wl.oW + wl.Co * wl.Ci * wl.kH * wl.kW + wl.N * wl.Ci * wl.H * wl.W)
    plan = {k: 0 for k in ("path", "tile_blocks", "slice_n", "chunk_k", "n_chunks", "grid", "n_work",
                           "b_resident", "smem_bytes", "tmem_cols")}
    peaks = {"tf32_tflops": 1000.0, "ffma_tflops": 70.0, "sm_count": 152, "ffma_nominal_tflops": 80.5}
    return wl, {**_rank_times(rank), "prepack_ms": 0.008, "fused_ms": 0.0, "clocks": None, "plan": plan,
                "flops": flops, "bytes": nbytes, "steps": 5, "peaks": peaks}


def _worker(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        wl, r = _fake_result(rank)
        bench.slowest_rank(torch, dist, r, "cpu")
        args = argparse.Namespace(warmup=3, precision="tf32")
        line = bench.build_line(args, wl, r, world)
        queue.put((rank, r["ms_per_step"], r["main_ms"], r["e2e_s"], line["value"], line["n_gpus"],
                   line["e2e"]["value"], line["config"]["parallelism"]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_report_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rank, world, port, queue)) for rank in range(world)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl, r0 = _fake_result(0)
    slow = {k: max(_rank_times(i)[k] for i in range(world)) for k in ("ms_per_step", "main_ms", "e2e_s")}
    for rank, step_ms, main_ms, e2e_s, value, n_gpus, e2e_value, par in results:
        # every rank ends with the same, slowest, times
        assert step_ms == pytest.approx(slow["ms_per_step"], rel=1e-12)
        assert main_ms == pytest.approx(slow["main_ms"], rel=1e-12)
        assert e2e_s == pytest.approx(slow["e2e_s"], rel=1e-12)
        # whole-job throughput: the FLOPs of both replicas over the slowest step
        assert value == pytest.approx(world * r0["flops"] / (slow["ms_per_step"] * 1e-3) / 1e12, rel=1e-12)
        assert e2e_value == pytest.approx(world * r0["flops"] / slow["e2e_s"] / 1e12, rel=1e-12)
        assert n_gpus == world
        assert par == f"replicas x{world}"


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from conv2d_backward_implicit_dgrad_gb300.workloads import WORKLOADS

    def no_oracle(*a, **k):
        raise AssertionError("a rank other than 0 ran the oracle")

    monkeypatch.setattr(bench, "cpu_oracle_run", no_oracle)
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(warmup=1, steps=1, gpus=2)
    assert bench.reference_arm(args, WORKLOADS["tiny"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_rank0_prints_one_line(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from conv2d_backward_implicit_dgrad_gb300.workloads import WORKLOADS

    monkeypatch.setenv("RANK", "0")
    args = argparse.Namespace(warmup=0, steps=1, gpus=2)
    assert bench.reference_arm(args, WORKLOADS["tiny"]) == 0
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
