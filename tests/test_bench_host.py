"""bench.py's host logic on the CPU: the max-over-ranks aggregation with two
gloo ranks, and the reference arm's JSON line (rank 0 prints it, other ranks
exit without work)."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, totals, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = _bench().aggregate_over_ranks(totals[rank], 2.0e12, 4, world, "cpu")
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    totals = [10.0, 12.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, totals, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 12.5, f"rank {rank} kept its own time"
        # every rank runs the whole workload: 2 ranks x 4 steps x 2 TFLOP in 12.5 ms
        assert value == pytest.approx(2 * 4 * 2.0 / 12.5e-3)


def test_one_rank_keeps_its_own_time():
    ms, value = _bench().aggregate_over_ranks(8.0, 1.0e12, 2, 1)
    assert ms == 8.0 and value == pytest.approx(2 * 1.0 / 8.0e-3)


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                           "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_other_ranks_exit_without_work():
    r = _run_reference(1, 2)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    r = _run_reference(0, 1)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    bench = _bench()
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"]
    assert d["config"] == bench.workload_config(bench.HEADLINE, 1)
    assert d["config"]["workload"] == "overfeat_stack"
    assert d["config"]["flops_per_step"] == (d["config"]["flops_per_pass"]
                                             * d["config"]["reps_per_step"])
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_bench_geometry_matches_the_oracle_extent():
    """The benchmark's per-layer output size and FLOP count (which set the
    reported TFLOP/s) agree with the pinned oracle's extent and with the
    direct-convolution count 2*N*K*P*Q*C*R*S, for every workload layer."""
    from oracle import oracle
    from deep_learning_convolution_gb300 import synth
    bench = _bench()
    for wl, layers in synth.WORKLOADS.items():
        for l in layers:
            P, Q = bench.layer_output_dims(l)
            assert P == oracle.out_extent(l.H, l.pad_top, l.pad_bottom, l.R, l.dil_h, l.u)
            assert Q == oracle.out_extent(l.W, l.pad_left, l.pad_right, l.S, l.dil_w, l.v)
            flops, _ = bench.layer_geometry(l, P, Q)
            assert flops == 2 * l.N * l.K * P * Q * l.C * l.R * l.S
        cfg = bench.workload_config(wl, 1)
        assert cfg["flops_per_pass"] == sum(
            bench.layer_geometry(l, *bench.layer_output_dims(l))[0] for l in layers)
        assert cfg["flops_per_step"] == cfg["flops_per_pass"] * cfg["reps_per_step"]


def test_per_launch_events_ride_on_one_pass_in_eight():
    """Every step carries per-launch events on at least one pass, on one pass in
    INST_EVERY when the step has that many, and never past the step's end; the
    timing descriptions name the same rate; every workload's step is whole
    blocks of INST_EVERY passes (one direct pass and one graph replay each)."""
    b = _bench()
    E, h = b.INST_EVERY, b.INST_EVERY // 2
    for reps in (1, 2, 7, 8, 9, 12, 13, 40, 80, 200, 2000):
        inst = b.instrumented_passes(reps)
        assert inst, reps
        assert all(0 <= r < reps for r in inst), (reps, inst)
        assert len(set(inst)) == len(inst)
        # passes r < reps with r = h mod E: ceil((reps - h) / E) of them, or one
        assert len(inst) == max(1, (reps - h + E - 1) // E), (reps, inst)
    assert f"of every {b.INST_EVERY} passes one" in b.TIMING
    assert f"{b.INST_EVERY - 1} are replayed" in b.TIMING
    assert f"one in {b.INST_EVERY}" in b.TIMING_DIRECT
    for reps in list(b.REPS_PER_STEP.values()) + list(b.EXTRA_REPS.values()):
        assert reps % b.INST_EVERY == 0, reps
