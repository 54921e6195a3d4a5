"""bench.py's multi-process path on CPU: two gloo ranks agree on the slowest
rank's time and the whole-job value; under torchrun the reference arm prints
one JSON line from rank 0 and the other rank exits 0 without work."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [1.25, 3.5][rank]
    m = bench.max_over_ranks(local, world, torch.device("cpu"))
    dist.barrier()
    out.put((rank, m, bench.whole_job_us_per_call(m, world)))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_and_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [3.5, 3.5]
    assert [g[2] for g in got] == [1750.0, 1750.0]


def test_single_rank_values():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.0, 1, None) == 2.0
    assert bench.whole_job_us_per_call(0.2384, 1) == 238.4
    assert bench.kernels_per_call(4096, 48) == 5
    assert bench.kernels_per_call(1024, 384) == 5
    assert bench.kernels_per_call(1024, 513) == 7
    assert bench.kernels_per_call(65536, 48) == 7


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us/call" and d["value"] > 0


def test_l2_flush_only_for_steps_that_fit_in_l2():
    import bench
    from w4a16_int4_mixture_gb300 import synth

    def step_bytes(wl, T=None):
        inp = synth.make_inputs(synth.workload(wl, T=T), weights=False)
        return bench.workload_bytes_flops(inp)["layer"]["bytes"]

    assert not bench.needs_l2_flush(step_bytes("ep8-decode"))  # ~1.2 GB of weights
    assert not bench.needs_l2_flush(step_bytes("tp8", 128))    # ~1.1 GB
    assert bench.needs_l2_flush(step_bytes("tp8", 1))          # 8 experts, ~25 MB
    assert bench.needs_l2_flush(step_bytes("tiny"))


def test_cpu_baseline_and_replay_spread():
    import bench
    import oracle
    from w4a16_int4_mixture_gb300 import synth
    oracle.build()
    cb = bench.cpu_baseline(synth.make_inputs(synth.workload("tiny")), single_thread_tokens=4)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert oracle.num_threads() == cb["cores"]  # restored after the one-thread run
    sp = bench.replay_spread_us([0.2, 0.1, 0.3, 0.25, 0.15])
    assert sp == {"median": 200.0, "p10": 100.0, "p90": 300.0, "replays": 5}
    assert bench.replay_spread_us([]) is None
