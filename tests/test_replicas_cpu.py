"""The multi-rank (replicas) path of bench.py on CPU with the gloo backend, world size 2.

Tokens are independent, so N GPUs run N replicas with no exchange on the data path; the
only cross-rank operations are the timing reduction (the job runs as long as its slowest
replica) and rank 0 alone printing the JSON line.  Both run here without a GPU."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    bench = _bench()
    # each replica's own time; every rank must see the slowest one
    got = bench.max_over_ranks(10.0 + 3.0 * rank, world, device="cpu")
    out.put((rank, got, bench.job_throughput(world, 16, 5, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_timing_reduction_takes_the_slowest_replica_on_every_rank():
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    slowest = 10.0 + 3.0 * (world - 1)
    for rank, got, thr in res:
        assert got == slowest
        # whole-job tokens/s: every replica's 16 tokens x 5 steps over the slowest time
        assert thr == pytest.approx(world * 16 * 5 / (slowest / 1e3))


def test_single_rank_needs_no_process_group():
    bench = _bench()
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_throughput(1, 4, 10, 20.0) == pytest.approx(2000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
           str(_free_port()), "bench.py", "--impl", "reference", "--gpus", "2", "--steps",
           "1", "--warmup", "3", "--workload", "tiny_m4_e16_k4"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
