"""The batch-sharded multi-GPU path's host logic with two gloo ranks on CPU.

Requests are independent, so each rank runs its own batch with no collective on the data
path; ranks only agree on the timing (max over ranks) and each draws a distinct batch.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads as wl
        # rank-dependent timings: the job is bounded by the slowest rank
        step_ms, e2e_ms, kern_ms = bench.reduce_max([1.0 + rank, 5.0 - rank, 2.0 * rank], world)
        inp = wl.make_decode_inputs(wl.SHAPES["tiny"], [40, 20], seed=bench.rank_seed(rank))
        np.save(os.path.join(out_dir, f"q{rank}.npy"), inp.q)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{step_ms} {e2e_ms} {kern_ms} {bench.job_gbs(1_000_000_000, world, step_ms)}")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_draw_distinct_batches(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [open(tmp_path / f"r{r}.txt").read().split() for r in range(world)]
    for r in res:
        step_ms, e2e_ms, kern_ms, gbs = map(float, r)
        assert (step_ms, e2e_ms, kern_ms) == (2.0, 5.0, 2.0)
        assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)
    q0, q1 = np.load(tmp_path / "q0.npy"), np.load(tmp_path / "q1.npy")
    assert not np.array_equal(q0, q1)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """The launch the benchmark contract uses for N > 1: only rank 0 runs and prints."""
    import json
    import subprocess
    import sys
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--seq-len", "256"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
