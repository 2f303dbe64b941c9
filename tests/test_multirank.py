"""The benchmark's multi-replica host path on CPU ranks (gloo, world size 2).

The layer forward does not shard: every GPU runs a whole replica on its own
tokens and no data-path collective exists.  What the replicas share is the
measurement: a barrier around the timed region, the slowest rank's time,
whole-job tokens/s, and one JSON line printed by rank 0.  These tests run
that logic as two CPU processes; no GPU is involved.
"""
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


def _rank_main(rank, world, port, times_ms, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times_ms[rank], world, "cpu")
        value = bench.job_tokens_per_s(world, 512, 10, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_and_throughput_counts_all_ranks(tmp_path):
    """Each rank times a different duration; both must report the larger
    one, and tokens/s must count the tokens of both replicas."""
    times = [4.0, 7.5]
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, times, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["ms"] == 7.5
        # 2 replicas x 512 tokens x 10 steps in 7.5 ms
        assert r["value"] == pytest.approx(2 * 512 * 10 / 7.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_tokens_per_s(1, 16, 4, 2.0) == pytest.approx(16 * 4 / 2e-3)


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference launched as two ranks (the driver's N > 1
    launch): rank 0 alone runs the oracle and prints one JSON line, the
    other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
