"""The multi-rank host logic of bench.py, on CPU: two ranks over gloo, as torchrun starts them.

Replicas share no data-path collective (requests are independent), so what needs checking
without a GPU is the rank bookkeeping, the max over ranks of the step time, the whole-job
throughput, and that only rank 0 of the reference arm works and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.rank_env()
        ms = bench.max_over_ranks(1.0 + 0.5 * rank, env[0])     # the last rank is the slowest
        value = bench.job_throughput(32, env[0], ms)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump({"env": list(env), "ms": ms, "value": value}, f)


def test_step_time_is_the_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        res = json.load(open(tmp_path / f"rank{r}.json"))
        assert res["env"] == [world, r, r]
        assert res["ms"] == 1.5
        assert res["value"] == pytest.approx(32 * world / 1.5e-3)


def test_single_rank_needs_no_process_group():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25, 1) == 2.25
    assert bench.job_throughput(64, 1, 0.5) == pytest.approx(128000.0)


def test_reference_arm_under_torchrun_prints_once():
    # two ranks as the driver launches them; rank 1 exits at once, rank 0 times the oracle
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "tiny_f32"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
