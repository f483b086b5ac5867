"""The N > 1 path of bench.py on CPU: two gloo ranks, as torchrun would start them.

The path shards by request with no exchange, so N GPUs run N independent replicas; the only
multi-rank logic is the host side: a barrier, the slowest rank's step time (max over ranks)
and the whole-job rate. Those are what these tests run, with the gloo backend on 127.0.0.1."""
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


def _rank_main(rank, ws, port, step_ms, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="env://")
    env_ws, env_rank, _ = bench.dist_env()
    dist.barrier()
    slowest = bench.max_over_ranks(step_ms[rank], env_ws, "cpu")
    rate = bench.replica_rate(1000.0, env_ws, slowest)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{env_rank} {env_ws} {slowest!r} {rate!r}\n")


@pytest.mark.parametrize("step_ms", [(2.0, 3.5), (4.0, 1.0)])
def test_two_replicas_take_the_slowest_rank(tmp_path, step_ms):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, _free_port(), step_ms, str(tmp_path)), nprocs=ws,
                       join=True, start_method="spawn")
    worst = max(step_ms)
    for r in range(ws):
        rank, got_ws, slowest, rate = open(tmp_path / f"r{r}.txt").read().split()
        assert int(rank) == r and int(got_ws) == ws
        assert float(slowest) == worst
        # whole-job rate: both replicas' units over the slowest replica's time
        assert float(rate) == pytest.approx(2 * 1000.0 / (worst * 1e-3))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.replica_rate(500.0, 1, 2.0) == pytest.approx(250000.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle arm runs on rank 0 alone: another rank exits 0 at once and
    prints nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
