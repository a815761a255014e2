"""bench.py's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

The decode path has no exchange step (each (sequence, KV head) depends only on
its own pages), so several GPUs run independent replicas; what bench.py adds
for N > 1 is the process group, the barriers around the timed region and the
max-over-ranks reduction of the elapsed time.  Those run here with the gloo
backend; the reference arm (the oracle on host cores) runs end to end under
torchrun with two ranks, rank 0 alone printing its line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    m = bench.reduce_max(1.5 + rank, w)  # each rank's elapsed time; the max wins
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": m}, f)
    dist.destroy_process_group()


def test_reduce_max_and_barriers_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for rank in range(world):
        with open(tmp_path / f"rank{rank}.json") as f:
            assert json.load(f)["max"] == pytest.approx(2.5)


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench

    assert bench.dist_setup() == (1, 0, 0)
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)  # no-op


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    env["CUDA_VISIBLE_DEVICES"] = ""  # CPU ranks: the reference arm needs no GPU
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "2",
           "--warmup", "3", "--reference-budget", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the oracle's flop rate: 4 D flops per token and query head against at least
    # 4 D bytes of K and V per token and KV head, so at most G = 2 flops per byte
    cb = line["cpu_baseline"]
    assert 0 < cb["gflop_per_s"] <= 2 * cb["value"] * 1.001
    assert line["e2e"]["h2d_bytes_per_step"] == 0
