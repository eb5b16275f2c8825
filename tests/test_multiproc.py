"""Multi-process host logic on CPU (gloo, world size 2): the benchmark's replicas take the
slowest rank's time, and the reference arm under torchrun prints one line from rank 0."""
import json
import os
import pathlib
import subprocess
import sys

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    import torch
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [3.5, 7.25]
        got = bench.max_over_ranks(torch, dist, times[rank])
        pathlib.Path(out_dir, f"rank{rank}.txt").write_text(repr(got))
    finally:
        dist.destroy_process_group()


def _free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_slowest_rank_time_is_taken(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 7.25


def test_single_process_keeps_its_own_time():
    import torch
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(torch, None, 4.0) == 4.0


def test_reference_arm_under_torchrun_prints_once(tmp_path):
    """Two ranks of `bench.py --impl reference`: rank 0 times the oracle and prints one
    JSON line, the other rank exits 0 without work."""
    pytest.importorskip("torch.distributed.run")
    env = dict(os.environ, PYTHONPATH=str(ROOT))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(ROOT / "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=str(tmp_path), timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
