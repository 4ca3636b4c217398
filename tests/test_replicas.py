"""The N > 1 path of bench.py: independent replicas, one per rank (the product
has no exchange step).  Its host logic -- the slowest rank's time on every
rank, the whole-job throughput, one JSON line from rank 0 -- runs here as two
gloo ranks on the CPU; the reference arm's other ranks exit 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    import contextlib
    import io

    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)  # rank 1 is the slow one
        value = bench.whole_job_value(world, 2.0 * 512 * 5120 * 5120, slowest / 4)
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            printed = bench.emit({"value": value, "n_gpus": world}, rank)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value, "printed": printed, "stdout": buf.getvalue()}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_agree_on_the_slowest_rank(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["slowest"] == r1["slowest"] == 15.0
    # two replicas' work over the slowest step: 2 x 26.8 G ops / 3.75 ms
    assert r0["value"] == pytest.approx(2 * 2.0 * 512 * 5120 * 5120 / 3.75e-3 / 1e12)
    assert r0["printed"] and json.loads(r0["stdout"])["n_gpus"] == 2
    assert not r1["printed"] and r1["stdout"] == ""


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_value(1, 1e12, 1000.0) == pytest.approx(1.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
