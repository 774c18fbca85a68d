"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): replicas share
nothing on the data path; only the step times meet, maxed over the ranks, and the
reference arm runs on rank 0 alone."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # each replica timed its own sweep; the job's time is the slowest one
    t = bench.max_over_ranks(torch, dist, 0.25 * (rank + 1), world)
    t1 = bench.max_over_ranks(torch, dist, 3.0 - rank, world)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, t, t1))


def test_max_over_ranks_with_gloo():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 0.5, 3.0), (1, 0.5, 3.0)]


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(None, None, 1.25, 1) == 1.25


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    """Under torchrun only rank 0 runs and prints the reference line."""
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(bench.parse())
    assert buf.getvalue() == ""


@pytest.mark.timeout(300)
def test_reference_arm_rank0_prints_one_line(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(bench.parse())
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    """roofline.traffic is read from a profiles/ record only while the kernel's sources
    still hash to the value recorded with the counters."""
    import hashlib

    sys.path.insert(0, ROOT)
    import bench

    csrc = tmp_path / "bit_q4_weight_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1\n")
    (csrc / "common.cuh").write_text("helpers\n")
    h = hashlib.sha256(b"kernel v1\n" + b"helpers\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "t.md").write_text(f"<!-- traffic kernel=k_kernel sources=k.cu,common.cuh sha256_16={h} "
                               "bytes_per_launch=12345 -->\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k_kernel") == 12345
    assert bench.profiled_traffic("other_kernel") is None
    (csrc / "k.cu").write_text("kernel v2\n")  # the kernel changed since the capture
    assert bench.profiled_traffic("k_kernel") is None
