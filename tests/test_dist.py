"""Multi-process logic of bench.py on CPU (gloo, world size 2): every rank
runs its own replica, the reported time is the max over ranks, and only
rank 0 runs the reference arm."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    v = bench.max_over_ranks(10.0 + 5.0 * rank)
    w, r, lr = bench.dist_env()
    out.put((rank, v, w, r, lr))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    assert [(r[2], r[3], r[4]) for r in res] == [(2, 0, 0), (2, 1, 1)]


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload = "C1"
        steps = 2
        warmup = 1
    bench.run_reference(A())
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_line(monkeypatch, capsys):
    import json

    import bench
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)

    class A:
        workload = "C1"
        steps = 3
        warmup = 1
    bench.run_reference(A())
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us/step" and d["higher_is_better"] is False
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
