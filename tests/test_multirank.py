"""The N>1 path of bench.py on CPU: two gloo ranks (world size 2) run the same aggregation the
bench uses (barrier, maximum of the per-rank times, whole-job throughput), and the reference arm's
non-zero ranks exit without work."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    ms = [3.0, 5.0][rank]
    m = bench.reduce_max(ms, world)
    v = bench.whole_job_tflops(2.0e12, 10, world, m)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, m, v))


def test_two_gloo_ranks_take_the_max_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in got:
        assert m == 5.0
        assert v == pytest.approx(2 * 2.0e12 * 10 / 5e-3 / 1e12)


def test_world_one_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(4.5, 1) == 4.5
    assert bench.whole_job_tflops(1e12, 2, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 1, 3, 2
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
