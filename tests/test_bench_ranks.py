"""The bench's multi-replica accounting, on CPU: two gloo ranks (127.0.0.1)
report different step times; both take the slowest rank's time, and the
job's throughput counts both ranks' bytes over it.  Also the check that
--gpus matches the launcher's WORLD_SIZE."""
import importlib.util
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    ms = b.max_over_ranks([3.0, 5.0][rank], dist, "cpu")
    dist.barrier()
    q.put((rank, ms, b.job_gbs(4.0e9, world, ms)))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [5.0, 5.0]
    assert out[0][2] == out[1][2] == pytest.approx(2 * 4.0e9 / 5e-3 / 1e9)


def test_one_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(3.0, None, "cpu") == 3.0
    assert b.job_gbs(4.0e9, 1, 2.0) == pytest.approx(2000.0)


def test_gpus_flag_must_match_world_size(monkeypatch):
    b = _bench()
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        b.dist_setup(4)
    assert b.dist_setup(2)[1] == 2
