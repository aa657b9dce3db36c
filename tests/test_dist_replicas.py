"""The benchmark's multi-process path, run as two gloo ranks on CPU.

Every rank runs its own verify step (replicas: the step has no exchange), so
the only cross-rank operations are a barrier and the maximum of the ranks'
timings; the whole-job value counts every rank's bytes over the slowest
rank's time.  The reference arm runs on rank 0 alone.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                          WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
        sys.path.insert(0, ROOT)
        import bench
        import torch.distributed as dist
        w, r, local = bench.dist_setup()
        assert dist.get_backend() == "gloo"
        bench.dist_barrier(w)
        slowest = bench.dist_max(w, 1.5 + rank)        # rank-dependent step times (ms)
        q.put((r, w, local, slowest))
        dist.destroy_process_group()
    except Exception as e:   # reported to the test
        q.put((rank, "error", repr(e), None))


def _cuda_visible() -> bool:
    import torch
    return torch.cuda.is_available()


@pytest.mark.skipif(_cuda_visible(), reason="with a GPU the ranks would use NCCL; this is the CPU (gloo) path")
def test_two_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.terminate()
    assert all(p.exitcode == 0 for p in procs)
    assert got == [(0, 2, 0, 2.5), (1, 2, 1, 2.5)]


def test_whole_job_value_counts_every_rank_over_the_slowest():
    sys.path.insert(0, ROOT)
    import bench
    b = 4_266_327_040
    assert bench.whole_job_gbs(1, b, 2.5) == pytest.approx(b / 2.5e-3 / 1e9)
    assert bench.whole_job_gbs(4, b, 2.5) == pytest.approx(4 * bench.whole_job_gbs(1, b, 2.5))


def test_reference_arm_does_nothing_off_rank_zero(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.argparse.Namespace(steps=1, warmup=0, ref_seconds=1.0, gpus=2)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
