"""The multi-rank host logic of bench.py on CPU: two gloo ranks, launched
like torchrun would (RANK / WORLD_SIZE / LOCAL_RANK / MASTER_* in the
environment).  The job time is the slowest rank's, the throughput counts
every rank's rows (weak-scaling replicas), and the reference arm runs on
rank 0 only."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        w, r, local = bench._dist()
        total = bench._max_over_ranks(1.5 + rank, w, "cpu")   # rank 1 is the slower one
        value = bench._job_rows_per_s(w, 256, 10, total)
        dist.barrier()
        q.put((r, w, local, total, value))
    finally:
        dist.destroy_process_group()


def test_bench_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    for r, (rank, ws, local, total, value) in enumerate(got):
        assert (rank, ws, local) == (r, 2, r)
        assert total == 2.5                              # the max over ranks, on every rank
        assert value == pytest.approx(2 * 256 * 10 / 2.5)


def _reference_rank(rank, ws, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import contextlib
    import io
    import types
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(types.SimpleNamespace(steps=1, warmup=0, gpus=ws))
    q.put((rank, buf.getvalue()))


def test_reference_arm_prints_on_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_reference_rank, args=(r, 2, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs)
    out = dict(q.get(timeout=5) for _ in range(2))
    assert '"impl": "reference"' in out[0] and out[0].count("\n") == 1
    assert out[1] == ""
