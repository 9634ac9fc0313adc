"""The N > 1 launch of the benchmark on CPU: two ranks over gloo (the data path
has no collective - replicas - so what is shared between ranks is the barrier
around the timed region, the max over ranks of the measured times, and the
reference arm running on rank 0 only)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()
    try:
        d.barrier()
        v = d.max(1.5 * (rank + 1))

        class Args:
            steps, warmup, gpus = 1, 0, world

        # rank 0 would run the CPU oracle; the other ranks return at once
        ref = bench.run_reference(Args, d) if rank != 0 else "rank 0"
        d.barrier()
        q.put((rank, v, ref, d.world, d.pg is not None))
    finally:
        d.close()


def test_two_ranks_share_barrier_max_and_leave_the_reference_to_rank_0():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(2):
            rank, v, ref, world, has_pg = q.get(timeout=120)
            out[rank] = (v, ref, world, has_pg)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert set(out) == {0, 1}
    for rank, (v, ref, world, has_pg) in out.items():
        assert v == 3.0 and world == 2 and has_pg  # the max over both ranks
    assert out[1][1] is None  # the reference arm prints from rank 0 only


def test_single_rank_has_no_process_group(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()
    assert d.world == 1 and d.pg is None and d.max(2.5) == 2.5
    d.barrier()
    d.close()


def test_reference_arm_line_on_cpu(monkeypatch):
    # The reference arm times the CPU oracle on a bounded sample of the
    # shared-expert step and reports it with the same metric and config as
    # the GPU arm, plus its cpu_baseline block and a zero-copy e2e.
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()

    class Args:
        steps, warmup, gpus = 1, 0, 1

    try:
        line = bench.run_reference(Args, d)
    finally:
        d.close()
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["higher_is_better"] is True and line["dtype"] == "f64"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"] == bench.config_block(1)
