"""World-size-2 gloo test (CPU) of the multi-replica timing in bench.py.

Each rank reports its own timed-region length; the job's time is the maximum over ranks and the
whole-job throughput counts the units of every rank.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, units, out):
    import sys
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_max, value = bench.aggregate_over_ranks(times[rank], units, world, torch.device("cpu"))
        out[rank] = (t_max, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(3.0, 5.0), (7.5, 2.5)])
def test_two_replicas_take_the_slowest_rank(times):
    world, units = 2, 1000
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, times, units, out), nprocs=world, join=True)
        res = dict(out)
    slowest = max(times)
    for r in range(world):
        t_max, value = res[r]
        assert t_max == slowest
        assert value == pytest.approx(units * world / (slowest * 1e-3))


def test_single_replica_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    t, v = bench.aggregate_over_ranks(4.0, 100, 1, None)
    assert t == 4.0 and v == pytest.approx(100 / 4e-3)


def test_decode_profile_traffic_tracks_the_sources(tmp_path):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    good = tmp_path / "p.md"
    good.write_text(f"- source_digest: `{bench.decode_source_digest()}`\n- traffic_bytes_per_launch: 12345\n")
    assert bench.profiled_traffic(str(good)) == 12345
    stale = tmp_path / "q.md"
    stale.write_text("- source_digest: `0000`\n- traffic_bytes_per_launch: 12345\n")
    assert bench.profiled_traffic(str(stale)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md")) is None
