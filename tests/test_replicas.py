"""The multi-GPU path of bench.py is replicas only: N independent sessions,
a gloo barrier around the timed region and the max over ranks of the time.
This runs that host logic as world_size-2 gloo ranks on the CPU."""
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


def _rank(rank, ws, port, ms_by_rank, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        assert bench.dist_info() == (ws, rank, rank)
        dist.barrier()
        ms, value = bench.combine_replicas(ms_by_rank[rank], ws)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ws, port = 2, _free_port()
    ms_by_rank = [17.5, 19.25]
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(ws, port, ms_by_rank, out), nprocs=ws, join=True)
        res = dict(out)
    import bench
    for r in range(ws):
        ms, value = res[r]
        assert ms == max(ms_by_rank)
        assert value == pytest.approx(ws * bench.DECODE / (max(ms_by_rank) * 1e-3))


def test_single_rank_needs_no_process_group():
    import bench
    ms, value = bench.combine_replicas(20.0, 1)
    assert ms == 20.0 and value == pytest.approx(bench.DECODE / 0.02)
