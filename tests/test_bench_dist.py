"""The benchmark's multi-rank host logic on CPU: world size 2 over gloo.

Each rank is an independent replica; the only cross-rank steps are the
barriers around the timed region and the max over ranks of the elapsed time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        bench.barrier(w)
        got = bench.reduce_max(10.0 + 5.0 * r, w)
        q.put((r, lr, w, got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [x[0] for x in res] == [0, 1]
    assert all(x[2] == 2 for x in res)
    assert all(x[3] == 15.0 for x in res)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)


@pytest.mark.parametrize("vis,rank,want", [(None, 0, "0"), ("3", 0, "3"), ("2,5", 1, "5"),
                                           ("GPU-abc", 0, "GPU-abc")])
def test_smi_index(monkeypatch, vis, rank, want):
    import bench
    if vis is None:
        monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    else:
        monkeypatch.setenv("CUDA_VISIBLE_DEVICES", vis)
    assert bench.smi_index(rank) == want


def test_probe_mhz_from_two_clock_probes():
    """The timed region's SM clock from two probe records {timer ns, clock64, SM id, claim}."""
    import bench
    # 2.07e9 cycles in 1 s on SM 5
    assert bench.probe_mhz([1_000_000_000, 10, 5, 1, 2_000_000_000, 10 + 2_070_000_000, 5, 1]) == 2070.0
    assert bench.probe_mhz([0, 0, 5, 1, 1000, 1500, 6, 1]) is None      # different SMs: counters differ
    assert bench.probe_mhz([0, 0, 5, 0, 1000, 1500, 5, 1]) is None      # a probe that never ran
    assert bench.probe_mhz([1000, 0, 5, 1, 1000, 1500, 5, 1]) is None   # no time elapsed
