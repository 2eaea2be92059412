"""Frame sharding on two gloo ranks (CPU): each rank scores its range with the
oracle and the gathered scores equal the oracle's on every frame."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

from ssimulacra2_image_scoring_gb300.shard import frame_range


@pytest.mark.parametrize("n,world", [(50, 2), (7, 3), (1, 4), (0, 2), (16, 8)])
def test_frame_range_covers_each_frame_once(n, world):
    ranges = [frame_range(n, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, b0), (a1, b1) in zip(ranges, ranges[1:]):
        assert b0 == a1
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_frame_range_rejects_bad_split():
    with pytest.raises(ValueError):
        frame_range(10, 0, 0)
    with pytest.raises(ValueError):
        frame_range(10, 2, 2)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import oracle
    import synth
    from ssimulacra2_image_scoring_gb300.shard import score_sharded
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.custom(40, 24, 8, 420, 5, seed=17)
        fn = lambda r, d: oracle.score_frames(r, d, 40, 24, 8, 420)[0]  # noqa: E731
        got = score_sharded(fn, wl.ref, wl.dis)
        q.put((rank, got.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_rank_gather_matches_single_process():
    import torch.multiprocessing as mp

    import oracle
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = synth.custom(40, 24, 8, 420, 5, seed=17)
    want, _ = oracle.score_frames(wl.ref, wl.dis, 40, 24, 8, 420)
    for r in (0, 1):
        assert np.array_equal(np.array(res[r]), want)
