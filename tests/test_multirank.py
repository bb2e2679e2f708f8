"""The multi-rank host path of bench.py on CPU (gloo, world size 2): every
rank gets its own sequences (same shapes, its own seed), and the job's time
is the slowest rank's, its rate the queries of all ranks over that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    import synth
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        w = bench.rank_workload(synth.CONFIGS[1].with_(n=512, planted=4), rank)
        ms, rate = bench.job_rate(1.0 + rank, queries_per_rank=3, world=world)
        x = synth.make(w)
        out[rank] = (w.seed, ms, rate, float(x["k"][0, 0, 5].astype("float64").sum()),
                     tuple(x["k"].shape))
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_the_slowest_time_and_own_their_sequences():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    (s0, ms0, r0, k0, sh0), (s1, ms1, r1, k1, sh1) = res[0], res[1]
    assert ms0 == ms1 == pytest.approx(2.0)          # max over ranks
    assert r0 == r1 == pytest.approx(3 * 2 / 2e-3)   # all ranks' queries / job time
    assert s0 != s1 and k0 != k1 and sh0 == sh1      # own seeds, same shapes
