"""The multi-rank path of bench.py on CPU (gloo, world size 2): ranks meet at the barrier, the
whole-job value sums every rank's bytes over the slowest rank's time, and the reference arm runs on
rank 0 only (the other ranks exit without work). No GPU and no collective on the data path."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    d = bench.Dist(world)
    try:
        assert d.world == world and d.rank == rank
        d.barrier()
        # rank r moved (r + 1) GB in (r + 1) * 0.1 s: total 3 GB over the slowest 0.2 s
        total, t, gbs = bench.aggregate((rank + 1) * 1e9, (rank + 1) * 0.1, d)
        args = bench.parse_args(["--impl", "reference", "--gpus", str(world), "--steps", "3",
                                 "--warmup", "3"])
        ref = bench.run_reference(args, d) if rank != 0 else "rank0-not-run"
        q.put((rank, total, t, gbs, ref))
    finally:
        d.close()


@pytest.mark.timeout(120)
def test_two_rank_aggregation_with_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    results = sorted(q.get() for _ in range(world))
    for rank, total, t, gbs, ref in results:
        assert total == pytest.approx(3e9)
        assert t == pytest.approx(0.2)
        assert gbs == pytest.approx(15.0)
        if rank != 0:
            assert ref is None            # the reference arm works on rank 0 only
