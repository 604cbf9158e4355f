"""Multi-process host logic of bench.py on CPU (gloo, world size 2): rendezvous,
barriers, the max-over-ranks timing reduction, per-rank batches, and the
reference arm running on rank 0 only."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    r, wsz = bench.dist_init("gloo")
    bench.barrier()
    m = bench.max_over_ranks(1.5 + rank)
    seed = bench.rank_batch_seed(10, rank)
    args = bench.parse_args(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "3"])
    rr, res = bench.run_reference(args)
    bench.barrier()
    out.put((r, wsz, m, seed, res is not None))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_gloo_plumbing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    assert all(r[1] == 2 for r in results)
    assert all(r[2] == 2.5 for r in results)          # max over ranks
    assert results[0][3] != results[1][3]             # distinct batches per rank
    assert results[0][4] is True and results[1][4] is False  # reference arm: rank 0 only
