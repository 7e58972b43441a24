"""Host logic of the multi-rank bench path on CPU: world_size 2 over gloo.

Ranks hold independent batches (sequences never exchange data), so the only
cross-rank steps are the max-over-ranks timing and the whole-job throughput."""
import os
import socket

import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    elapsed = [10.0, 12.5][rank]
    m = bench.max_over_ranks(elapsed)
    out[rank] = (m, bench.whole_job_throughput(256 * 100, world, m))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo_world2():
    ctx = tmp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 12.5
    assert abs(out[0][1] - 2 * 256 * 100 / 12.5e-3) < 1e-6


def test_single_process_identity():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_throughput(256, 1, 1.0) == 256000.0
