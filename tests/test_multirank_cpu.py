"""The benchmark's multi-rank logic on CPU: world size 2 over gloo.  Every
rank runs its own replica of the workload (weak scaling, no data-path
collective); the reported time is the max over ranks and the value counts
the work of all ranks."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    ws, r = bench.init_dist("gloo")
    assert (ws, r) == (world, rank)
    # rank r "took" (r + 1) * 10 ms for its replica
    t = bench.reduce_max((rank + 1) * 10.0)
    bench.barrier()
    v = bench.whole_job_tflops(1e12, ws, t / 1e3)
    out.put((rank, t, v))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time (20 ms); 2 x 1 TFLOP in 20 ms = 100 TFLOP/s
    assert [r[1] for r in res] == [20.0, 20.0]
    assert all(abs(r[2] - 100.0) < 1e-9 for r in res)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_tflops(2e12, 1, 0.5) == 4.0
