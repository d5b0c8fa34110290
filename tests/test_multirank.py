"""The N>1 path of the benchmark, as 2 gloo ranks on CPU: rank discovery from
the torchrun environment, the barrier, the max-over-ranks of the timed
region, per-rank seeds, and sharding rows across ranks (rows are
independent, so each rank's rows of a batch equal the full batch's)."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, tmpdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import bench
    import oracle
    import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    # slowest rank's time is the one reported
    assert bench.max_over_ranks(1.5 * (rank + 1), w) == 1.5 * world
    bench.barrier(w)
    # each rank draws its own batch of the same shape
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.rank_seed(1002, rank))
    assert len(set(seeds)) == world
    # rows sharded across ranks reproduce the full batch
    wl = W.make_decode("multirank", [100, 5, 64, 700, 3, 129], seed=3, table_pages=11)
    args = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    mine = list(range(rank, wl.R, world))
    out, err = oracle.decode(W.bits(wl.K0).copy(), W.bits(wl.V0).copy(), *args, wl.step_positions.numpy(),
                             wl.table.numpy(), sel=mine, nthreads=1)
    parts = [None] * world
    dist.all_gather_object(parts, (mine, out[mine]))
    if rank == 0:
        full, _ = oracle.decode(W.bits(wl.K0).copy(), W.bits(wl.V0).copy(), *args, wl.step_positions.numpy(),
                                wl.table.numpy(), nthreads=1)
        got = np.zeros_like(full)
        for rows, o in parts:
            got[rows] = o
        assert np.array_equal(got, full)
        open(os.path.join(tmpdir, "ok"), "w").write("ok")
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    import oracle
    oracle.build()   # compile once before the ranks start
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    assert (tmp_path / "ok").exists()
