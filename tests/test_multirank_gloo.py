"""The multi-rank host logic of the bench on CPU with gloo, world size 2:
each rank draws its own seeded batch, the job time is the slowest rank's,
and throughput counts every rank's tokens.  No GPU and no data-path
collective is involved (the path shards over independent batches)."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, l = bench.rank_env()
    wl = synth.Workload("mr", 16, 32, 64, 2, "bf16", 0.02, "zipf", seed=1003)
    inp = synth.make_inputs(wl, seed=bench.rank_seed(wl, r))
    t = bench.max_over_ranks(1.5 + r, w)       # rank 1 is the slow one
    q.put((r, w, l, inp.X_bits.copy(), inp.targets.copy(), t, bench.job_tokens_per_s(wl.N, w, 10, t)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_weak_scaling_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted([q.get(timeout=120) for _ in procs], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, x0, y0, t0, v0), (r1, w1, l1, x1, y1, t1, v1) = out
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert not np.array_equal(x0, x1)             # independent batches per rank
    assert t0 == t1 == 2.5                        # the slowest rank's time
    assert v0 == v1 == 2 * 16 * 10 / 2.5          # all ranks' tokens over that time
