"""The T-rank form run as T processes ("Vocab Parallelism" sec. 5.3; the
interview note's figure 2 and key formulas): each process holds one shard
W_t = W[t V/T, (t+1) V/T), runs the library's shard forward on the GPU,
all-gathers the statistics through torch.distributed (gloo), merges them,
runs its shard backward and all-reduces the fp32 dX parts
(vocab_parallel_lmhead_ce).  The parent checks every rank's loss, lse, mean,
n_bad and dX, and the stacked dW_t, against the oracle.

The processes share this machine's one GPU.  Every rank's kernels complete
before its collective is issued, and the collectives run on the host (gloo),
so no kernel ever waits on another rank's; the processes use spawn."""
import datetime
import os
import socket

import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
from gpu_util import (assert_grads_elementwise, assert_loss_close, assert_lse_close, grad_tol, rel_fro)

pytestmark = pytest.mark.gpu

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

CASES = [  # N, H, V, T (= ranks), dtype, seed
    (300, 128, 1000, 2, "bf16", 71),    # V/T = 500: the shard edge inside a 256-wide tile
    (77, 40, 99, 3, "f32", 72),
]


def _inputs(case):
    N, H, V, T, dtype, seed = case
    inp = synth.small_case(N, H, V, T, dtype, seed=seed, ignore_frac=0.1)
    inp.targets[:2] = [V, -7]           # out of range: ignored and counted
    return inp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, case, port, q):
    import sys
    for p in (ROOT, TESTS):
        if p not in sys.path:
            sys.path.insert(0, p)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        import torch.distributed as dist

        import vocab_lm_head_vp_b300 as vp
        from gpu_util import dev_inputs, np64

        N, H, V, T, dtype, _ = case
        dist.init_process_group("gloo", rank=rank, world_size=T, timeout=datetime.timedelta(seconds=180))
        X, W, y = dev_inputs(_inputs(case), "cuda:0")
        Vs = V // T
        fwd, dX, dW_t = vp.vocab_parallel_lmhead_ce(X, W[rank * Vs:(rank + 1) * Vs], y, V, T, rank)
        torch.cuda.synchronize()
        q.put((rank, np64(fwd["loss"]), np64(fwd["lse"]), float(fwd["mean"].item()), int(fwd["n_bad"].item()),
               np64(dX), np64(dW_t)))
        dist.barrier()
        dist.destroy_process_group()
    except BaseException as e:   # reported to the parent, which fails the test
        q.put((rank, "error", repr(e)))
        raise


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[3]}-{c[4]}")
def test_ranks_as_processes_match_the_oracle(case):
    import torch.multiprocessing as mp

    N, H, V, T, dtype, _ = case
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, case, port, q)) for r in range(T)]
    for p in procs:
        p.start()
    try:
        out = [q.get(timeout=300) for _ in procs]
    finally:
        for p in procs:
            p.join(timeout=120)
            if p.is_alive():
                p.kill()
                p.join()
    errors = [o for o in out if isinstance(o[1], str)]
    assert not errors, errors
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    out.sort(key=lambda o: o[0])

    inp = _inputs(case)
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, V, T)
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, V)
    for rank, loss, lse, mean, n_bad, dX, _ in out:
        # every rank merges the same gathered statistics with the same kernel
        assert np.array_equal(loss, out[0][1]) and np.array_equal(lse, out[0][2]), rank
        assert_loss_close(loss, o["loss"], dtype, what=f"loss (rank {rank})")
        assert_lse_close(lse, o["lse"], inp, what=f"lse (rank {rank})")
        assert_loss_close([mean], [o["mean"]], dtype, what=f"mean (rank {rank})")
        assert n_bad == o["n_bad"] == 2
        assert rel_fro(dX, b["dX"]) <= grad_tol(dtype), rank
    dW = np.concatenate([r[6] for r in out])          # the shards' dW_t in rank order
    assert rel_fro(dW, b["dW"]) <= grad_tol(dtype)
    assert_grads_elementwise(inp, torch.from_numpy(out[0][5]), torch.from_numpy(dW), b)
