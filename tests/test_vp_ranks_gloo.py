"""The T-rank exchange of vocab_parallel_lmhead_ce on CPU ranks (gloo, world
size 2): each rank holds its shard W_t, its statistics are all-gathered in
rank order, every rank merges the same [T, 3, N] and gets the dense loss and
lse, and the all-reduce of the dX parts gives the dense dX while dW_t stays
local.  The shard kernels need a GPU, so here the library's three shard calls
are replaced in each rank by float64 stand-ins written from the oracle; what
runs for real is the rank function's choreography of the two collectives.
On hardware this path is unmeasured (every box here has one GPU)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

V, T, N, H = 24, 2, 7, 8
IGN = -100


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((N, H)) * 2.0
    W = rng.standard_normal((V, H))
    y = rng.integers(0, V, N)
    y[3] = IGN
    return X, W, y


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle.ref as ref
    import vocab_lm_head_vp_b300 as vp

    def shard_fwd(X, W_t, targets, V_, T_, t, ignore_index=IGN, **_):
        Vs = V_ // T_
        Zt = ref.logits(X.numpy(), W_t.numpy())
        s = ref.shard_local_stats(Zt, targets.numpy() - t * Vs, Vs, 1, ignore_index - t * Vs)[0]
        s[1] -= 1.0                                 # the exchanged statistic is R_t = S_t - 1
        return torch.from_numpy(s)

    def merge_stats(stats, targets, V_, T_, ignore_index=IGN, **_):
        st = stats.numpy().copy()
        st[:, 1] += 1.0
        mg = ref.merge_local_stats(st)
        valid, _ = ref.target_masks(targets.numpy(), V_, ignore_index)
        loss = np.where(valid, mg["lse"] - mg["z_y"], 0.0)
        return {"loss": torch.from_numpy(loss), "lse": torch.from_numpy(mg["lse"]),
                "gathered": stats.clone()}

    def shard_bwd(X, W_t, targets, lse, V_, T_, t, ignore_index=IGN, dmean=None, **_):
        Vs = V_ // T_
        y = targets.numpy()
        Zt = ref.logits(X.numpy(), W_t.numpy())
        g = ref.upstream_scale(y, V_, ignore_index)
        local = np.where((y >= t * Vs) & (y < (t + 1) * Vs), y - t * Vs, -1)
        dZ = ref.grad_logits(Zt, local, lse.numpy(), g)
        dX, dW = ref.lmhead_grads(X.numpy(), W_t.numpy(), dZ)
        return torch.from_numpy(dX), torch.from_numpy(dW)

    vp.lmhead_ce_shard_fwd, vp.lmhead_ce_merge_stats, vp.lmhead_ce_shard_bwd = shard_fwd, merge_stats, shard_bwd
    dist.init_process_group("gloo", rank=rank, world_size=world)
    X, W, y = _inputs()
    Vs = V // T
    fwd, dX, dW_t = vp.vocab_parallel_lmhead_ce(torch.from_numpy(X), torch.from_numpy(W[rank * Vs:(rank + 1) * Vs]),
                                                torch.from_numpy(y), V, T, rank)
    q.put((rank, fwd["loss"].numpy(), fwd["lse"].numpy(), fwd["gathered"].numpy(), dX.numpy(), dW_t.numpy()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_exchange():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, T, port, q)) for r in range(T)]
    for p in procs:
        p.start()
    out = sorted([q.get(timeout=120) for _ in procs], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle.ref as ref
    X, W, y = _inputs()
    o = ref.lmhead_ce_forward(X, W, y, V, T)
    b = ref.lmhead_ce_backward(X, W, y, V)
    Vs = V // T
    for rank, loss, lse, gathered, dX, dW_t in out:
        np.testing.assert_allclose(loss, o["loss"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, o["lse"], rtol=1e-12)
        st = gathered.copy()
        st[:, 1] += 1.0
        np.testing.assert_allclose(st, o["shard_stats"], rtol=1e-12, atol=1e-12)   # [T, 3, N] in rank order
        np.testing.assert_allclose(dX, b["dX"], rtol=1e-12, atol=1e-12)             # the all-reduced dX
        np.testing.assert_allclose(dW_t, b["dW"][rank * Vs:(rank + 1) * Vs], rtol=1e-12, atol=1e-12)
