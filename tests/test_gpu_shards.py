"""The T-rank form's building blocks on one GPU: each shard's call sees only
its rows W_t = W[t V/T, (t+1) V/T) and the ranks run one after another (no
kernel waits on another).  The shards' statistics, gathered in rank order,
merge into the oracle's loss and lse; the shards' fp32 dX parts sum to the
oracle's dX and their dW_t stack into its dW ("Vocab Parallelism" sec.
5.3.1-5.3.2; the interview note's figure 2 and key formulas)."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import (assert_grads_elementwise, assert_loss_close, assert_lse_close, assert_stats_close, dev_inputs, grad_tol, np64,
                      rel_fro)
from test_gpu_ce import _argmax_case

pytestmark = pytest.mark.gpu
IGN = -100


def _emulate(inp, T, ignore_index=IGN):
    """The T ranks' calls in sequence; the all-gather is a stack in rank order
    and the all-reduce a sum over ranks, both in fp32."""
    X, W, y = dev_inputs(inp)
    V = inp.wl.V
    Vs = V // T
    stats = torch.stack([vp.lmhead_ce_shard_fwd(X, W[t * Vs:(t + 1) * Vs], y, V, T, t, ignore_index)
                         for t in range(T)])
    fwd = vp.lmhead_ce_merge_stats(stats, y, V, T, ignore_index)
    dX = torch.zeros(X.shape, dtype=torch.float32, device=X.device)
    dWs = []
    for t in range(T):
        dX_t, dW_t = vp.lmhead_ce_shard_bwd(X, W[t * Vs:(t + 1) * Vs], y, fwd["lse"], V, T, t, ignore_index)
        dX += dX_t
        dWs.append(dW_t)
    torch.cuda.synchronize()
    return stats, fwd, dX, torch.cat(dWs)


CASES = [  # N, H, V, T, dtype
    (300, 200, 1000, 4, "bf16"),     # V/T = 250: every shard's tiles start off the 256 grid
    (257, 136, 770, 7, "bf16"),
    (130, 64, 520, 2, "bf16"),
    (40, 64, 512, 16, "bf16"),       # V/T = 32: one partial tile per shard
    (77, 40, 99, 3, "f32"),
    (200, 96, 640, 10, "f32"),
]


@pytest.mark.parametrize("N,H,V,T,dtype", CASES)
def test_shards_match_the_oracle(N, H, V, T, dtype):
    inp = synth.small_case(N, H, V, T, dtype, seed=N + V + T, ignore_frac=0.1)
    inp.targets[:3] = [V, -5, V + 7]     # out of range: ignored and counted
    stats, fwd, dX, dW = _emulate(inp, T)
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, V, T)
    st = np64(stats)
    st[:, 1] += 1.0                      # R_t -> S_t = 1 + R_t, the oracle's statistic
    assert_stats_close(st, o["shard_stats"], inp, T)
    assert_lse_close(np64(fwd["lse"]), o["lse"], inp)
    assert_loss_close(np64(fwd["loss"]), o["loss"], dtype, what="loss")
    assert_loss_close(np64(fwd["mean"]), [o["mean"]], dtype, what="mean")
    assert int(fwd["n_bad"].item()) == o["n_bad"] == 3
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, V)
    tol = grad_tol(dtype)
    assert rel_fro(np64(dX), b["dX"]) <= tol and rel_fro(np64(dW), b["dW"]) <= tol
    assert_grads_elementwise(inp, dX, dW, b)


@pytest.mark.parametrize("dtype,V", [("f32", 192), ("bf16", 512)])
def test_shards_keep_tiny_losses(dtype, V):
    """Targets that are the row's maximum by a wide margin (loss 1e-7..1e-3):
    the shards exchange R_t, not S_t, so the merged loss keeps rel 1e-5."""
    inp = _argmax_case(300, V, dtype, seed=V + 4)
    _, fwd, _, _ = _emulate(inp, 4)
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, V, 4)
    assert_loss_close(np64(fwd["loss"]), o["loss"], "f32", what="loss")


def test_shards_agree_with_the_one_call_form():
    """The MiniMind workload: the T = 2 ranks' merged loss and lse against the
    single call over the whole vocabulary (same arithmetic, tile boundaries at
    each shard's start instead of the vocabulary's), and the gradients."""
    inp = synth.make_inputs("minimind")
    wl = inp.wl
    stats, fwd, dX, dW = _emulate(inp, wl.T)
    X, W, y = dev_inputs(inp)
    one = vp.lmhead_ce_fwd_bwd(X, W, y, wl.T)
    torch.cuda.synchronize()
    np.testing.assert_allclose(np64(fwd["loss"]), np64(one["loss"]), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(np64(fwd["lse"]), np64(one["lse"]), rtol=1e-6, atol=1e-6)
    assert rel_fro(np64(dX), np64(one["dX"])) <= 5e-3 and rel_fro(np64(dW), np64(one["dW"])) <= 5e-3
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, wl.V, wl.T)
    assert_loss_close(np64(fwd["loss"]), o["loss"], "bf16")
