"""Parity at the full workload sizes, in the launch configuration the bench
times (one vocab chunk): the oracle recomputes sampled token rows one at a
time (loss, lse, dX rows) and sampled vocab rows of dW; dW is also checked
through identities that hold at any size, and in full at the V32k shape with
fewer tokens.  Gradient entries are compared one by one against the bound of
gpu_util.assert_grads_elementwise, besides the per-tensor tolerance."""
import gc

import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import (abs_matmul, assert_grads_elementwise, assert_loss_close, assert_within, dev_inputs,
                      elementwise_u, np64, rel_fro, term_magnitudes)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("name", ["v32k", "v128k", "v152k"])
def test_fullsize_sampled_rows(name, path):
    """``split``: vp_lmhead_ce_fwd + vp_lmhead_ce_bwd; ``fused``:
    vp_lmhead_ce_fwd_bwd (the call the bench times), all tokens in one chunk."""
    inp = synth.make_inputs(name)
    wl = inp.wl
    X, W, y = dev_inputs(inp)
    if path == "split":
        f = vp.lmhead_ce_fwd(X, W, y, wl.T)
        dX, dW = vp.lmhead_ce_bwd(X, W, y, f["lse"], wl.T)
    else:
        f = vp.lmhead_ce_fwd_bwd(X, W, y, wl.T)
        dX, dW = f["dX"], f["dW"]
    torch.cuda.synchronize()
    assert vp.read_device_status(f["workspace"]) == 0
    valid = (inp.targets >= 0) & (inp.targets < wl.V)
    n_valid = int(valid.sum())
    assert int(f["n_bad"].item()) == 0
    rng = np.random.default_rng(99)
    rows = np.sort(rng.choice(wl.N, 24, replace=False))
    o = ref.lmhead_ce_rows(inp.X, inp.W, inp.targets, rows, n_valid)
    rt = torch.from_numpy(rows).cuda()
    assert_loss_close(np64(f["lse"][rt]), o["lse"], "bf16", what="lse")
    assert_loss_close(np64(f["loss"][rt]), o["loss"], "bf16", scale=o["lse"], what="loss")
    e = rel_fro(np64(dX[rt]), o["dX"])
    assert e <= 2e-2, f"dX sampled rows rel Frobenius {e:.3e}"
    M = term_magnitudes(o["dZ"], o["g"], inp.targets[rows])
    assert_within("dX rows", np64(dX[rt]), o["dX"], elementwise_u("bf16") * abs_matmul(M, inp.W))
    # mean over valid tokens is the mean of the per-token losses
    loss = np64(f["loss"])
    assert abs(float(f["mean"].item()) - loss.sum() / n_valid) <= 1e-5 * abs(loss.sum() / n_valid)
    # dW identities: sum_v dW[v,:] = 0 (dZ rows sum to 0); <dW, W> = <dX, X> (= <dZ, Z>)
    dWd = dW.double()
    # bf16 rounding of dZ leaves |sum_v dZ[n,v]| ~ 2^-9 |dZ[n]|, i.e. a column-sum
    # norm ~ 2e-3 |dW|; a dropped or misplaced onehot term gives ~ |dW|
    colsum = dWd.sum(0).norm().item()
    assert colsum <= 1e-2 * dWd.norm().item(), (colsum, dWd.norm().item())
    a = (dWd * W.double()).sum().item()
    b = (dX.double() * X.double()).sum().item()
    assert abs(a - b) <= 2e-2 * max(abs(a), abs(b)) + 1e-6, (a, b)


@pytest.mark.parametrize("path", ["split", "fused"])
def test_v32k_shape_full_gradients(path):
    """H=4096, V=32000, T=4 with 512 tokens: every loss and every dX/dW entry."""
    inp = synth.make_inputs("v32k", N=512)
    wl = inp.wl
    X, W, y = dev_inputs(inp)
    if path == "split":
        f = vp.lmhead_ce_fwd(X, W, y, wl.T, shard_stats=True)
        dX, dW = vp.lmhead_ce_bwd(X, W, y, f["lse"], wl.T)
    else:
        f = vp.lmhead_ce_fwd_bwd(X, W, y, wl.T, shard_stats=True)
        dX, dW = f["dX"], f["dW"]
    torch.cuda.synchronize()
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, wl.V, wl.T)
    assert_loss_close(np64(f["loss"]), o["loss"], "bf16", scale=o["lse"])
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, wl.V)
    ex, ew = rel_fro(np64(dX), b["dX"]), rel_fro(np64(dW), b["dW"])
    assert ex <= 2e-2 and ew <= 2e-2, (ex, ew)
    assert_grads_elementwise(inp, dX, dW, b)


def test_fused_full_size_repeatable():
    """Two fused calls at the V32k shape (all tokens) give bit-identical loss,
    dX and dW: no atomics in any reduction of the path."""
    inp = synth.make_inputs("v32k")
    wl = inp.wl
    X, W, y = dev_inputs(inp)
    a = vp.lmhead_ce_fwd_bwd(X, W, y, wl.T)
    b = vp.lmhead_ce_fwd_bwd(X, W, y, wl.T)
    torch.cuda.synchronize()
    for k in ("loss", "lse", "mean", "dX", "dW"):
        assert torch.equal(a[k], b[k]), k


def test_v128k_fused_every_token_and_sampled_dw_rows():
    """The bench's workload through the fused call it times: every token's loss
    and lse against the oracle's (all 16384 rows in float64, row batches), and
    dW rows of sampled vocab ids -- the most frequent Zipf targets, random ids,
    never-targeted ones -- against the oracle's own columns of the logit
    gradient."""
    inp = synth.make_inputs("v128k")
    wl = inp.wl
    X, W, y = dev_inputs(inp)
    o = vp.lmhead_ce_fwd_bwd(X, W, y, wl.T)
    torch.cuda.synchronize()
    assert vp.read_device_status(o["workspace"]) == 0
    valid = (inp.targets >= 0) & (inp.targets < wl.V)
    n_valid = int(valid.sum())
    parts = [ref.lmhead_ce_rows(inp.X, inp.W, inp.targets, np.arange(a, min(a + 2048, wl.N)), n_valid,
                                with_dx=False) for a in range(0, wl.N, 2048)]
    lse = np.concatenate([p["lse"] for p in parts])
    loss = np.concatenate([p["loss"] for p in parts])
    assert_loss_close(np64(o["lse"]), lse, "bf16", what="lse")
    assert_loss_close(np64(o["loss"]), loss, "bf16", scale=lse, what="loss")
    rng = np.random.default_rng(123)
    counts = np.bincount(inp.targets[valid], minlength=wl.V)
    never = np.flatnonzero(counts == 0)
    rows = np.unique(np.concatenate([np.arange(8), rng.choice(wl.V, 32, replace=False),
                                     rng.choice(never, 8, replace=False)]))
    want, dZv, g = ref.lmhead_ce_dw_rows(inp.X, inp.W, inp.targets, lse, rows, n_valid, return_dz=True)
    got = np64(o["dW"][torch.from_numpy(rows).cuda()])
    M = term_magnitudes(dZv, g, inp.targets, cols=rows)
    assert_within("dW rows", got, want, elementwise_u("bf16") * abs_matmul(M.T, inp.X))
    e = rel_fro(got, want)
    assert e <= 2e-2, f"dW sampled rows rel Frobenius {e:.3e}"
    # the frequent ids' rows carry the one-hot term: each is checked on its own too
    for k in range(8):
        ek = rel_fro(got[k], want[k])
        assert ek <= 2e-2, (int(rows[k]), ek)
