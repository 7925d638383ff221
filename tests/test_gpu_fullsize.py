"""Parity at every workload's full size, for both LM-head paths and for every
shard count T in {1, 2, the workload's T, 16} (each divides V), in the launch
configuration the bench times (the library's default, bounded workspaces).

- MiniMind (N=4096, H=512, V=6400) and V32k (N=8192, H=4096, V=32000): every
  token's loss and lse, every shard statistic, and every dX and dW entry.
- V128k (N=16384, H=4096, V=128256) and V152k (N=32768, H=5120, V=151936, 10%
  of positions ignore_index): every token's loss and lse (float64 oracle over
  all rows, in row batches), 256 sampled dX rows, and dW rows of the 8 most
  frequent, 32 random and 8 never-targeted vocab ids; ignored positions give a
  zero loss and zero dX rows; dW identities that hold at any size.

The oracle is computed once per workload (it does not depend on T or on the
path).  Gradient entries are held to the elementwise bound of
gpu_util.assert_grads_elementwise as well as the per-tensor tolerance."""
import gc

import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import (abs_matmul, assert_loss_close, assert_stats_close, assert_within, dev_inputs, elementwise_u,
                      np64, rel_fro, term_magnitudes, with_p16_floor)

pytestmark = pytest.mark.gpu
IGN = -100
SHARDS = {"minimind": (1, 2, 16), "v32k": (1, 2, 4, 16), "v128k": (1, 2, 8, 16), "v152k": (1, 2, 8, 16)}
# "_all": one chunk (all N tokens' probabilities, or all V ids' dZ, held at once), at the workload's own T
CASES = [(name, T, path) for name, ts in SHARDS.items() for T in ts for path in ("fused", "split")]
CASES = CASES[:CASES.index(("v128k", 16, "split")) + 1] + [("v128k", 8, "fused_all"), ("v128k", 8, "split_all")] \
    + CASES[CASES.index(("v128k", 16, "split")) + 1:]
_CACHE = {}


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _dense(name):
    """MiniMind / V32k: the whole oracle, and the elementwise gradient bounds."""
    inp = synth.make_inputs(name)
    wl = inp.wl
    Z = ref.logits(inp.X, inp.W)
    fwd = ref.cross_entropy(Z, inp.targets)
    stats = {T: ref.shard_local_stats(Z, inp.targets, wl.V, T) for T in SHARDS[name]}
    g = ref.upstream_scale(inp.targets, wl.V)
    dZ = ref.grad_logits(Z, inp.targets, fwd["lse"], g)
    del Z
    dX, dW = ref.lmhead_grads(inp.X, inp.W, dZ)
    M = with_p16_floor(term_magnitudes(dZ, g, inp.targets), g, "bf16")
    del dZ
    u = elementwise_u("bf16")
    bx, bw = u * abs_matmul(M, inp.W), u * abs_matmul(M.T, inp.X)
    return {"inp": inp, "fwd": fwd, "stats": stats, "dX": dX, "dW": dW, "bx": bx, "bw": bw}


def _sampled(name):
    """V128k / V152k: every token's loss and lse; sampled dX and dW rows."""
    inp = synth.make_inputs(name)
    wl = inp.wl
    valid, _ = ref.target_masks(inp.targets, wl.V)
    n_valid = int(valid.sum())
    parts = [ref.lmhead_ce_rows(inp.X, inp.W, inp.targets, np.arange(a, min(a + 2048, wl.N)), n_valid,
                                with_dx=False) for a in range(0, wl.N, 2048)]
    lse = np.concatenate([p["lse"] for p in parts])
    loss = np.concatenate([p["loss"] for p in parts])
    rng = np.random.default_rng(99)
    rows = np.sort(rng.choice(wl.N, 256, replace=False))
    o = ref.lmhead_ce_rows(inp.X, inp.W, inp.targets, rows, n_valid)
    u = elementwise_u("bf16")
    Mx = with_p16_floor(term_magnitudes(o["dZ"], o["g"], inp.targets[rows]), o["g"], "bf16")
    counts = np.bincount(inp.targets[valid], minlength=wl.V)
    never = np.flatnonzero(counts == 0)
    vrows = np.unique(np.concatenate([np.argsort(-counts, kind="stable")[:8], rng.choice(wl.V, 32, replace=False),
                                      rng.choice(never, 8, replace=False)]))
    want_w, dZv, g = ref.lmhead_ce_dw_rows(inp.X, inp.W, inp.targets, lse, vrows, n_valid, return_dz=True)
    Mw = with_p16_floor(term_magnitudes(dZv, g, inp.targets, cols=vrows), g, "bf16")
    return {"inp": inp, "lse": lse, "loss": loss, "mean": float(loss.sum()) / max(1, n_valid),
            "n_valid": n_valid, "rows": rows, "dX_rows": o["dX"], "bx": u * abs_matmul(Mx, inp.W),
            "vrows": vrows, "dW_rows": want_w, "bw": u * abs_matmul(Mw.T, inp.X), "top8": np.argsort(-counts)[:8]}


def _oracle(name):
    if name not in _CACHE:
        _CACHE.clear()   # one workload's oracle at a time (the cases run grouped by workload)
        _CACHE[name] = _dense(name) if name in ("minimind", "v32k") else _sampled(name)
    return _CACHE[name]


def _run(inp, T, path, stats):
    X, W, y = dev_inputs(inp)
    wl = inp.wl
    if path.startswith("split"):
        f = vp.lmhead_ce_fwd(X, W, y, T, shard_stats=stats)
        dX, dW = vp.lmhead_ce_bwd(X, W, y, f["lse"], T, vocab_chunk=wl.V if path.endswith("_all") else None)
        ws = f["workspace"]
    else:
        f = vp.lmhead_ce_fwd_bwd(X, W, y, T, shard_stats=stats, token_chunk=wl.N if path.endswith("_all") else None)
        dX, dW, ws = f["dX"], f["dW"], f["workspace"]
    torch.cuda.synchronize()
    assert vp.read_device_status(ws) == 0
    return X, W, f, dX, dW


@pytest.mark.parametrize("name,T,path", CASES)
def test_config_parity(name, T, path):
    o = _oracle(name)
    inp = o["inp"]
    wl = inp.wl
    dense = "fwd" in o
    X, W, f, dX, dW = _run(inp, T, path, stats=dense)
    assert int(f["n_bad"].item()) == 0
    if dense:
        assert_loss_close(np64(f["lse"]), o["fwd"]["lse"], "bf16", what="lse")
        assert_loss_close(np64(f["loss"]), o["fwd"]["loss"], "bf16", what="loss")
        assert_loss_close(np64(f["mean"]), [o["fwd"]["mean"]], "bf16", what="mean")
        assert_stats_close(np64(f["shard_stats"]), o["stats"][T], inp, T)
        ex, ew = rel_fro(np64(dX), o["dX"]), rel_fro(np64(dW), o["dW"])
        assert ex <= 2e-2 and ew <= 2e-2, (ex, ew)
        assert_within("dX", np64(dX), o["dX"], o["bx"])
        assert_within("dW", np64(dW), o["dW"], o["bw"])
        return
    assert_loss_close(np64(f["lse"]), o["lse"], "bf16", what="lse")
    assert_loss_close(np64(f["loss"]), o["loss"], "bf16", what="loss")
    assert_loss_close(np64(f["mean"]), [o["mean"]], "bf16", what="mean")
    rt = torch.from_numpy(o["rows"]).cuda()
    got = np64(dX[rt])
    assert rel_fro(got, o["dX_rows"]) <= 2e-2
    assert_within("dX rows", got, o["dX_rows"], o["bx"])
    vt = torch.from_numpy(o["vrows"]).cuda()
    gw = np64(dW[vt])
    assert rel_fro(gw, o["dW_rows"]) <= 2e-2
    assert_within("dW rows", gw, o["dW_rows"], o["bw"])
    for k, v in enumerate(o["vrows"]):   # the frequent ids' rows carry the one-hot term: each on its own too
        if v in o["top8"]:
            assert rel_fro(gw[k], o["dW_rows"][k]) <= 2e-2, int(v)
    ign = np.flatnonzero(inp.targets == IGN)
    if len(ign):
        it = torch.from_numpy(ign).cuda()
        assert bool((f["loss"][it] == 0).all()) and bool((dX[it] == 0).all())
    # dW identities: sum_v dW[v,:] = 0 (dZ rows sum to 0); <dW, W> = <dX, X> (= <dZ, Z>)
    dWd = dW.double()
    # bf16 rounding of dZ leaves |sum_v dZ[n,v]| ~ 2^-9 |dZ[n]|, i.e. a column-sum
    # norm ~ 2e-3 |dW|; a dropped or misplaced onehot term gives ~ |dW|
    assert dWd.sum(0).norm().item() <= 1e-2 * dWd.norm().item()
    a = (dWd * W.double()).sum().item()
    b = (dX.double() * X.double()).sum().item()
    assert abs(a - b) <= 2e-2 * max(abs(a), abs(b)) + 1e-6, (a, b)


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
