"""GPU parity of vp_lmhead_ce_fwd_bwd (forward and backward in one call, the
tile probabilities saved in fp16 instead of recomputed) against the float64
oracle, on the same cases as the split calls, plus token chunking and its
agreement with the split path."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import dev_inputs, np64, rel_fro
from test_gpu_ce import CASES, _check, _run

pytestmark = pytest.mark.gpu
IGN = -100


def _fused(inp, T, ignore_index=IGN, dloss=None, token_chunk=None, shard_stats=True):
    X, W, y = dev_inputs(inp)
    dl = None if dloss is None else torch.from_numpy(dloss.astype(np.float32)).cuda()
    o = vp.lmhead_ce_fwd_bwd(X, W, y, T, ignore_index, dloss=dl, shard_stats=shard_stats, token_chunk=token_chunk)
    torch.cuda.synchronize()
    assert vp.read_device_status(o["workspace"]) == 0
    return o, o["dX"], o["dW"]


@pytest.mark.parametrize("N,H,V,T,dtype", CASES)
def test_fused_small_cases(N, H, V, T, dtype):
    inp = synth.small_case(N, H, V, T, dtype, seed=N + H + V + T, ignore_frac=0.1)
    o, dX, dW = _fused(inp, T)
    _check(inp, T, o, dX, dW)


@pytest.mark.parametrize("chunk", [128, 256, 384])
def test_fused_token_chunks(chunk):
    """Token chunks of 128..384 rows over N=520 (a ragged last chunk): the dW
    sum over chunks and the per-chunk dX rows and statistics."""
    inp = synth.small_case(520, 192, 2000, 4, "bf16", seed=11, ignore_frac=0.1)
    o, dX, dW = _fused(inp, 4, token_chunk=chunk)
    _check(inp, 4, o, dX, dW)


def test_fused_chunk_from_workspace_bytes():
    """A workspace sized for 256-row chunks makes the call run 256-row chunks
    (the same results as one chunk within the bf16 tolerance)."""
    inp = synth.small_case(700, 128, 1500, 3, "bf16", seed=12)
    X, W, y = dev_inputs(inp)
    nb = vp.workspace_size(700, 128, 1500, 3, vp.VP_BF16, 2, 256)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    o = vp.lmhead_ce_fwd_bwd(X, W, y, 3, workspace=ws, shard_stats=True)
    torch.cuda.synchronize()
    _check(inp, 3, o, o["dX"], o["dW"])
    with pytest.raises(vp.VpError):
        small = torch.empty(4096, dtype=torch.uint8, device="cuda")
        vp.lmhead_ce_fwd_bwd(X, W, y, 3, workspace=small)


def test_fused_agrees_with_split_path():
    """The fused forward runs the split forward's statistics code: loss, lse and
    the shard statistics are bit-identical; dX/dW differ only by the fp16
    probabilities against the recomputed fp32 logits."""
    inp = synth.small_case(600, 256, 3000, 6, "bf16", seed=31, ignore_frac=0.1)
    f, dXs, dWs = _run(inp, 6)
    o, dXf, dWf = _fused(inp, 6)
    for k in ("loss", "lse", "shard_stats", "mean", "n_bad"):
        assert torch.equal(f[k], o[k]), k
    assert rel_fro(np64(dXf), np64(dXs)) <= 5e-3
    assert rel_fro(np64(dWf), np64(dWs)) <= 5e-3


def test_fused_shard_count_invariance():
    inp = synth.small_case(384, 256, 2048, 1, "bf16", seed=3)
    for T in (1, 2, 4, 8, 16):
        o, dX, dW = _fused(inp, T)
        _check(inp, T, o, dX, dW)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_ignore_index_in_range_and_bad_targets(dtype):
    inp = synth.small_case(150, 64, 300, 3, dtype, seed=21)
    y = inp.targets
    y[:10] = 5
    y[10:14] = [300, 1000, -1, -7]
    o, dX, dW = _fused(inp, 3, ignore_index=5)
    _check(inp, 3, o, dX, dW, ignore_index=5)
    assert np.all(np64(o["loss"])[:14] == 0.0)
    assert np.all(np64(dX)[:14] == 0.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_all_ignored(dtype):
    inp = synth.small_case(70, 64, 300, 3, dtype, seed=5)
    inp.targets[:] = IGN
    o, dX, dW = _fused(inp, 3)
    assert float(o["mean"].item()) == 0.0 and int(o["n_bad"].item()) == 0
    assert np.all(np64(dX) == 0.0) and np.all(np64(dW) == 0.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_upstream_gradient_vector(dtype):
    inp = synth.small_case(200, 128, 900, 3, dtype, seed=8)
    dloss = np.random.default_rng(1).standard_normal(200)
    o, dX, dW = _fused(inp, 3, dloss=dloss)
    _check(inp, 3, o, dX, dW, dloss=dloss)


def test_fused_minimind_config():
    inp = synth.make_inputs("minimind")
    o, dX, dW = _fused(inp, inp.wl.T)
    ex, ew = _check(inp, inp.wl.T, o, dX, dW)
    print(f"minimind fused rel Frobenius dX {ex:.3e} dW {ew:.3e}")


@pytest.mark.parametrize("T", [1, 2, 4, 16])   # every T in {1, 2, the config's 4, 16}: all divide V = 16
def test_fused_tiny_config(T):
    inp = synth.make_inputs("tiny")
    o, dX, dW = _fused(inp, T)
    _check(inp, T, o, dX, dW)


def test_fused_repeatable():
    inp = synth.small_case(300, 256, 1500, 3, "bf16", seed=2)
    a = _fused(inp, 3)
    b = _fused(inp, 3)
    assert torch.equal(a[0]["loss"], b[0]["loss"]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_fused_gemm_forms(variant):
    vp.set_gemm_variant(variant)
    try:
        inp = synth.small_case(333, 264, 1800, 6, "bf16", seed=77, ignore_frac=0.1)
        o, dX, dW = _fused(inp, 6, token_chunk=256)
        _check(inp, 6, o, dX, dW)
    finally:
        vp.set_gemm_variant(0)


def test_fused_loss_scale_dmean():
    """dmean (a device scalar, e.g. a loss scale) multiplies the mean's gradient."""
    inp = synth.small_case(300, 128, 1000, 4, "bf16", seed=9, ignore_frac=0.1)
    X, W, y = dev_inputs(inp)
    scale = torch.tensor([1024.0], device="cuda")
    o = vp.lmhead_ce_fwd_bwd(X, W, y, 4, dmean=scale)
    torch.cuda.synchronize()
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, inp.wl.V)
    assert rel_fro(np64(o["dX"]), 1024.0 * b["dX"]) <= 2e-2
    assert rel_fro(np64(o["dW"]), 1024.0 * b["dW"]) <= 2e-2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_keep_and_saved_backward_match_the_fused_call(dtype):
    """vp_lmhead_ce_fwd_keep + vp_lmhead_ce_bwd_saved: the oracle's results,
    and (bf16) the one-call form's bits, with a per-token upstream gradient."""
    inp = synth.small_case(520, 192, 2000, 4, dtype, seed=41, ignore_frac=0.1)
    X, W, y = dev_inputs(inp)
    dloss = np.random.default_rng(3).standard_normal(520)
    dl = torch.from_numpy(dloss.astype(np.float32)).cuda()
    f = vp.lmhead_ce_fwd(X, W, y, 4, shard_stats=True, keep=True)
    dX, dW = vp.lmhead_ce_bwd(X, W, y, f["lse"], 4, dloss=dl, saved=f["saved"])
    torch.cuda.synchronize()
    assert vp.read_device_status(f["saved"]) == 0
    _check(inp, 4, f, dX, dW, dloss=dloss)
    if dtype == "bf16":
        o = vp.lmhead_ce_fwd_bwd(X, W, y, 4, dloss=dl, shard_stats=True)
        torch.cuda.synchronize()
        for k in ("loss", "lse", "shard_stats", "mean", "n_bad"):
            assert torch.equal(f[k], o[k]), k
        assert torch.equal(dX, o["dX"]) and torch.equal(dW, o["dW"])


def test_autograd_with_saved_probabilities():
    inp = synth.small_case(300, 128, 1000, 4, "bf16", seed=42, ignore_frac=0.1)
    X, W, y = dev_inputs(inp)
    X.requires_grad_(True)
    W.requires_grad_(True)
    (2.0 * vp.lmhead_ce(X, W, y, 4, save_probs=True)).backward()
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, inp.wl.V)
    assert rel_fro(np64(X.grad), 2.0 * b["dX"]) <= 2e-2
    assert rel_fro(np64(W.grad), 2.0 * b["dW"]) <= 2e-2


def test_multicast_logits_bit_identical():
    """GEMM form 3 runs the logits GEMMs in clusters of two CTAs that share the
    W tile by TMA multicast, each CTA's MMAs on its own shared memory: the same
    products in the same order as one SM per tile, so every output is
    bit-identical (ragged N: the last cluster's second CTA has no rows)."""
    inp = synth.small_case(333, 264, 1800, 6, "bf16", seed=78, ignore_frac=0.1)
    outs = []
    for variant in (0, 3):
        vp.set_gemm_variant(variant)
        try:
            outs.append(_fused(inp, 6, token_chunk=256))
        finally:
            vp.set_gemm_variant(0)
    (o0, x0, w0), (o3, x3, w3) = outs
    for k in ("loss", "lse", "mean"):
        assert torch.equal(o0[k], o3[k]), k
    assert torch.equal(x0, x3) and torch.equal(w0, w3)
