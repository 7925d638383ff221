"""GPU parity of the vocab-parallel embedding and the fused LM head + CE
(forward and backward) against the float64 oracle, element by element, on
seeded inputs spanning several tiles with ragged tails, plus edge cases."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
import vocab_lm_head_vp_b300 as vp
from golden_io import read
from gpu_util import (assert_grads_elementwise, assert_loss_close, assert_lse_close, assert_stats_close, dev_inputs,
                      grad_tol, np64, rel_fro)

pytestmark = pytest.mark.gpu
IGN = -100


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


def _oracle_embed_bits(ids, W_np, V, T, dtype):
    o = ref.embed(ids, W_np.astype(np.float64), V, T)
    if dtype == "bf16":
        return torch.from_numpy(o.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    return o.astype(np.float32).view(np.int32)


# ------------------------------------------------------------------ embedding
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_embed_worked_example(dtype):
    """The V=8, T=2, ids [1,6] table of sec. 5.2.1 and figure 1's id 5."""
    for name in ("embed_v8_t2_ids_1_6.txt", "embed_v8_t2_id5.txt"):
        g = read(name)
        V, T = int(g["V"][0]), int(g["T"][0])
        ids = np.array([int(v) for v in g["ids"]])
        H = 8
        Wn = (np.arange(V * H, dtype=np.float32).reshape(V, H) + 1.0)
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        W = torch.from_numpy(Wn).to(tdt).cuda()
        out = vp.embed_fwd(torch.from_numpy(ids).cuda(), W, T)
        want = np.stack([Wn[int(s[1:])] if s != "0" else np.zeros(H, np.float32) for s in g["sum"]])
        assert np.array_equal(out.float().cpu().numpy(), want)


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 2), ("tiny", 4), ("tiny", 16),
                                    ("minimind", 1), ("minimind", 2), ("minimind", 16)])
def test_embed_workload_bit_exact(name, T):
    """Each workload's ids gathered at every T in {1, 2, its own T, 16} that
    divides V: bit-exact against the oracle's shard sum at that T."""
    inp = synth.make_inputs(name)
    wl = inp.wl
    X, W, y = dev_inputs(inp)
    ids = inp.targets
    out = vp.embed_fwd(y, W, T)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), _oracle_embed_bits(ids, inp.W, wl.V, T, wl.dtype))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_embed_edge_ids_and_negative_zero(dtype):
    rng = np.random.default_rng(9)
    V, H, T = 1000, 136, 8
    Wn = rng.standard_normal((V, H)).astype(np.float32)
    Wn[7, 5] = -0.0
    Wn[7, 6] = 0.0
    ids = rng.integers(0, V, 333)
    ids[:8] = [7, -1, V, -100, 0, V - 1, 7, 2 ** 40]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Wt = torch.from_numpy(Wn).to(tdt)
    out = vp.embed_fwd(torch.from_numpy(ids).cuda(), Wt.cuda(), T)
    Wexact = Wt.float().numpy()
    want = _oracle_embed_bits(ids, Wexact, V, T, dtype)
    assert np.array_equal(_bits(out), want)
    assert _bits(out)[0, 5] == 0                      # -0.0 came out +0.0


def test_embed_large_uniform_and_zipf():
    """Full V128k shapes of the gather (N=16384, H=4096, V=128256), bit-exact
    on sampled rows: uniform and Zipf ids."""
    wl = synth.WORKLOADS["v128k"]
    g = torch.Generator(device="cuda").manual_seed(5)
    W = torch.randn(wl.V, wl.H, generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(17)
    for ids in (rng.integers(0, wl.V, wl.N), synth.zipf_ids(rng, wl.N, wl.V, 1.1)):
        idt = torch.from_numpy(ids).cuda()
        out = vp.embed_fwd(idt, W, wl.T)
        rows = rng.choice(wl.N, 64, replace=False)
        got = out[torch.from_numpy(rows).cuda()].view(torch.int16).cpu()
        want = W[idt[torch.from_numpy(rows).cuda()]].view(torch.int16).cpu()
        assert torch.equal(got, want)


# ------------------------------------------------------------------ forward + backward
def _run(inp, T, ignore_index=IGN, dloss=None, vocab_chunk=None, shard_stats=True):
    X, W, y = dev_inputs(inp)
    f = vp.lmhead_ce_fwd(X, W, y, T, ignore_index, shard_stats=shard_stats)
    dl = None if dloss is None else torch.from_numpy(dloss.astype(np.float32)).cuda()
    dX, dW = vp.lmhead_ce_bwd(X, W, y, f["lse"], T, ignore_index, dloss=dl, vocab_chunk=vocab_chunk)
    torch.cuda.synchronize()
    assert vp.read_device_status(f["workspace"]) == 0
    return f, dX, dW


def _check(inp, T, f, dX, dW, ignore_index=IGN, dloss=None, check_stats=True):
    wl = inp.wl
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, wl.V, T, ignore_index)
    # l_n = log1p(R) + (m - z_y): both terms are non-negative (z_y is one of the
    # logits the maximum m is taken over), so no token's loss is below 0
    assert (np64(f["loss"]) >= 0.0).all(), "negative per-token loss"
    assert_lse_close(np64(f["lse"]), o["lse"], inp)
    assert_loss_close(np64(f["loss"]), o["loss"], wl.dtype, what="loss")
    assert_loss_close(np64(f["mean"]), [o["mean"]], wl.dtype, what="mean")
    assert int(f["n_bad"].item()) == o["n_bad"]
    if check_stats:
        # S_t >= 1 (the max term); its log is what the loss uses
        assert_stats_close(np64(f["shard_stats"]), o["shard_stats"], inp, T)
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, wl.V, ignore_index, dloss)
    ex, ew = rel_fro(np64(dX), b["dX"]), rel_fro(np64(dW), b["dW"])
    tol = grad_tol(wl.dtype)
    assert ex <= tol and ew <= tol, f"rel Frobenius dX {ex:.2e} dW {ew:.2e} (tol {tol})"
    assert_grads_elementwise(inp, dX, dW, b)
    return ex, ew


@pytest.mark.parametrize("T", [1, 2, 4, 16])   # every T in {1, 2, the config's 4, 16}: all divide V = 16
def test_tiny_config_f32(T):
    inp = synth.make_inputs("tiny")
    f, dX, dW = _run(inp, T)
    _check(inp, T, f, dX, dW)


def test_page_t4_simulation_f32():
    """The interview note's t=4 NumPy setup through the GPU: X = z, W = I
    (H = V = 16), so the kernel's logits are exactly the page's z."""
    z, y = synth.page_t4_simulation()
    X = z.astype(np.float32)
    W = np.eye(16, dtype=np.float32)
    inp = synth.Inputs(synth.Workload("page_t4", 6, 16, 16, 4, "f32", 0.0, "uniform"), X, W, y, None, None)
    f, dX, dW = _run(inp, 4)
    _check(inp, 4, f, dX, dW)
    dense = ref.cross_entropy(X.astype(np.float64), y)
    assert np.allclose(np64(f["loss"]), dense["loss"])          # the page's printed True


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("zero", ["W", "X"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_constant_logits_closed_form(dtype, zero, path):
    """Every logit 0 (W = 0, or X = 0; several tiles, a ragged token tail,
    shard edges inside tiles): the GPU path against the closed form rather
    than the oracle.  Each valid token's loss and every lse are log V, each
    shard reports m_t = 0, S_t = V/T, z_y^(t) = 0, and dZ = g (1/V - 1[j=y]):
    with W = 0 dX is exactly 0 and dW = dZ^T X, with X = 0 dW is exactly 0 and
    dX = dZ W ("Vocab Parallelism" sec. 5.3.1-5.3.2)."""
    N, H, V, T = 300, 64, 1000, 8
    inp = synth.small_case(N, H, V, T, dtype, seed=91, ignore_frac=0.1)
    inp.targets[:2] = [V, -3]                      # out of range: ignored and counted
    for a in ((inp.W, inp.W_bits) if zero == "W" else (inp.X, inp.X_bits)):
        if a is not None:
            a[...] = 0
    if path == "split":
        f, dX, dW = _run(inp, T)
    else:
        X, W, y = dev_inputs(inp)
        f = vp.lmhead_ce_fwd_bwd(X, W, y, T, shard_stats=True)
        torch.cuda.synchronize()
        assert vp.read_device_status(f["workspace"]) == 0
        dX, dW = f["dX"], f["dW"]
    y = inp.targets
    valid = (y >= 0) & (y < V)
    logV = np.log(V)
    loss, lse = np64(f["loss"]), np64(f["lse"])
    assert np.all(np.abs(loss[valid] - logV) <= 1e-5 * logV) and np.all(loss[~valid] == 0.0)
    assert np.all(np.abs(lse - logV) <= 1e-5 * logV)
    assert abs(float(f["mean"].item()) - logV) <= 1e-5 * logV
    assert int(f["n_bad"].item()) == 2
    st = np64(f["shard_stats"])
    assert np.all(st[:, 0] == 0.0) and np.all(st[:, 2] == 0.0)
    assert np.all(np.abs(st[:, 1] - V / T) <= 1e-5 * V / T)
    g = np.where(valid, 1.0 / valid.sum(), 0.0)
    onehot = np.zeros((N, V))
    onehot[np.nonzero(valid)[0], y[valid]] = 1.0
    dZ = g[:, None] * (1.0 / V - onehot)
    if zero == "W":
        assert np.all(np64(dX) == 0.0)
        assert rel_fro(np64(dW), dZ.T @ np.asarray(inp.X, np.float64)) <= grad_tol(dtype)
    else:
        assert np.all(np64(dW) == 0.0)
        assert rel_fro(np64(dX), dZ @ np.asarray(inp.W, np.float64)) <= grad_tol(dtype)


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("c", [1000.0, -1000.0])
def test_large_logits_bf16(c, path):
    """Every logit of every row moved by c = +-1000 (X gets a column of ones,
    W a column of c; exact in bf16): e^z would overflow or vanish without the
    max shift, and softmax and loss are unchanged by it.  Both paths against
    the oracle on the shifted inputs, statistics and gradients element by
    element ("Vocab Parallelism" sec. 5.3.1, CE(x,k) = -x_k + m + log sum
    e^(x_i - m))."""
    N, H, V, T = 300, 64, 1000, 4
    base = synth.small_case(N, H, V, T, "bf16", seed=93, ignore_frac=0.1)
    pad = np.zeros((N, 8), np.float32)
    pad[:, 0] = 1.0
    wpad = np.zeros((V, 8), np.float32)
    wpad[:, 0] = c
    X = np.concatenate([base.X, pad], axis=1)
    W = np.concatenate([base.W, wpad], axis=1)
    bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    wl = synth.Workload("shifted", N, H + 8, V, T, "bf16", 0.0, "uniform")
    inp = synth.Inputs(wl, X, W, base.targets, bits(X), bits(W))
    assert np.array_equal(torch.from_numpy(bits(W).view(np.int16)).view(torch.bfloat16).float().numpy(), W)
    if path == "split":
        f, dX, dW = _run(inp, T)
    else:
        Xd, Wd, y = dev_inputs(inp)
        f = vp.lmhead_ce_fwd_bwd(Xd, Wd, y, T, shard_stats=True)
        torch.cuda.synchronize()
        assert vp.read_device_status(f["workspace"]) == 0
        dX, dW = f["dX"], f["dW"]
    assert torch.isfinite(f["loss"]).all() and torch.isfinite(f["lse"]).all()
    assert (np64(f["loss"]) >= 0.0).all()
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, V, T)
    assert_lse_close(np64(f["lse"]), o["lse"], inp)
    assert_loss_close(np64(f["loss"]), o["loss"], "bf16", what="loss")
    assert_loss_close(np64(f["mean"]), [o["mean"]], "bf16", what="mean")
    assert int(f["n_bad"].item()) == o["n_bad"]
    assert_stats_close(np64(f["shard_stats"]), o["shard_stats"], inp, T)
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, V)
    # dX's column of the constant feature is c * sum_v dZ[n, v], exactly 0 (the
    # rows of dZ sum to 0) but made of terms up to c * g: the bf16 rounding of
    # dZ leaves ~c * g * 2^-9 there, larger than the other columns' entries, so
    # a per-tensor relative norm says nothing for it; the elementwise bound,
    # which scales with each entry's terms, covers every column
    dXn = np64(dX)
    assert rel_fro(dXn[:, :H], b["dX"][:, :H]) <= grad_tol("bf16") and rel_fro(np64(dW), b["dW"]) <= grad_tol("bf16")
    assert np.all(dXn[:, H + 1:] == 0.0)
    assert_grads_elementwise(inp, dX, dW, b)


def _argmax_case(N, V, dtype, seed):
    """Logits chosen directly (X = Z, W = I, H = V, so the kernel's logits are
    exactly X): most targets are the row's maximum by a margin that puts the
    loss between about 1e-7 and 1e-3, where lse - z_y would cancel to nothing
    in fp32; a few rows have the target tied with another maximum, a few a
    target below the maximum, a few are ignored."""
    rng = np.random.default_rng(seed)
    y = rng.integers(0, V, N)
    top = rng.uniform(-4.0, 4.0, N)
    gap = rng.uniform(np.log(V) + 7.0, np.log(V) + 16.0, N)       # l ~ V e^-gap in [1e-7, 1e-3]
    Z = top[:, None] - gap[:, None] - np.abs(rng.standard_normal((N, V))) * 0.5
    Z[np.arange(N), y] = top
    tie = np.arange(0, N, 17)                                      # a second maximum: l ~ log 2
    Z[tie, (y[tie] + 1) % V] = top[tie]
    below = np.arange(5, N, 23)                                    # target under the maximum
    Z[below, (y[below] + 3) % V] = top[below] + 0.75
    y[np.arange(9, N, 31)] = IGN
    if dtype == "bf16":
        bits = synth.round_to_bf16_bits(Z.astype(np.float32))
        X = synth.bf16_bits_to_f32(bits)
        Wb = synth.round_to_bf16_bits(np.eye(V, dtype=np.float32))
        W = synth.bf16_bits_to_f32(Wb)
    else:
        X, W, bits, Wb = Z.astype(np.float32), np.eye(V, dtype=np.float32), None, None
    wl = synth.Workload(f"argmax_{N}x{V}", N, V, V, 1, dtype, 0.0, "uniform")
    return synth.Inputs(wl, X, W, y.astype(np.int64), bits, Wb)


@pytest.mark.parametrize("dtype,V", [("f32", 192), ("bf16", 512)])
@pytest.mark.parametrize("T", [1, 2, 4, 16])
def test_loss_when_target_is_the_maximum(dtype, V, T):
    """Per-token loss within rel 1e-5 of the oracle's where it is tiny: the
    merge forms log1p(R) + (m - z_y) (R = the sum without the maximal term),
    the pages' log sum e^(z-m) - (z_y - m) without cancellation.  The logits
    are exact here, so the bound holds for the bf16 path's arithmetic too."""
    inp = _argmax_case(300, V, dtype, seed=V + T)
    X, W, y = dev_inputs(inp)
    f = vp.lmhead_ce_fwd(X, W, y, T, shard_stats=True)
    torch.cuda.synchronize()
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, V, T)
    valid = inp.targets >= 0
    small = valid & (o["loss"] < 1e-3)
    assert small.sum() > 200 and o["loss"][small].min() < 1e-6      # the regime this test is about
    assert_loss_close(np64(f["loss"]), o["loss"], "f32", what="loss")
    assert_loss_close(np64(f["lse"]), o["lse"], "f32", what="lse")
    assert_stats_close(np64(f["shard_stats"]), o["shard_stats"], inp, T)


CASES = [  # N, H, V, T, dtype: several tiles, ragged tails, shard edges inside tiles
    (300, 200, 1000, 4, "bf16"),
    (130, 64, 520, 2, "bf16"),
    (1, 64, 256, 1, "bf16"),
    (257, 136, 770, 7, "bf16"),     # V/T = 110 < 256: one tile spans up to 4 shards
    (64, 512, 6400, 16, "bf16"),
    (50, 8, 48, 3, "bf16"),         # H = 8 (one 16-byte row), V < 64: a tile spans all 3 shards
    (40, 64, 512, 512, "bf16"),     # T = V: every shard one id, 256 shard records per tile
    (77, 40, 99, 3, "f32"),
    (200, 96, 640, 10, "f32"),
]


@pytest.mark.parametrize("N,H,V,T,dtype", CASES)
def test_small_cases(N, H, V, T, dtype):
    inp = synth.small_case(N, H, V, T, dtype, seed=N + H + V + T, ignore_frac=0.1)
    f, dX, dW = _run(inp, T)
    _check(inp, T, f, dX, dW)


def test_shard_count_invariance_bf16():
    """Loss, dX and dW agree with the oracle for every T dividing V."""
    inp = synth.small_case(384, 256, 2048, 1, "bf16", seed=3)
    losses = []
    for T in (1, 2, 4, 8, 16):
        f, dX, dW = _run(inp, T)
        _check(inp, T, f, dX, dW)
        losses.append(np64(f["loss"]))
    for l in losses[1:]:
        np.testing.assert_allclose(l, losses[0], rtol=0, atol=1e-4)


@pytest.mark.parametrize("chunk", [256, 768, 1536])
def test_chunked_backward(chunk):
    inp = synth.small_case(520, 192, 2000, 4, "bf16", seed=11)
    f, dX, dW = _run(inp, 4, vocab_chunk=chunk)
    _check(inp, 4, f, dX, dW)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ignore_index_in_range_and_bad_targets(dtype):
    inp = synth.small_case(150, 64, 300, 3, dtype, seed=21)
    y = inp.targets
    y[:10] = 5                     # ignore_index inside [0, V)
    y[10:14] = [300, 1000, -1, -7]  # out of range: ignored and counted
    f, dX, dW = _run(inp, 3, ignore_index=5)
    _check(inp, 3, f, dX, dW, ignore_index=5)
    loss = np64(f["loss"])
    assert np.all(loss[:14] == 0.0)
    assert np.all(np64(dX)[:14] == 0.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_ignored(dtype):
    inp = synth.small_case(70, 64, 300, 3, dtype, seed=5)
    inp.targets[:] = IGN
    f, dX, dW = _run(inp, 3)
    assert float(f["mean"].item()) == 0.0 and int(f["n_bad"].item()) == 0
    assert np.all(np64(f["loss"]) == 0.0)
    assert np.all(np64(dX) == 0.0) and np.all(np64(dW) == 0.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_upstream_gradient_vector(dtype):
    inp = synth.small_case(200, 128, 900, 3, dtype, seed=8)
    dloss = np.random.default_rng(1).standard_normal(200)
    f, dX, dW = _run(inp, 3, dloss=dloss)
    _check(inp, 3, f, dX, dW, dloss=dloss)


def test_minimind_config():
    """Full MiniMind-scale workload (N=4096, H=512, V=6400, T=2, bf16) against
    the dense float64 oracle, every token and every gradient entry."""
    inp = synth.make_inputs("minimind")
    f, dX, dW = _run(inp, inp.wl.T)
    ex, ew = _check(inp, inp.wl.T, f, dX, dW)
    print(f"minimind rel Frobenius dX {ex:.3e} dW {ew:.3e}")


def test_autograd_wrapper():
    inp = synth.small_case(96, 64, 512, 2, "bf16", seed=4)
    X, W, y = dev_inputs(inp)
    X.requires_grad_(True)
    W.requires_grad_(True)
    loss = vp.lmhead_ce(X, W, y, 2)
    loss.backward()
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, inp.wl.V)
    assert rel_fro(np64(X.grad), b["dX"]) <= 2e-2
    assert rel_fro(np64(W.grad), b["dW"]) <= 2e-2
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, inp.wl.V, 2)
    assert abs(loss.item() - o["mean"]) <= 2e-2 + 1e-2 * abs(o["mean"])


def test_autograd_upstream_scale():
    """(3 * loss).backward(): the incoming gradient reaches the library as a
    device scalar and scales dX and dW by 3."""
    inp = synth.small_case(96, 64, 512, 2, "bf16", seed=4, ignore_frac=0.1)
    X, W, y = dev_inputs(inp)
    X.requires_grad_(True)
    W.requires_grad_(True)
    (3.0 * vp.lmhead_ce(X, W, y, 2)).backward()
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, inp.wl.V)
    assert rel_fro(np64(X.grad), 3.0 * b["dX"]) <= 2e-2
    assert rel_fro(np64(W.grad), 3.0 * b["dW"]) <= 2e-2


def test_results_repeatable():
    """Two calls on the same inputs give bit-identical results (no atomics in
    any reduction)."""
    inp = synth.small_case(300, 256, 1500, 3, "bf16", seed=2)
    a = _run(inp, 3)
    b = _run(inp, 3)
    assert torch.equal(a[0]["loss"], b[0]["loss"]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_gemm_forms_agree_on_the_path(variant):
    """The split fwd/bwd with each GEMM form (the default: dX tiles chosen per
    launch, dW^T on SM pairs; SM pairs everywhere; one SM with 128-row tiles
    everywhere) matches the oracle (ragged N and V, a shard edge inside tiles,
    two vocab chunks)."""
    vp.set_gemm_variant(variant)
    try:
        inp = synth.small_case(333, 264, 1800, 6, "bf16", seed=77, ignore_frac=0.1)
        f, dX, dW = _run(inp, 6, vocab_chunk=1024)
        _check(inp, 6, f, dX, dW)
    finally:
        vp.set_gemm_variant(0)


@pytest.mark.parametrize("N,H,V,chunk,streamk", [
    (300, 264, 1800, 1800, False), (1100, 512, 3000, 3000, False), (77, 64, 700, 256, False),
    (2600, 1032, 6000, 1536, True),      # ragged rows and columns, four vocab chunks (fp32 store / add / bf16)
    (768, 4096, 2000, 2000, True),       # 48 tiles of 256 x 256 for 148 SMs: each split over ~3 CTAs
    (700, 4104, 12000, 2048, True),      # ragged, six vocab chunks through stream-K (fp32 store / add / bf16)
])
def test_dx_tile_forms(N, H, V, chunk, streamk):
    """dX from 256 x 256 tiles (two 128-row accumulators sharing each B stage)
    against dX from 128 x 256 tiles, and dW through X^T against dW = dZ^T X.  Without stream-K every output element runs
    the same K loop in the same order: bit-identical.  With stream-K (tiles that
    do not fill whole waves) a split tile's k-blocks are summed per CTA and the
    fp32 partial sums added in k order, so the two differ by fp32 summation
    order only; both are held to the oracle's elementwise bound.  N not a
    multiple of 256 leaves the second 128-row block of the last tile partly or
    wholly past the end."""
    inp = synth.small_case(N, H, V, 4, "bf16", seed=N + V, ignore_frac=0.1)
    outs = []
    for variant in (0, 2):
        vp.set_gemm_variant(variant)
        vp.stage_timing_enable(256)
        try:
            f, dX, dW = _run(inp, 4, vocab_chunk=chunk)
            stages = vp.stage_timing_read()
        finally:
            vp.stage_timing_enable(0)
            vp.set_gemm_variant(0)
        _check(inp, 4, f, dX, dW)
        outs.append((f["loss"], dX, dW, stages["dx_gemm"][1], stages["dw_gemm"][1]))
    (l0, x0, w0, k0, c0), (l2, x2, w2, k2, c2) = outs
    assert c0 == c2                                 # vocab chunks: one dW launch each
    assert k2 == c2                                 # 128-row tiles: whole tiles, one dX kernel per chunk
    assert k0 == (2 * c2 if streamk else c2)        # stream-K: the GEMM and its fix-up pass
    # dW: through X^T (form 0) or directly (form 2); the same products summed in the same K order
    assert torch.equal(l0, l2) and rel_fro(np64(w0), np64(w2)) <= 1e-5
    if streamk:
        assert rel_fro(np64(x0), np64(x2)) <= 1e-3
    else:
        assert torch.equal(x0, x2)
