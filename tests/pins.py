"""Checks that pin the float64 oracle to facts other than itself.

Each ``pin_*`` takes the oracle module and raises AssertionError when the
oracle disagrees with what the pages or the mathematics fix.  They are run on
the real oracle (tests/test_oracle_pins.py) and on copies with planted
mistakes (tests/test_oracle_mutants.py), which each must fail at least one.
"""
import math

import numpy as np
import torch

import synth
from golden_io import read

IGN = -100


def _row_of(symbol, W):
    if symbol == "0":
        return np.zeros(W.shape[1])
    assert symbol.startswith("E")
    return np.asarray(W[int(symbol[1:])], dtype=np.float64)


# ---------------------------------------------------------------- embedding
def pin_embed_worked_table(o):
    """The V=8, T=2, ids [1,6] table of the Vocab Parallelism chapter, sec. 5.2.1."""
    g = read("embed_v8_t2_ids_1_6.txt")
    V, T = int(g["V"][0]), int(g["T"][0])
    ids = np.array([int(v) for v in g["ids"]])
    W = np.random.default_rng(5).standard_normal((V, 3)) + 10.0   # rows distinct, none zero
    for t in range(T):
        want = np.stack([_row_of(s, W) for s in g[f"shard{t}"]])
        assert np.array_equal(o.embed_shard_partial(ids, W, V, T, t), want), f"shard {t}"
    want = np.stack([_row_of(s, W) for s in g["sum"]])
    assert np.array_equal(o.embed(ids, W, V, T), want)


def pin_embed_figure1(o):
    """Figure 1 of the interview note: id 5 on V=8, t=2."""
    g = read("embed_v8_t2_id5.txt")
    V, T = int(g["V"][0]), int(g["T"][0])
    ids = np.array([int(v) for v in g["ids"]])
    W = np.arange(V * 4, dtype=np.float64).reshape(V, 4) + 1.0
    for t in range(T):
        want = np.stack([_row_of(s, W) for s in g[f"shard{t}"]])
        assert np.array_equal(o.embed_shard_partial(ids, W, V, T, t), want), f"shard {t}"
    # the owning shard's local row index: shard 1 starts at 4, 5 - 4 = 1
    start1 = o.shard_bounds(V, T)[1][0]
    assert int(ids[0]) - start1 == int(g["shard1_local_row"][0])
    assert np.array_equal(o.embed(ids, W, V, T), np.stack([_row_of(s, W) for s in g["sum"]]))


def pin_embed_brute_force(o):
    """out[n] = W[id_n] for 0 <= id_n < V, zero otherwise, for every T | V;
    -0.0 comes out as +0.0 (sum of shards from +0.0)."""
    rng = np.random.default_rng(11)
    V, H = 12, 5
    W = rng.standard_normal((V, H))
    W[3, 2] = -0.0
    ids = np.array([0, 3, 11, 7, -1, 12, -100, 5, 3, 6])
    for T in (1, 2, 3, 4, 6, 12):
        out = o.embed(ids, W, V, T)
        for n, i in enumerate(ids):
            want = W[i] if 0 <= i < V else np.zeros(H)
            assert np.array_equal(out[n], want), (T, n)
        assert not np.signbit(out[1, 2]), "-0.0 must be summed to +0.0"
    for bad_T in (5, 7, 0):
        try:
            o.shard_bounds(V, bad_T)
        except ValueError:
            continue
        raise AssertionError(f"V % T != 0 must be rejected (T={bad_T})")


# ---------------------------------------------------------------- forward
def _torch_ce(Z, y, reduction):
    return torch.nn.functional.cross_entropy(torch.from_numpy(Z), torch.from_numpy(y),
                                             ignore_index=IGN, reduction=reduction).numpy()


def pin_ce_library(o):
    """Per-token loss and the mean over valid tokens equal float64 torch
    cross_entropy with ignore_index (a library routine for the same definition)."""
    rng = np.random.default_rng(3)
    for (n, V) in [(7, 5), (33, 40), (64, 129)]:
        Z = rng.standard_normal((n, V)) * 4
        y = rng.integers(0, V, n)
        y[::5] = IGN
        r = o.cross_entropy(Z, y, IGN)
        np.testing.assert_allclose(r["loss"], _torch_ce(Z, y, "none"), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["mean"], float(_torch_ce(Z, y, "mean")), rtol=1e-12)
        lse = torch.logsumexp(torch.from_numpy(Z), dim=1).numpy()
        np.testing.assert_allclose(r["lse"], lse, rtol=1e-12, atol=1e-12)
        assert r["n_valid"] == int((y != IGN).sum())


def pin_ce_closed_form(o):
    """Constant logits give l = log V for every token (and every T)."""
    for V, T in [(16, 4), (6400, 2), (12, 3)]:
        X = np.random.default_rng(1).standard_normal((9, 8))
        W = np.zeros((V, 8))
        y = np.arange(9) % V
        r = o.lmhead_ce_forward(X, W, y, V, T)
        np.testing.assert_allclose(r["loss"], math.log(V), rtol=1e-14)
        np.testing.assert_allclose(r["mean"], math.log(V), rtol=1e-14)
        st = r["shard_stats"]
        np.testing.assert_allclose(st[:, 0], 0.0)
        np.testing.assert_allclose(st[:, 1], V // T)
        np.testing.assert_allclose(st[:, 2], 0.0)


def pin_ce_shift_invariance(o):
    """Moving every logit of a row by the same constant c leaves the softmax,
    the loss and the logit gradient unchanged and moves lse by c.  With logits
    near +-1000, where e^z overflows or underflows in float64, only the
    max-shifted forms ([VP-book] sec. 5.3.1 CE(x,k) = -x_k + m + log sum
    e^(x_i - m); the interview note's key formulas) stay finite and agree with
    the unshifted row: the dense form, its gradient and the shard merge."""
    rng = np.random.default_rng(12)
    n, V = 7, 20
    Z = rng.standard_normal((n, V)) * 3
    y = rng.integers(0, V, n)
    y[4] = IGN
    base = o.cross_entropy(Z, y, IGN)
    g = o.upstream_scale(y, V, IGN)
    dZ = o.grad_logits(Z, y, base["lse"], g)
    for c in (1000.0, -1000.0):
        r = o.cross_entropy(Z + c, y, IGN)
        assert np.all(np.isfinite(r["lse"])) and np.all(np.isfinite(r["loss"])), c
        np.testing.assert_allclose(r["loss"], base["loss"], rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(r["lse"] - c, base["lse"], rtol=0, atol=1e-9)
        np.testing.assert_allclose(o.grad_logits(Z + c, y, r["lse"], g), dZ, rtol=1e-9, atol=1e-15)
        for T in (2, 4, 5):
            mg = o.merge_local_stats(o.shard_local_stats(Z + c, y, V, T))
            np.testing.assert_allclose(mg["lse"] - c, base["lse"], rtol=0, atol=1e-9)


def pin_ce_ignore_and_bad(o):
    """Ignored and out-of-range targets: loss 0, excluded from the mean; all
    ignored gives mean 0; out-of-range non-ignored targets are counted."""
    Z = np.random.default_rng(2).standard_normal((6, 10))
    y = np.array([IGN, 3, 10, -5, 9, IGN])
    r = o.cross_entropy(Z, y, IGN)
    assert r["n_valid"] == 2 and r["n_bad"] == 2
    assert np.all(r["loss"][[0, 2, 3, 5]] == 0.0)
    ref = _torch_ce(Z[[1, 4]], y[[1, 4]], "none")
    np.testing.assert_allclose(r["loss"][[1, 4]], ref, rtol=1e-12)
    np.testing.assert_allclose(r["mean"], ref.mean(), rtol=1e-12)
    r0 = o.cross_entropy(Z, np.full(6, IGN), IGN)
    assert r0["mean"] == 0.0 and r0["n_valid"] == 0
    # an ignore_index inside [0, V) marks its positions ignored, as torch does
    y3 = np.array([3, 3, 1, 9, 0, 3])
    r3 = o.cross_entropy(Z, y3, 3)
    t3 = torch.nn.functional.cross_entropy(torch.from_numpy(Z), torch.from_numpy(y3), ignore_index=3,
                                           reduction="none").numpy()
    np.testing.assert_allclose(r3["loss"], t3, rtol=1e-12)
    assert r3["n_valid"] == 3 and r3["n_bad"] == 0
    g3 = o.upstream_scale(y3, 10, 3)
    np.testing.assert_allclose(g3, [0, 0, 1 / 3, 1 / 3, 1 / 3, 0])


def pin_shard_invariance(o):
    """The pages' three-reduction form and the local-stat merge reproduce the
    dense loss for every T dividing V, and the shard stats are the plain
    per-shard max / sum-exp / owned target logit (brute force)."""
    rng = np.random.default_rng(4)
    V = 24
    Z = rng.standard_normal((10, V)) * 6
    y = rng.integers(0, V, 10)
    y[2] = IGN
    dense = o.cross_entropy(Z, y, IGN)
    for T in (1, 2, 3, 4, 6, 8, 12, 24):
        r = o.cross_entropy_three_reductions(Z, y, V, T, IGN)
        np.testing.assert_allclose(r["loss"], dense["loss"], rtol=1e-12, atol=1e-12)
        st = o.shard_local_stats(Z, y, V, T)
        mg = o.merge_local_stats(st)
        np.testing.assert_allclose(mg["lse"], dense["lse"], rtol=1e-12)
        vs = V // T
        for t in range(T):
            for n in range(10):
                seg = Z[n, t * vs:(t + 1) * vs]
                mx = max(seg)
                assert st[t, 0, n] == mx
                np.testing.assert_allclose(st[t, 1, n], sum(math.exp(v - mx) for v in seg), rtol=1e-13)
                own = t * vs <= y[n] < (t + 1) * vs
                assert st[t, 2, n] == (Z[n, y[n]] if own else 0.0)


def pin_page_t4_simulation(o):
    """The interview note's NumPy t=4 check: same seeded inputs, sharded merge
    allclose to the dense CE (the page prints True); the dense CE also matches
    torch cross_entropy on those logits."""
    g = read("ce_numpy_t4_simulation.txt")
    z, y = synth.page_t4_simulation()
    assert z.shape == (int(g["n"][0]), int(g["V"][0]))
    T = int(g["t"][0])
    V = z.shape[1]
    dense = o.cross_entropy(z, y, IGN)
    shard = o.cross_entropy_three_reductions(z, y, V, T, IGN)
    assert str(bool(np.allclose(shard["loss"], dense["loss"]))) == g["allclose"][0]
    np.testing.assert_allclose(dense["loss"], _torch_ce(z, y, "none"), rtol=1e-12)
    mg = o.merge_local_stats(o.shard_local_stats(z, y, V, T))
    np.testing.assert_allclose(mg["lse"] - mg["z_y"], dense["loss"], rtol=1e-12)


# ---------------------------------------------------------------- backward
def pin_grad_library(o):
    """dZ equals torch autograd of float64 cross_entropy(mean, ignore_index);
    rows sum to 0; dZ[n,y] in [-g_n, 0]; ignored rows are zero."""
    rng = np.random.default_rng(6)
    n, V, H = 12, 20, 7
    X = rng.standard_normal((n, H))
    W = rng.standard_normal((V, H)) * 0.7
    y = rng.integers(0, V, n)
    y[[1, 8]] = IGN
    b = o.lmhead_ce_backward(X, W, y, V, IGN)
    Zt = torch.from_numpy(X @ W.T).requires_grad_(True)
    torch.nn.functional.cross_entropy(Zt, torch.from_numpy(y), ignore_index=IGN).backward()
    np.testing.assert_allclose(b["dZ"], Zt.grad.numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b["dZ"].sum(axis=1), 0.0, atol=1e-15)
    g = 1.0 / 10
    for i in range(n):
        if y[i] == IGN:
            assert np.all(b["dZ"][i] == 0.0)
        else:
            assert -g <= b["dZ"][i, y[i]] <= 0.0


def _fd(f, A, eps=1e-6):
    G = np.zeros_like(A)
    it = np.nditer(A, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = A[idx]
        A[idx] = old + eps
        fp = f()
        A[idx] = old - eps
        fm = f()
        A[idx] = old
        G[idx] = (fp - fm) / (2 * eps)
    return G


def pin_grad_finite_differences(o):
    """dX and dW match central finite differences of the mean loss (and of
    sum_n dloss_n l_n).  V = H so that a transposed operand cannot pass."""
    rng = np.random.default_rng(7)
    for (n, H, V, dl) in [(5, 6, 6, False), (4, 8, 8, True), (6, 5, 9, False)]:
        X = rng.standard_normal((n, H))
        W = rng.standard_normal((V, H)) * 0.8
        y = rng.integers(0, V, n)
        y[1] = IGN
        dloss = rng.standard_normal(n) if dl else None

        def total():
            r = o.lmhead_ce_forward(X, W, y, V, 1, IGN)
            return float((r["loss"] * dloss).sum()) if dl else r["mean"]

        b = o.lmhead_ce_backward(X, W, y, V, IGN, dloss)
        np.testing.assert_allclose(b["dX"], _fd(total, X), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(b["dW"], _fd(total, W), rtol=1e-6, atol=1e-8)


def pin_rows_variant(o):
    """The row-at-a-time form (used at full size) equals the dense form."""
    rng = np.random.default_rng(8)
    n, H, V = 16, 12, 50
    X = rng.standard_normal((n, H))
    W = (rng.standard_normal((V, H)) * 0.5).astype(np.float32)
    y = rng.integers(0, V, n)
    y[3] = IGN
    rows = np.array([0, 3, 7, 15])
    nv = int((y != IGN).sum())
    r = o.lmhead_ce_rows(X, W, y, rows, nv, IGN, w_chunk=7)
    Zt = torch.from_numpy(X @ W.astype(np.float64).T)
    lt = torch.nn.functional.cross_entropy(Zt, torch.from_numpy(y), ignore_index=IGN,
                                           reduction="none").numpy()
    np.testing.assert_allclose(r["loss"], lt[rows], rtol=1e-12)
    b = o.lmhead_ce_backward(X, W, y, V, IGN)
    np.testing.assert_allclose(r["dX"], b["dX"][rows], rtol=1e-12, atol=1e-15)


def pin_dw_rows_variant(o):
    """dW rows for selected vocab ids (used at full size) equal torch's autograd
    of the mean cross-entropy (float64, CPU), ignored and repeated targets in."""
    rng = np.random.default_rng(9)
    n, H, V = 20, 6, 40
    X = rng.standard_normal((n, H))
    W = (rng.standard_normal((V, H)) * 0.5).astype(np.float32)
    y = rng.integers(0, V, n)
    y[:4] = [IGN, 7, 7, 7]
    Wt = torch.from_numpy(W.astype(np.float64)).requires_grad_(True)
    Z = torch.from_numpy(X) @ Wt.T
    torch.nn.functional.cross_entropy(Z, torch.from_numpy(y), ignore_index=IGN).backward()
    nv = int((y != IGN).sum())
    lse = o.lmhead_ce_rows(X, W, y, np.arange(n), nv, IGN, with_dx=False)["lse"]
    rows = np.array([0, 7, 13, V - 1])
    np.testing.assert_allclose(o.lmhead_ce_dw_rows(X, W, y, lse, rows, nv, IGN), Wt.grad.numpy()[rows],
                               rtol=1e-10, atol=1e-14)


def pin_embed_sp(o):
    """SP on (sec. 5.2.1, reduce-scatter): with the V=8, T=2, ids [1,6] table,
    rank 0 keeps token 1's row E1 and rank 1 token 6's row E6; in general the
    ranks' slices, stacked in rank order, are the SP-off result (all-reduce)."""
    g = read("embed_v8_t2_ids_1_6.txt")
    V, T = int(g["V"][0]), int(g["T"][0])
    ids = np.array([int(v) for v in g["ids"]])
    W = np.random.default_rng(8).standard_normal((V, 3)) + 10.0
    for r in range(T):
        assert np.array_equal(o.embed_sp(ids, W, V, T, r), _row_of(g["sum"][r], W)[None, :]), r
    rng = np.random.default_rng(15)
    V, H, N = 24, 5, 48
    ids = rng.integers(-2, V + 2, N)
    W = rng.standard_normal((V, H))
    W[3, 1] = -0.0
    for T in (1, 2, 3, 4, 6, 8, 12, 24):
        whole = np.concatenate([o.embed_sp(ids, W, V, T, r) for r in range(T)])
        assert np.array_equal(whole, o.embed(ids, W, V, T)), T
    try:
        o.embed_sp(ids[:47], W, V, 2, 0)
    except ValueError:
        pass
    else:
        raise AssertionError("N % T != 0 must be rejected")


# ---------------------------------------------------------------- embedding backward
def pin_embed_bwd_worked_table(o):
    """Backward of the V=8, T=2, ids [1,6] table (sec. 5.2.1): position n's
    output row is the weight row the table's SUM line names, so its upstream
    row lands in that weight row and nowhere else -- not in the local row 0
    (global rows 0 and 4) that the masked positions looked up."""
    g = read("embed_v8_t2_ids_1_6.txt")
    V, T = int(g["V"][0]), int(g["T"][0])
    ids = np.array([int(v) for v in g["ids"]])
    G = np.random.default_rng(6).standard_normal((len(ids), 3)) + 10.0
    want = np.zeros((V, 3))
    for n, s in enumerate(g["sum"]):
        if s != "0":
            want[int(s[1:])] += G[n]
    assert np.array_equal(o.embed_backward(ids, G, V, T), want)


def pin_embed_bwd_adjoint(o):
    """<embed(ids, W), G> = <W, embed_backward(ids, G)> for random W, G: the
    backward is the adjoint of the (separately pinned) forward, for every
    T | V, with out-of-range ids and repeated ids."""
    rng = np.random.default_rng(12)
    V, H, N = 24, 7, 40
    ids = rng.integers(-3, V + 3, N)
    ids[:6] = [0, 0, 6, 6, V - 1, 12]
    W = rng.standard_normal((V, H))
    G = rng.standard_normal((N, H))
    for T in (1, 2, 3, 4, 6, 8, 12, 24):
        lhs = float((o.embed(ids, W, V, T) * G).sum())
        dW = o.embed_backward(ids, G, V, T)
        rhs = float((W * dW).sum())
        assert abs(lhs - rhs) <= 1e-12 * (np.abs(G).sum() * np.abs(W).max()), (T, lhs, rhs)
        # rows no valid id names (local row 0 of a shard included) get nothing
        assert not dW[np.setdiff1d(np.arange(V), ids)].any(), T


def pin_embed_bwd_library(o):
    """torch.nn.functional.embedding's autograd (float64, CPU) on the valid ids
    equals the oracle for every T, and a given dW0 is added (the tied weight)."""
    rng = np.random.default_rng(13)
    V, H, N = 30, 5, 64
    ids = rng.integers(0, V, N)
    ids[:10] = 3                                   # a heavily repeated id
    ids[10:13] = [-1, V, -100]                     # out of range: no gradient
    G = rng.standard_normal((N, H))
    valid = (ids >= 0) & (ids < V)
    W = torch.zeros((V, H), dtype=torch.float64, requires_grad=True)
    out = torch.nn.functional.embedding(torch.from_numpy(ids[valid]), W)
    out.backward(torch.from_numpy(G[valid]))
    want = W.grad.numpy()
    D = rng.standard_normal((V, H))
    for T in (1, 2, 3, 5, 6, 10, 15, 30):
        np.testing.assert_allclose(o.embed_backward(ids, G, V, T), want, rtol=0, atol=1e-12)
        np.testing.assert_allclose(o.embed_backward(ids, G, V, T, dW0=D), want + D, rtol=0, atol=1e-12)


def pin_embed_bwd_finite_differences(o):
    """Central differences of L(W) = sum <embed(ids, W), G> in every weight
    entry (L is linear, so they are exact up to rounding)."""
    rng = np.random.default_rng(14)
    V, H, N, T = 8, 3, 11, 4
    ids = rng.integers(-1, V + 1, N)
    W = rng.standard_normal((V, H))
    G = rng.standard_normal((N, H))
    dW = o.embed_backward(ids, G, V, T)
    h = 0.5
    for v in range(V):
        for c in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, c] += h
            Wm[v, c] -= h
            fd = ((o.embed(ids, Wp, V, T) * G).sum() - (o.embed(ids, Wm, V, T) * G).sum()) / (2 * h)
            assert abs(fd - dW[v, c]) <= 1e-12, (v, c, fd, dW[v, c])


ALL_PINS = [pin_embed_worked_table, pin_embed_figure1, pin_embed_brute_force,
            pin_embed_sp, pin_embed_bwd_worked_table, pin_embed_bwd_adjoint, pin_embed_bwd_library,
            pin_embed_bwd_finite_differences,
            pin_ce_library, pin_ce_closed_form, pin_ce_shift_invariance, pin_ce_ignore_and_bad,
            pin_shard_invariance, pin_page_t4_simulation,
            pin_grad_library, pin_grad_finite_differences, pin_rows_variant, pin_dw_rows_variant]
