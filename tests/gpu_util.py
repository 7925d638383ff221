"""Helpers for the GPU parity tests: move seeded inputs to the device and
compare with the oracle under the tolerances the tests state."""
import numpy as np
import torch


def dev_inputs(inp, device="cuda"):
    """synth.Inputs -> (X, W, targets) device tensors with the exact same values."""
    if inp.X_bits is not None:
        X = torch.from_numpy(inp.X_bits.view(np.int16)).view(torch.bfloat16).to(device)
        W = torch.from_numpy(inp.W_bits.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        X = torch.from_numpy(np.ascontiguousarray(inp.X, dtype=np.float32)).to(device)
        W = torch.from_numpy(np.ascontiguousarray(inp.W, dtype=np.float32)).to(device)
    y = torch.from_numpy(inp.targets.astype(np.int64)).to(device)
    return X, W, y


def loss_tol(dtype):
    """(atol, rtol) for per-token loss / lse: fp32 rel 1e-5, bf16 abs 2e-2 + rel 1e-2."""
    return (0.0, 1e-5) if dtype == "f32" else (2e-2, 1e-2)


def assert_loss_close(got, ref, dtype, what="loss"):
    """|got - ref| <= atol + rtol * |ref| per token (the stated tolerance)."""
    atol, rtol = loss_tol(dtype)
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst err "
                           f"{np.nanmax(err):.3e} at {int(np.nanargmax(err))} "
                           f"(ref {ref.flat[int(np.nanargmax(err))]:.6g})")


def assert_lse_close(got, ref, inp, what="lse"):
    """lse per token.  bf16: the loss tolerance.  fp32: lse = m + log1p(R) is
    a smooth function of the logits with weights (the softmax) summing to 1, so
    it moves by at most the largest logit error, an H-term fp32 dot product
    held to gamma_H sum_i |x_i w_i| (Higham), plus the rounding of the sum of
    exps, gamma_(V+8); and by rel 1e-5 of itself.  A relative bound alone would
    be meaningless for an lse near zero (it changes sign with the logits)."""
    wl = inp.wl
    if wl.dtype == "bf16":
        assert_loss_close(got, ref, "bf16", what=what)
        return
    A = np.abs(np.asarray(inp.X, np.float64)) @ np.abs(np.asarray(inp.W, np.float64)).T   # [N, V]
    bound = 1e-5 * np.abs(np.asarray(ref, np.float64)) + gamma(wl.H) * A.max(axis=1) + gamma(wl.V + 8)
    assert_within(what, got, ref, bound)


def gamma(n, u=2.0 ** -24):
    """Higham's gamma_n = n u / (1 - n u): the relative bound of an n-term fp32 sum."""
    return n * u / (1.0 - n * u)


def assert_stats_close(st, so, inp, T, what=""):
    """Shard statistics (m_t, S_t, z_y^(t)) [T,3,N] against the oracle's.
    bf16: the stated bf16 tolerance on each.  fp32: m_t and z_y^(t) are single
    logits, an H-term fp32 dot product each, held to gamma_H sum_i |x_i w_i|
    (Higham, dot products); log S_t moves by at most twice the largest logit
    error in the shard plus the rounding of its exps and sum."""
    wl = inp.wl
    if wl.dtype == "bf16":
        assert_loss_close(st[:, 0], so[:, 0], "bf16", what="m_t" + what)
        assert_loss_close(st[:, 2], so[:, 2], "bf16", what="z_y^(t)" + what)
        assert_loss_close(np.log(st[:, 1]), np.log(so[:, 1]), "bf16", what="log S_t" + what)
        return
    A = np.abs(np.asarray(inp.X, np.float64)) @ np.abs(np.asarray(inp.W, np.float64)).T   # [N, V]
    V, N = wl.V, A.shape[0]
    Vs = V // T
    g = gamma(wl.H)
    y = np.asarray(inp.targets)
    for t in range(T):
        At = A[:, t * Vs:(t + 1) * Vs]
        bm = g * At.max(axis=1)
        assert_within(f"m_t[{t}]" + what, st[t, 0], so[t, 0], bm)
        own = (y >= t * Vs) & (y < (t + 1) * Vs)
        by = np.where(own, g * A[np.arange(N), np.where(own, y, 0)], 0.0)
        assert_within(f"z_y^({t})" + what, st[t, 2], so[t, 2], by)
        bs = 2.0 * bm + gamma(Vs + 8)
        assert_within(f"log S_t[{t}]" + what, np.log(st[t, 1]), np.log(so[t, 1]), bs)


def rel_fro(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def grad_tol(dtype):
    """Per-tensor relative Frobenius error bound for dX / dW: bf16 2e-2 (the
    stated bar), fp32 1e-5."""
    return 1e-5 if dtype == "f32" else 2e-2


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def term_magnitudes(dZ, g, y, cols=None):
    """M[n, c] = |g_n| (p_nc + 1[c = y_n]) >= |dZ[n, c]|: the size of the terms
    that form each logit-gradient entry (softmax minus one-hot, "Vocab
    Parallelism" sec. 5.3.2), from the oracle's dZ block.  Rows are tokens with
    targets y; cols are the block's vocab ids (all of them when None)."""
    M = np.abs(dZ)
    g = np.asarray(g, dtype=np.float64)
    y = np.asarray(y)
    cols = np.arange(dZ.shape[1]) if cols is None else np.asarray(cols)
    pos = {int(c): k for k, c in enumerate(cols)}
    for n in np.nonzero(g != 0)[0]:
        k = pos.get(int(y[n]))
        if k is not None:
            # at the target |dZ| = |g| (1 - p_y), while the terms are |g| p_y and |g|
            M[n, k] += 2.0 * abs(g[n]) * (dZ[n, k] / g[n] + 1.0)
    return M


# The saved probabilities are fp16 relative to their tile's maximum: below
# 2^-14 they are subnormal, with an absolute error up to 2^-25 (r15), scaled
# by g and by exp(m_tile - lse) <= 1.  In units of u this adds 2^-25 / u to
# every term of a bf16 row with g != 0.
P16_FLOOR = 2.0 ** -25


def with_p16_floor(M, g, dtype):
    """M plus, for bf16, the fp16 quantum of the saved probabilities on every
    entry of a row (the elementwise bound then holds for tiny probabilities too,
    e.g. a batch of one token, where no larger term of a sum dilutes them)."""
    if dtype != "bf16":
        return M
    M += (P16_FLOOR / elementwise_u(dtype)) * np.abs(np.asarray(g, np.float64))[:, None]
    return M


def elementwise_u(dtype):
    """The bound's factor: for bf16, 2^-7 covers the bf16 rounding of dZ
    (2^-9), the bf16 rounding of dX itself (2^-9), the fp16 rounding of saved
    probabilities (2^-11) and the fp32 error of the logits and of the sums;
    1e-4 for fp32 inputs."""
    return 2.0 ** -7 if dtype == "bf16" else 1e-4


def abs_matmul(A, B, chunk=16384):
    """|A| @ |B| in float64, B taken in row chunks (B may be a large float32 array)."""
    out = np.zeros((A.shape[0], B.shape[1]))
    for a in range(0, B.shape[0], chunk):
        out += np.abs(A[:, a:a + chunk]) @ np.abs(np.asarray(B[a:a + chunk], dtype=np.float64))
    return out


def assert_within(name, got, want, bound):
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(int(np.argmax(err - bound)), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} entries outside the elementwise bound; "
                             f"worst at {i}: err {err[i]:.3e}, bound {bound[i]:.3e}, ref {want[i]:.3e}")


def assert_grads_elementwise(inp, dX, dW, b):
    """dX and dW element by element against a bound derived from the arithmetic:

        |dX_gpu - dX| <= u (M |W|),      |dW_gpu - dW| <= u (M^T |X|)

    with M from term_magnitudes (plus the fp16 quantum of the saved
    probabilities, with_p16_floor) and u from elementwise_u.  b is the oracle's
    backward (dZ, g, dX, dW).  A mistake confined to a few small entries (a
    ragged tail tile, a rarely targeted vocab row) fails this although the
    tensor's relative Frobenius error stays small."""
    M = with_p16_floor(term_magnitudes(b["dZ"], b["g"], inp.targets), b["g"], inp.wl.dtype)
    u = elementwise_u(inp.wl.dtype)
    assert_within("dX", np64(dX), b["dX"], u * abs_matmul(M, inp.W))
    assert_within("dW", np64(dW), b["dW"], u * abs_matmul(M.T, inp.X))
