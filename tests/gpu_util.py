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


def assert_loss_close(got, ref, dtype, scale=None, what="loss"):
    """|got - ref| <= atol + rtol * s per token, s = max(|ref|, scale).  For a
    difference of two fp32 terms (loss = lse - z_y) the attainable relative
    accuracy is set by the size of the terms, so callers pass scale = |lse|."""
    atol, rtol = loss_tol(dtype)
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    s = np.abs(ref) if scale is None else np.maximum(np.abs(ref), np.abs(scale))
    err = np.abs(got - ref)
    bad = err > atol + rtol * s
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst err "
                           f"{err.max():.3e} at {int(err.argmax())} (ref {ref.flat[int(err.argmax())]:.6f})")


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


def assert_grads_elementwise(inp, dX, dW, b):
    """dX and dW element by element against a bound derived from the arithmetic.

    b is the oracle's backward (dZ, g, dX, dW).  With M[n, j] = |g_n| (p_nj +
    1[j = y_n]) >= |dZ[n, j]|, the size of the terms that form the logit
    gradient ("Vocab Parallelism" sec. 5.3.2),

        |dX_gpu - dX| <= u (M |W|),      |dW_gpu - dW| <= u (M^T |X|)

    elementwise.  For bf16, u = 2^-7 covers the bf16 rounding of dZ (2^-9), the
    bf16 rounding of dX itself (2^-9), the fp16 rounding of saved probabilities
    (2^-11) and the fp32 error of the logits and of the sums; for fp32 inputs
    u = 1e-4.  A mistake confined to a few small entries (a ragged tail tile, a
    rarely targeted vocab row) fails this although the tensor's relative
    Frobenius error stays small.
    """
    dZ, g = b["dZ"], b["g"]
    M = np.abs(dZ)
    rows = np.nonzero(g != 0)[0]
    y = np.asarray(inp.targets)[rows]
    # at the target |dZ| = |g| (1 - p_y), while the terms are |g| p_y and |g|
    M[rows, y] += 2.0 * np.abs(g[rows]) * (dZ[rows, y] / g[rows] + 1.0)
    X = np.abs(np.asarray(inp.X, dtype=np.float64))
    W = np.abs(np.asarray(inp.W, dtype=np.float64))
    u = 2.0 ** -7 if inp.wl.dtype == "bf16" else 1e-4
    for name, got, want, bound in (("dX", np64(dX), b["dX"], u * (M @ W)),
                                   ("dW", np64(dW), b["dW"], u * (M.T @ X))):
        err = np.abs(got - want)
        bad = err > bound
        if bad.any():
            i = np.unravel_index(int(np.argmax(err - bound)), err.shape)
            raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} entries outside the elementwise bound; "
                                 f"worst at {i}: err {err[i]:.3e}, bound {bound[i]:.3e}, ref {want[i]:.3e}")
