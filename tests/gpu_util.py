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
