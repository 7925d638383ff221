"""The allocation-free forward, vp_lmhead_ce_fwd_noalloc, called through the C
ABI, against the workspace forward vp_lmhead_ce_fwd on the same inputs.

It serves callers that cannot allocate device memory (a plugin given only its
input and output buffers, a loop that must never call cudaMalloc); its scratch
is a fixed 32 MiB array inside libvp, shared by every call.  Two calls in a row
with different shapes check that the leftovers of one call do not leak into
the next.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import assert_loss_close, dev_inputs, np64

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    L = vp._load()
    f = L.vp_lmhead_ce_fwd_noalloc
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.restype = I32
    f.argtypes = [P, P, P, I64, I64, I64, I32, I64, I32, P, P, P, P, P, P]
    return f


def _call_noalloc(f, X, W, y, T, ignore_index=-100):
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    out = {"loss": torch.full((N,), float("nan"), device=dev), "lse": torch.full((N,), float("nan"), device=dev),
           "mean": torch.full((1,), float("nan"), device=dev), "n_bad": torch.full((1,), -1, dtype=torch.int32,
                                                                                   device=dev),
           "shard_stats": torch.full((T, 3, N), float("nan"), device=dev)}
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    dt = vp.VP_BF16 if X.dtype == torch.bfloat16 else vp.VP_F32
    code = f(p(X), p(W), p(y), N, H, V, T, ignore_index, dt, p(out["loss"]), p(out["lse"]), p(out["mean"]),
             p(out["shard_stats"]), p(out["n_bad"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, vp._STATUS.get(code, code)
    return out


CASES = [  # two calls in a row: a larger bf16 case, then a smaller one with other shapes
    (synth.small_case(1000, 256, 6400, 2, "bf16", seed=41, ignore_frac=0.1), 2),
    (synth.small_case(300, 200, 1000, 4, "bf16", seed=42, ignore_frac=0.1), 4),
]


def test_noalloc_matches_workspace_forward_twice():
    f = _noalloc_fn()
    for inp, T in CASES:
        X, W, y = dev_inputs(inp)
        ref = vp.lmhead_ce_fwd(X, W, y, T, shard_stats=True)
        got = _call_noalloc(f, X, W, y, T)
        torch.cuda.synchronize()
        lse = np64(ref["lse"])
        assert_loss_close(np64(got["lse"]), lse, "bf16", what="lse")
        assert_loss_close(np64(got["loss"]), np64(ref["loss"]), "bf16", scale=lse, what="loss")
        assert_loss_close(np64(got["mean"]), np64(ref["mean"]), "bf16", what="mean")
        assert int(got["n_bad"].item()) == int(ref["n_bad"].item())
        st, sr = np64(got["shard_stats"]), np64(ref["shard_stats"])
        scale = np.broadcast_to(np.abs(lse)[None, :], sr[:, 0].shape)
        assert_loss_close(st[:, 0], sr[:, 0], "bf16", scale=scale, what="m_t")
        assert_loss_close(st[:, 2], sr[:, 2], "bf16", scale=scale, what="z_y^(t)")
        assert_loss_close(np.log(st[:, 1]), np.log(sr[:, 1]), "bf16", scale=sr[:, 0], what="log S_t")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    f = _noalloc_fn()
    inp = synth.small_case(64, 64, 512, 2, "bf16", seed=3)
    X, W, y = dev_inputs(inp)
    big_N, big_V = 16384, 128256     # needs ~131 MB of records: refused before any launch
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    loss = torch.empty(64, device="cuda")
    code = f(p(X), p(W), p(y), big_N, 64, big_V, 8, -100, vp.VP_BF16, p(loss), p(loss), None, None, None,
             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 3   # VP_ERR_WORKSPACE
