"""The allocation-free forward, vp_lmhead_ce_fwd_noalloc, called through the C
ABI, against the workspace forward vp_lmhead_ce_fwd on the same inputs.

It serves callers that cannot allocate device memory (a plugin given only its
input and output buffers, a loop that must never call cudaMalloc); its scratch
is a fixed 32 MiB array inside libvp, shared by every call.  It launches the
same kernels with the same launch shapes as the workspace forward, so every
output must be bit-identical.  Calls in a row with different shapes and dtypes
check that the leftovers of one call do not leak into the next.  This file is
collected last on purpose."""
import ctypes

import pytest
import torch

import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import dev_inputs

pytestmark = pytest.mark.gpu
KEYS = ("loss", "lse", "mean", "n_bad", "shard_stats")


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(X, W, y, T, ignore_index=-100, expect=0):
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    out = {"loss": torch.full((N,), float("nan"), device=dev), "lse": torch.full((N,), float("nan"), device=dev),
           "mean": torch.full((1,), float("nan"), device=dev),
           "n_bad": torch.full((1,), -1, dtype=torch.int32, device=dev),
           "shard_stats": torch.full((T, 3, N), float("nan"), device=dev)}
    dt = vp.VP_BF16 if X.dtype == torch.bfloat16 else vp.VP_F32
    code = vp._load().vp_lmhead_ce_fwd_noalloc(
        _p(X), _p(W), _p(y), N, H, V, T, ignore_index, dt, _p(out["loss"]), _p(out["lse"]), _p(out["mean"]),
        _p(out["shard_stats"]), _p(out["n_bad"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == expect, vp._STATUS.get(code, code)
    return out


CASES = [  # calls in a row: a larger bf16 case, the tiny fp32 config, a smaller bf16 case
    (synth.small_case(1000, 256, 6400, 2, "bf16", seed=41, ignore_frac=0.1), 2),
    (synth.make_inputs("tiny"), 4),
    (synth.small_case(300, 200, 1000, 4, "bf16", seed=42, ignore_frac=0.1), 4),
    (synth.small_case(77, 40, 99, 3, "f32", seed=43, ignore_frac=0.1), 3),
]


def test_noalloc_bit_identical_to_workspace_forward():
    for _ in range(2):
        for inp, T in CASES:
            X, W, y = dev_inputs(inp)
            want = vp.lmhead_ce_fwd(X, W, y, T, shard_stats=True)
            got = _call_noalloc(X, W, y, T)
            torch.cuda.synchronize()
            for k in KEYS:
                assert torch.equal(got[k], want[k]), (inp.wl.name, k)


def test_noalloc_wait_failure_shows_as_nan():
    """A GEMM wait that runs out (the diagnostic hold of the TMA producer) makes
    the merge write NaN: the status word of the shared array is not readable
    through vp_read_device_status, so the outputs carry the failure.  The next
    call computes normally again."""
    inp, T = CASES[2]
    X, W, y = dev_inputs(inp)
    vp.set_wait_fault(1, 50_000_000)
    try:
        bad = _call_noalloc(X, W, y, T)
        torch.cuda.synchronize()
    finally:
        vp.set_wait_fault(0, 0)
    assert torch.isnan(bad["loss"]).all() and torch.isnan(bad["lse"]).all() and torch.isnan(bad["mean"]).all()
    want = vp.lmhead_ce_fwd(X, W, y, T, shard_stats=True)
    got = _call_noalloc(X, W, y, T)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(got[k], want[k]), k


def test_noalloc_rejects_sizes_beyond_its_scratch():
    inp = synth.small_case(64, 64, 512, 2, "bf16", seed=3)
    X, W, y = dev_inputs(inp)
    big_N, big_V = 16384, 128256     # needs ~131 MB of records: refused before any launch
    loss = torch.empty(64, device="cuda")
    code = vp._load().vp_lmhead_ce_fwd_noalloc(
        _p(X), _p(W), _p(y), big_N, 64, big_V, 8, -100, vp.VP_BF16, _p(loss), _p(loss), None, None, None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 3   # VP_ERR_WORKSPACE
