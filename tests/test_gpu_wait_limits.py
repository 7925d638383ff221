"""The bounded waits of the tcgen05 GEMMs, made to run out on purpose.

Every mbarrier wait in the GEMM core gives up after a time limit, records a bit
in the device status word and lets the CTA drain what it issued, free its
tensor memory and exit.  vp_test_set_wait_fault holds one role back (no TMA
load, or no MMA) with a short limit, so the other roles' waits run out.  The
tests read the status bits, check that the forward's outputs come out NaN, and
then check that a normal call right after still matches the oracle: the
context stays usable, tensor memory was freed and no load was left in flight.
No wait is removed and nothing is left unbounded; only the first role's work
is skipped."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import assert_loss_close, dev_inputs, np64, rel_fro

pytestmark = pytest.mark.gpu

WAIT_NS = 50_000_000   # 50 ms
PRODUCER, MMA, EPILOGUE = 0x1, 0x2, 0x4


@pytest.fixture
def inp():
    # H = 512: 8 K blocks per tile, more than the pipeline's 4 stages (6 on SM
    # pairs), so a producer whose stages are never released blocks with loads
    # in flight
    return synth.small_case(256, 512, 1024, 2, "bf16", seed=31)


@pytest.fixture(autouse=True)
def _restore():
    yield
    vp.set_wait_fault(0, 0)
    vp.set_gemm_variant(0)


def _normal_call_matches_oracle(inp):
    X, W, y = dev_inputs(inp)
    f = vp.lmhead_ce_fwd(X, W, y, 2)
    dX, dW = vp.lmhead_ce_bwd(X, W, y, f["lse"], 2)
    torch.cuda.synchronize()
    assert vp.read_device_status(f["workspace"]) == 0
    o = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, inp.wl.V, 2)
    assert_loss_close(np64(f["loss"]), o["loss"], "bf16")
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, inp.wl.V)
    assert rel_fro(np64(dX), b["dX"]) <= 2e-2 and rel_fro(np64(dW), b["dW"]) <= 2e-2


@pytest.mark.parametrize("variant", [0, 1, 3])   # the forward GEMM on one SM per tile, on SM pairs, in multicast clusters
@pytest.mark.parametrize("mode,bits", [(1, MMA | EPILOGUE), (2, PRODUCER | EPILOGUE)])
def test_forward_wait_runs_out_then_recovers(inp, mode, bits, variant):
    X, W, y = dev_inputs(inp)
    vp.set_gemm_variant(variant)
    vp.set_wait_fault(mode, WAIT_NS)
    f = vp.lmhead_ce_fwd(X, W, y, 2, shard_stats=True)
    torch.cuda.synchronize()
    assert vp.read_device_status(f["workspace"]) == bits
    assert torch.isnan(f["loss"]).all() and torch.isnan(f["lse"]).all()
    assert torch.isnan(f["shard_stats"]).all() and torch.isnan(f["mean"]).all()
    vp.set_wait_fault(0, 0)
    _normal_call_matches_oracle(inp)


def test_fused_call_reports_and_recovers(inp):
    X, W, y = dev_inputs(inp)
    vp.set_wait_fault(2, WAIT_NS)
    o = vp.lmhead_ce_fwd_bwd(X, W, y, 2)
    torch.cuda.synchronize()
    # every GEMM of the call gave up (forward and dX on one SM per tile, dW^T on SM pairs);
    # the forward's outputs are NaN
    assert vp.read_device_status(o["workspace"]) == PRODUCER | EPILOGUE
    assert torch.isnan(o["loss"]).all() and torch.isnan(o["lse"]).all()
    vp.set_wait_fault(0, 0)
    o = vp.lmhead_ce_fwd_bwd(X, W, y, 2)
    torch.cuda.synchronize()
    assert vp.read_device_status(o["workspace"]) == 0
    f = ref.lmhead_ce_forward(inp.X, inp.W, inp.targets, inp.wl.V, 2)
    assert_loss_close(np64(o["loss"]), f["loss"], "bf16")
    _normal_call_matches_oracle(inp)
