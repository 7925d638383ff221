"""Per-launch event timing used by the benchmark: every timed region lands in its
stage, and regions past the enabled capacity are counted, never silently lost."""
import pytest
import torch

import vocab_lm_head_vp_b300 as vp

pytestmark = pytest.mark.gpu


def _gather(k):
    torch.manual_seed(0)
    W = torch.randn(1024, 256, device="cuda", dtype=torch.bfloat16)
    ids = torch.randint(0, 1024, (512,), device="cuda", dtype=torch.int64)
    for _ in range(k):
        vp.embed_fwd(ids, W, 4)
    torch.cuda.synchronize()


def test_stage_timing_counts_every_launch():
    vp.stage_timing_enable(8)
    try:
        _gather(3)
        st = vp.stage_timing_read()
    finally:
        vp.stage_timing_enable(0)
    ms, n = st["embed_gather"]
    assert n == 3 and ms > 0.0
    assert all(c == 0 for name, (_, c) in st.items() if name != "embed_gather")


def test_stage_timing_rejects_partial_totals():
    vp.stage_timing_enable(2)
    try:
        _gather(3)
        assert vp._load().vp_stage_timing_dropped() == 1
        with pytest.raises(RuntimeError, match="not recorded"):
            vp.stage_timing_read()
    finally:
        vp.stage_timing_enable(0)
    assert vp._load().vp_stage_timing_dropped() == 0
