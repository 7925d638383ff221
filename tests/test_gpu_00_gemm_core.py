"""The tcgen05 GEMM core alone against a float64 matmul of the same bf16
operands, for every operand major-ness the path uses, on sizes with several
tiles and ragged tails, in both forms (one 256x256 tile per SM pair, one
128x256 tile per SM).  Collected first: a core fault stops the GPU run."""
import numpy as np
import pytest
import torch

import vocab_lm_head_vp_b300 as vp

pytestmark = pytest.mark.gpu

SHAPES = [(128, 256, 64), (304, 520, 200), (1024, 768, 1024), (136, 264, 4104), (8, 8, 8)]


@pytest.fixture(params=["pair", "single"])
def variant(request):
    vp.set_gemm_variant(request.param == "pair")
    yield request.param
    vp.set_gemm_variant(False)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_core(M, N, K, a_mn, b_mn, variant):
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    Ad = (A.t().contiguous() if a_mn else A).cuda()
    Bd = (B.t().contiguous() if b_mn else B).cuda()
    D, ws = vp.test_gemm_bf16(Ad, Bd, bool(a_mn), bool(b_mn))
    torch.cuda.synchronize()
    assert vp.read_device_status(ws) == 0
    ref = A.double() @ B.double().t()
    got = D.cpu().double()
    # fp32 accumulation of exact bf16 products: error ~ K * 2^-24 * |a||b|
    err = (got - ref).abs().max().item()
    assert err <= 1e-5 * K ** 0.5 * 4 + 1e-6 * ref.abs().max().item(), f"max err {err}"
