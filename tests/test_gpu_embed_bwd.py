"""GPU parity of vp_embed_bwd (the tied weight's gradient from the masked
shard lookup) against the float64 oracle.

Tolerance, from the arithmetic: each output element is an fp32 sum of k
values (the existing row, when accumulating, and the k - 1 upstream entries
of its tokens), each exactly representable in fp32.  Any order of k - 1 fp32
additions is within gamma_k * sum |terms| of the exact sum, gamma_k =
k u / (1 - k u), u = 2^-24 (Higham, Accuracy and Stability of Numerical
Algorithms, sec. 4.2).  The tests check that bound element by element."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
import synth
import vocab_lm_head_vp_b300 as vp
from golden_io import read
from gpu_util import dev_inputs, np64, rel_fro

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def _tdt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def _check_sum_bound(got, ids, G64, V, T, dW0=None):
    """|got - exact| <= gamma_k * (|dW0| + sum |dOut|) per element."""
    want = ref.embed_backward(ids, G64, V, T, dW0=dW0)
    mag = ref.embed_backward(ids, np.abs(G64), V, T, dW0=None if dW0 is None else np.abs(dW0))
    valid = ids[(ids >= 0) & (ids < V)]
    k = np.bincount(valid, minlength=V)[:, None] + 1.0
    bound = k * U / (1 - k * U) * mag + 1e-30
    err = np.abs(got - want)
    assert (err <= bound).all(), f"worst {err.max():.3e} vs bound {bound[np.unravel_index(err.argmax(), err.shape)]:.3e}"


def _run(ids, G, V, T, dW=None, accumulate=False):
    out = vp.embed_bwd(torch.from_numpy(ids).cuda(), G, V, T, dW=dW, accumulate=accumulate)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_worked_example_backward(dtype):
    """V=8, T=2, ids [1,6] (sec. 5.2.1): the upstream rows land in weight rows
    1 and 6 only, not in the masked positions' local row 0 (rows 0 and 4)."""
    g = read("embed_v8_t2_ids_1_6.txt")
    V, T = int(g["V"][0]), int(g["T"][0])
    ids = np.array([int(v) for v in g["ids"]])
    H = 8
    G = torch.arange(2 * H, dtype=torch.float32).reshape(2, H).add(1.0).to(_tdt(dtype)).cuda()
    dW = _run(ids, G, V, T)
    want = np.zeros((V, H))
    want[1], want[6] = np64(G)[0], np64(G)[1]
    assert np.array_equal(np64(dW), want)


CASES = [  # N, H, V, T, dtype, ids
    (1, 8, 16, 4, "f32", "uniform"),
    (77, 40, 99, 3, "f32", "uniform"),
    (300, 136, 1000, 8, "bf16", "uniform"),
    (300, 64, 50, 5, "bf16", "uniform"),          # ids repeat ~6 times: segments cross runs
    (1000, 256, 5000, 4, "bf16", "zipf"),         # id 0 spans many runs
    (2049, 64, 700, 2, "bf16", "uniform"),        # n_pad 4096: 8 sorted chunks, one 8-way merge
    (4097, 64, 2048, 2, "bf16", "zipf"),          # n_pad 8192: 16 sorted chunks, 8-way then 2-way merges
    (9000, 128, 4000, 8, "f32", "zipf"),          # n_pad 16384: 32 sorted chunks, 8-way then 4-way merges
    (16384, 64, 128256, 8, "bf16", "uniform"),    # the V128k id count, uniform: mostly one token per id
    (20000, 64, 3000, 4, "bf16", "zipf"),         # n_pad 32768: 64 sorted chunks, two 8-way merges
    (70000, 16, 9000, 3, "bf16", "zipf"),         # n_pad 131072: 256 sorted chunks, 8-, 8- and 4-way merges
]


@pytest.mark.parametrize("accumulate", [False, True])
def test_plan_then_planned_equals_one_call(accumulate):
    """vp_embed_bwd_plan on a side stream (the ids' sort, ahead of time), then
    vp_embed_bwd_planned on the main stream: the same bits as vp_embed_bwd."""
    rng = np.random.default_rng(8)
    N, H, V, T = 9000, 256, 5000, 4
    ids = torch.from_numpy(synth.zipf_ids(rng, N, V, 1.1)).cuda()
    G = torch.from_numpy(rng.standard_normal((N, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    D = torch.from_numpy(rng.standard_normal((V, H)).astype(np.float32)).cuda()
    want = vp.embed_bwd(ids, G, V, T, dW=D.clone() if accumulate else None, accumulate=accumulate)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan = vp.embed_bwd_plan(ids, H, V, T)
    torch.cuda.current_stream().wait_stream(side)
    got = vp.embed_bwd_planned(plan, G, V, T, dW=D.clone() if accumulate else None, accumulate=accumulate)
    torch.cuda.synchronize()
    assert torch.equal(got, want)


@pytest.mark.parametrize("N,H,V,T,dtype,kind", CASES)
def test_embed_bwd_cases(N, H, V, T, dtype, kind):
    rng = np.random.default_rng(N + H + V)
    ids = rng.integers(0, V, N) if kind == "uniform" else synth.zipf_ids(rng, N, V, 1.1)
    ids[: min(N, 4)] = [-1, V, -100, 2 ** 40][: min(N, 4)] if N >= 4 else ids[:N]
    G32 = rng.standard_normal((N, H)).astype(np.float32)
    G = torch.from_numpy(G32).to(_tdt(dtype)).cuda()
    G64 = np64(G)
    dW = torch.full((V, H), float("nan"), device="cuda")
    out = _run(ids, G, V, T, dW=dW)                     # overwrite: every row written
    _check_sum_bound(np64(out), ids, G64, V, T)
    D = rng.standard_normal((V, H)).astype(np.float32)
    acc = torch.from_numpy(D).cuda()
    _run(ids, G, V, T, dW=acc, accumulate=True)
    _check_sum_bound(np64(acc), ids, G64, V, T, dW0=D.astype(np.float64))


def test_embed_bwd_repeatable_and_T_invariant():
    rng = np.random.default_rng(3)
    N, H, V = 2000, 96, 600
    ids = synth.zipf_ids(rng, N, V, 1.1)
    G = torch.from_numpy(rng.standard_normal((N, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    first = _run(ids, G, V, 1)
    for T in (1, 2, 3, 4, 6, 8, 600):
        assert torch.equal(_run(ids, G, V, T), first), T


def test_embed_bwd_full_size_sampled_rows():
    """V128k shapes (N=16384, H=4096, V=128256) with Zipf ids, overwrite mode:
    every row of a sample of vocab ids -- the most frequent (its tokens span
    dozens of runs), random ones and never-seen ones -- against the oracle."""
    wl = synth.WORKLOADS["v128k"]
    rng = np.random.default_rng(wl.seed)
    ids = synth.zipf_ids(rng, wl.N, wl.V, 1.1)
    g = torch.Generator(device="cuda").manual_seed(7)
    G = torch.randn(wl.N, wl.H, generator=g, device="cuda").to(torch.bfloat16)
    dW = _run(ids, G, wl.V, wl.T)
    rows = np.unique(np.concatenate([np.arange(8), rng.choice(wl.V, 40, replace=False)]))
    # the oracle on the sampled rows only: ids of the sample renumbered 0..len-1, others out of range
    remap = np.full(wl.V, -1, dtype=np.int64)
    remap[rows] = np.arange(len(rows))
    sub_ids = np.where((ids >= 0) & (ids < wl.V), remap[np.clip(ids, 0, wl.V - 1)], -1)
    G64 = np64(G)
    got = np64(dW[torch.from_numpy(rows).cuda()])
    _check_sum_bound(got, sub_ids, G64, len(rows), 1)
    assert np.bincount(ids, minlength=wl.V)[0] > 32 * 10          # id 0 really crosses many runs


def test_tied_weight_gradient():
    """The tied weight's full gradient: LM head dW (vp_lmhead_ce_fwd_bwd) plus
    the embedding's (vp_embed_bwd, accumulate) against the oracle's sum."""
    inp = synth.small_case(256, 128, 1000, 4, "bf16", seed=5, ignore_frac=0.1)
    X, W, y = dev_inputs(inp)
    o = vp.lmhead_ce_fwd_bwd(X, W, y, 4)
    ids = np.random.default_rng(6).integers(0, 1000, 256)
    G = torch.from_numpy(np.random.default_rng(7).standard_normal((256, 128)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    vp.embed_bwd(torch.from_numpy(ids).cuda(), G, 1000, 4, dW=o["dW"], accumulate=True)
    torch.cuda.synchronize()
    b = ref.lmhead_ce_backward(inp.X, inp.W, inp.targets, 1000)
    want = ref.embed_backward(ids, np64(G), 1000, 4, dW0=b["dW"])
    assert rel_fro(np64(o["dW"]), want) <= 2e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_embed_sp_ranks(dtype):
    """SP on: every rank's slice bit-exact against the oracle's reduce-scatter,
    the V=8 worked table included (rank 0 keeps E1, rank 1 E6)."""
    g = read("embed_v8_t2_ids_1_6.txt")
    V, T = int(g["V"][0]), int(g["T"][0])
    ids = np.array([int(v) for v in g["ids"]])
    W = torch.arange(V * 8, dtype=torch.float32).reshape(V, 8).add(1.0).to(_tdt(dtype)).cuda()
    for r in range(T):
        out = vp.embed_fwd_sp(torch.from_numpy(ids).cuda(), W, T, r)
        assert np.array_equal(np64(out), ref.embed_sp(ids, np64(W), V, T, r)), r
    rng = np.random.default_rng(4)
    V, H, N, T = 1200, 136, 960, 8
    ids = rng.integers(-5, V + 5, N)
    Wn = torch.from_numpy(rng.standard_normal((V, H)).astype(np.float32)).to(_tdt(dtype))
    Wn[7, 3] = -0.0
    ids[0] = 7
    Wd = Wn.cuda()
    W64 = np64(Wn)
    idt = torch.from_numpy(ids).cuda()
    for r in range(T):
        out = vp.embed_fwd_sp(idt, Wd, T, r)
        torch.cuda.synchronize()
        want = ref.embed_sp(ids, W64, V, T, r)
        assert np.array_equal(np64(out), want), r
        if r == 0:
            bits = out.view(torch.int16 if dtype == "bf16" else torch.int32).cpu().numpy()
            assert bits[0, 3] == 0          # -0.0 came out +0.0
