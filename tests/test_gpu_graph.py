"""The library's calls enqueue only asynchronous work (a status memset and
kernels; tensor maps are encoded on the host), so a whole training step of
the path can be captured once in a CUDA graph and replayed.  Replays give the
eager calls' results bit for bit."""
import numpy as np
import pytest
import torch

import synth
import vocab_lm_head_vp_b300 as vp
from gpu_util import dev_inputs

pytestmark = pytest.mark.gpu


def test_fused_step_in_a_cuda_graph():
    inp = synth.small_case(640, 256, 3000, 6, "bf16", seed=51, ignore_frac=0.1)
    X, W, y = dev_inputs(inp)
    N, H = X.shape
    V, T = W.shape[0], 6
    ids = torch.from_numpy(np.random.default_rng(2).integers(0, V, N)).cuda()
    emb = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 2), dtype=torch.uint8, device="cuda")
    ews = torch.empty(vp._load().vp_embed_bwd_workspace_size(N, H, V, T, vp.VP_BF16), dtype=torch.uint8,
                      device="cuda")
    out = {"loss": torch.empty(N, device="cuda"), "lse": torch.empty(N, device="cuda"),
           "mean": torch.empty(1, device="cuda"), "n_bad": torch.empty(1, dtype=torch.int32, device="cuda"),
           "dX": torch.empty_like(X), "dW": torch.empty((V, H), device="cuda")}

    def step():
        vp.embed_fwd(ids, W, T, out=emb)
        vp.lmhead_ce_fwd_bwd(X, W, y, T, workspace=ws, out=out)
        vp.embed_bwd(ids, emb, V, T, dW=out["dW"], accumulate=True, workspace=ews)   # tied weight

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # eager, also the first-call set-up
        torch.cuda.synchronize()
        eager = {k: out[k].clone() for k in ("loss", "lse", "mean", "dX", "dW")}
        eager_emb = emb.clone()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for k in ("loss", "lse", "dX", "dW"):
            out[k].zero_()
        emb.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert vp.read_device_status(ws) == 0
        for k, v in eager.items():
            assert torch.equal(out[k], v), k
        assert torch.equal(emb, eager_emb)


def _outputs(X, V):
    N, H = X.shape
    dev = X.device
    return {"loss": torch.empty(N, device=dev), "lse": torch.empty(N, device=dev), "mean": torch.empty(1, device=dev),
            "n_bad": torch.empty(1, dtype=torch.int32, device=dev), "dX": torch.empty_like(X),
            "dW": torch.empty((V, H), device=dev)}


@pytest.mark.parametrize("path", ["fused", "split"])
def test_graph_replay_on_new_inputs(path):
    """One capture, replayed after other X, W and targets (another ignored
    fraction, so another valid count and upstream scale) are copied into its
    buffers: each replay equals eager calls on those inputs.  Fused with two
    token chunks, split with three vocab chunks."""
    N, H, V, T = 1100, 512, 3000, 4
    cases = [dev_inputs(synth.small_case(N, H, V, T, "bf16", seed=s, ignore_frac=f)) for s, f in ((5, 0.1), (6, 0.3))]
    dev = cases[0][0].device

    def workspaces():
        if path == "fused":
            return [torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, 640), dtype=torch.uint8, device=dev)]
        return [torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 0), dtype=torch.uint8, device=dev),
                torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 1, 1024), dtype=torch.uint8, device=dev)]

    def step(X, W, y, o, ws):
        if path == "fused":
            vp.lmhead_ce_fwd_bwd(X, W, y, T, workspace=ws[0], out=o)
        else:
            vp.lmhead_ce_fwd(X, W, y, T, workspace=ws[0], out=o)
            vp.lmhead_ce_bwd(X, W, y, o["lse"], T, workspace=ws[1], dX=o["dX"], dW=o["dW"], vocab_chunk=1024)

    X, W, y = (t.clone() for t in cases[0])
    o, ws = _outputs(X, V), workspaces()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(X, W, y, o, ws)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step(X, W, y, o, ws)
    torch.cuda.current_stream().wait_stream(side)
    for Xs, Ws, ys in cases[::-1]:
        X.copy_(Xs)
        W.copy_(Ws)
        y.copy_(ys)
        graph.replay()
        e, ews = _outputs(Xs, V), workspaces()
        step(Xs, Ws, ys, e, ews)
        torch.cuda.synchronize()
        assert all(vp.read_device_status(w) == 0 for w in ws + ews)
        for k in ("loss", "lse", "mean", "dX", "dW"):
            assert torch.equal(o[k], e[k]), k
