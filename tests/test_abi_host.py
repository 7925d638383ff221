"""libvp on the host, without a GPU: it loads, exports every function that
include/*.h declares, and rejects bad arguments before launching anything."""
import ctypes
import glob
import os
import re

import pytest

import vocab_lm_head_vp_b300 as vp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(vp_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from vocab_lm_head_vp_b300 import build
    build.build()
    return vp._load()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"vp_embed_fwd", "vp_lmhead_ce_fwd", "vp_lmhead_ce_bwd", "vp_lmhead_ce_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libvp.so does not export {n}"


def test_status_strings(lib):
    for code, name in vp._STATUS.items():
        assert lib.vp_status_string(code).decode() == name
    assert b"sm_103a" in lib.vp_version()


P = ctypes.c_void_p


def test_embed_rejects_bad_arguments(lib):
    ids, W, out = P(0x1000), P(0x2000), P(0x3000)
    f = lib.vp_embed_fwd
    assert f(ids, W, out, 4, 8, 10, 3, vp.VP_BF16, None) == 1       # V % T != 0
    assert f(None, W, out, 4, 8, 10, 2, vp.VP_BF16, None) == 1      # null ids
    assert f(ids, W, out, 0, 8, 10, 2, vp.VP_BF16, None) == 1       # N = 0
    assert f(ids, W, out, 4, 8, 10, 2, 7, None) == 1                # unknown dtype
    assert f(ids, P(0x2008), out, 4, 8, 10, 2, vp.VP_BF16, None) == 2  # W not 16-byte aligned
    assert f(ids, W, out, 4, 6, 10, 2, vp.VP_BF16, None) == 2       # H*2 not a multiple of 16
    assert f(ids, W, out, 4, 3, 10, 2, vp.VP_F32, None) == 2        # H*4 not a multiple of 16


def test_ce_rejects_bad_arguments(lib):
    X, W, y, ws = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    loss, lse = P(0x50000), P(0x60000)
    fwd = lib.vp_lmhead_ce_fwd
    args = lambda **k: dict(dict(X=X, W=W, y=y, N=6, H=64, V=16, T=4, dt=vp.VP_F32, loss=loss, lse=lse, ws=ws,
                                 wsb=1 << 20), **k)

    def call(a):
        return fwd(a["X"], a["W"], a["y"], a["N"], a["H"], a["V"], a["T"], -100, a["dt"], a["loss"], a["lse"],
                   None, None, None, a["ws"], a["wsb"], None)
    assert call(args(T=5)) == 1
    assert call(args(loss=None)) == 1
    assert call(args(X=None)) == 1
    assert call(args(V=-16)) == 1
    assert call(args(X=P(0x10004))) == 2
    assert call(args(H=63)) == 2
    assert call(args(wsb=16)) == 3                                   # workspace too small
    bwd = lib.vp_lmhead_ce_bwd
    assert bwd(X, W, y, lse, None, None, 6, 64, 16, 3, -100, vp.VP_F32, P(0x70000), P(0x80000), ws, 1 << 20,
               None) == 1
    assert bwd(X, W, y, None, None, None, 6, 64, 16, 4, -100, vp.VP_F32, P(0x70000), P(0x80000), ws, 1 << 20,
               None) == 1
    assert bwd(X, W, y, lse, None, None, 6, 64, 16, 4, -100, vp.VP_F32, P(0x70008), P(0x80000), ws, 1 << 20,
               None) == 2
    assert bwd(X, W, y, lse, None, None, 6, 64, 16, 4, -100, vp.VP_F32, P(0x70000), P(0x80000), ws, 64, None) == 3


SK = 2 * 160 * 256 * 256 * 4   # bf16 backward: stream-K partial tiles of the dX GEMM


def XT(rows, H):                # bf16 backward: X^T (rows rounded up to 8) for the dW GEMM
    return H * ((rows + 7) // 8 * 8) * 2


def test_workspace_sizes(lib):
    N, H, V, T = 16384, 4096, 128256, 8
    fwd = vp.workspace_size(N, H, V, T, vp.VP_BF16, 0)
    # records: ceil(V/256) tiles x 2 segment slots x N tokens x (m, R) fp32, plus z_y
    assert fwd >= 501 * 2 * N * 8 + N * 4 and fwd < 501 * 2 * N * 8 + N * 4 + 4096
    one = vp.workspace_size(N, H, V, T, vp.VP_BF16, 1, V)
    one_body = N * V * 2 + SK + XT(N, H)
    assert one_body <= one < one_body + N * 4 + 4096       # one chunk: bf16 dZ, no fp32 dX partial
    # default: one shard's dZ (V/T = 16032 rounded up to 16128) plus the fp32 dX partial
    d = vp.workspace_size(N, H, V, T, vp.VP_BF16, 1)
    d_body = N * 16128 * 2 + N * H * 4 + SK + XT(N, H)
    assert d_body <= d < d_body + N * 4 + 4096
    assert vp.workspace_size(N, H, V, T, vp.VP_BF16, 1, 16032) == d
    assert vp.workspace_size(N, H, V, 1, vp.VP_BF16, 1) == one          # T = 1: the shard is all of V
    assert vp.workspace_size(N, H, V, 7, vp.VP_BF16, 1) == 0           # V % T != 0
    assert vp.workspace_size(6, 64, 16, 4, vp.VP_F32, 4) == 0          # unknown pass


def test_fused_workspace_sizes(lib):
    N, H, V, T = 16384, 4096, 128256, 8
    full = vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, N)
    # fp16 p / bf16 dZ [N, V] + per tile and token: 2 (m, R) slots, the tile max; + z_y, g
    body = N * V * 2 + 501 * N * (2 * 8 + 4) + 2 * N * 4 + SK + XT(N, H)
    assert body <= full < body + 8192
    half = vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, 8192)
    assert half - SK < (full - SK) / 2 + N * 8 and half - SK > (full - SK) / 2 - N * V - XT(N, H)
    assert vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, 100) == vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, 128)
    # default: saved probabilities of at most 1.25 GiB, in the chunk that fills the dX GEMM's
    # waves best by the dX cost model (4608 token rows of V = 128256: 288 tiles of 256 x 256, two waves
    # of 148, three chunks and one of 2560 rows)
    assert vp.workspace_size(N, H, V, T, vp.VP_BF16, 2) == vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, 4608)
    # small problems fit in one chunk by default
    assert vp.workspace_size(4096, 512, 6400, 2, vp.VP_BF16, 2) == vp.workspace_size(4096, 512, 6400, 2,
                                                                                        vp.VP_BF16, 2, 4096)
    # fp32: the larger of the split forward and backward
    f32 = vp.workspace_size(6, 64, 16, 4, vp.VP_F32, 2)
    assert f32 == max(vp.workspace_size(6, 64, 16, 4, vp.VP_F32, 0), vp.workspace_size(6, 64, 16, 4, vp.VP_F32, 1))


def test_fused_rejects_bad_arguments(lib):
    X, W, y, ws = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    loss, lse, dX, dW = P(0x50000), P(0x60000), P(0x70000), P(0x80000)
    f = lib.vp_lmhead_ce_fwd_bwd

    def call(N=300, H=64, V=1000, T=4, dt=vp.VP_BF16, X=X, dX=dX, dW=dW, wsb=1 << 30):
        return f(X, W, y, None, None, N, H, V, T, -100, dt, loss, lse, None, None, None, dX, dW, ws, wsb, None)
    assert call(T=3) == 1                    # V % T != 0
    assert call(dX=None) == 1
    assert call(dW=None) == 1
    assert call(X=P(0x10008)) == 2           # X not 16-byte aligned
    assert call(dX=P(0x70008)) == 2
    assert call(H=60) == 2                   # H * 2 bytes not a multiple of 16
    assert call(wsb=4096) == 3               # no token chunk fits
    assert call(dt=vp.VP_F32, wsb=64) == 3


def test_embed_bwd_rejects_bad_arguments(lib):
    ids, G, dW, ws = P(0x1000), P(0x2000), P(0x3000), P(0x4000)
    f = lib.vp_embed_bwd
    nb = lib.vp_embed_bwd_workspace_size(100, 64, 1000, 4, vp.VP_BF16)
    # sort keys (next power of two of N) + two partial sums of H floats per 32-token run
    assert nb >= 128 * 8 + 2 * 4 * 64 * 4
    assert lib.vp_embed_bwd_workspace_size(100, 64, 1000, 3, vp.VP_BF16) == 0     # V % T != 0
    assert f(ids, G, dW, 100, 64, 1000, 3, vp.VP_BF16, 0, ws, nb, None) == 1
    assert f(None, G, dW, 100, 64, 1000, 4, vp.VP_BF16, 0, ws, nb, None) == 1
    assert f(ids, P(0x2008), dW, 100, 64, 1000, 4, vp.VP_BF16, 0, ws, nb, None) == 2
    assert f(ids, G, P(0x3004), 100, 64, 1000, 4, vp.VP_BF16, 0, ws, nb, None) == 2
    assert f(ids, G, dW, 100, 60, 1000, 4, vp.VP_BF16, 0, ws, nb, None) == 2   # H*2 % 16 != 0
    assert f(ids, G, dW, 100, 64, 1000, 4, vp.VP_BF16, 0, ws, 64, None) == 3


def test_embed_sp_rejects_bad_arguments(lib):
    ids, W, out = P(0x1000), P(0x2000), P(0x3000)
    f = lib.vp_embed_fwd_sp
    assert f(ids, W, out, 10, 8, 16, 4, 0, vp.VP_BF16, None) == 1     # N % T != 0
    assert f(ids, W, out, 12, 8, 16, 4, 4, vp.VP_BF16, None) == 1     # rank >= T
    assert f(ids, W, out, 12, 8, 16, 4, -1, vp.VP_BF16, None) == 1
    assert f(ids, W, P(0x3008), 12, 8, 16, 4, 1, vp.VP_BF16, None) == 2


def test_rejects_tile_counts_beyond_int32(lib):
    X, W, y, ws = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    loss, lse = P(0x50000), P(0x60000)
    N, V = (1 << 31) - 1, (1 << 31) - 2          # 2^24 x 2^23 logits tiles
    assert lib.vp_lmhead_ce_fwd(X, W, y, N, 64, V, 2, -100, vp.VP_BF16, loss, lse, None, None, None, ws, 1 << 40,
                                None) == 2


def test_keep_saved_rejects_bad_arguments(lib):
    X, W, y, sv = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    loss, lse, dX, dW = P(0x50000), P(0x60000), P(0x70000), P(0x80000)
    N, H, V, T = 16384, 4096, 128256, 8
    full = vp.workspace_size(N, H, V, T, vp.VP_BF16, 3)
    assert full == vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, N)  # the whole batch's fused state
    fk, bs = lib.vp_lmhead_ce_fwd_keep, lib.vp_lmhead_ce_bwd_saved
    assert fk(X, W, y, 300, 64, 1000, 3, -100, vp.VP_BF16, loss, lse, None, None, None, sv, 1 << 30, None) == 1
    assert fk(X, W, y, 300, 64, 1000, 4, -100, vp.VP_BF16, None, lse, None, None, None, sv, 1 << 30, None) == 1
    assert fk(X, W, y, 300, 64, 1000, 4, -100, vp.VP_BF16, loss, lse, None, None, None, P(0x40008), 1 << 30,
              None) == 2
    assert fk(X, W, y, 300, 64, 1000, 4, -100, vp.VP_BF16, loss, lse, None, None, None, sv, 4096, None) == 3
    assert bs(X, W, y, lse, None, None, 300, 64, 1000, 4, -100, vp.VP_BF16, None, dW, sv, 1 << 30, None) == 1
    assert bs(X, W, y, lse, None, None, 300, 64, 1000, 4, -100, vp.VP_BF16, P(0x70008), dW, sv, 1 << 30,
              None) == 2
    assert bs(X, W, y, lse, None, None, 300, 64, 1000, 4, -100, vp.VP_BF16, dX, dW, sv, 4096, None) == 3


def test_stage_timing_off_records_nothing(lib):
    # Disabled (the default), no region is recorded or counted as dropped;
    # disabling again resets the dropped count.
    assert lib.vp_stage_timing_enable(0) == 0
    assert lib.vp_stage_timing_dropped() == 0
    ms = (ctypes.c_float * 16)()
    k = lib.vp_stage_timing_read(ms, None, 16)
    assert k > 0 and lib.vp_stage_name(k - 1) and not lib.vp_stage_name(k)
    assert all(x == 0.0 for x in ms)


def test_suggested_workspaces_are_accepted(lib):
    """For seeded random shapes and chunks, the bytes vp_lmhead_ce_workspace_size
    suggests pass the call's workspace check: without a GPU the call then stops
    at the driver (VP_ERR_CUDA), never at VP_ERR_WORKSPACE.  Small workspaces,
    where the sections' 256-byte alignment weighs against the rows, included
    (N=376, H=56, V=1512, T=7 with 128-token chunks was once refused)."""
    import numpy as np
    X, W, y, ws = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    loss, lse, dX, dW = P(0x50000), P(0x60000), P(0x70000), P(0x80000)
    rng = np.random.default_rng(11)
    shapes = [(376, 56, 1512, 7, 128)]
    for _ in range(300):
        T = int(rng.choice([1, 2, 3, 4, 7, 8, 16]))
        shapes.append((int(rng.integers(1, 5000)), 8 * int(rng.integers(1, 80)), T * int(rng.integers(1, 600)), T,
                       int(rng.choice([0, 128, 256, 384, 1000]))))
    for N, H, V, T, chunk in shapes:
        nb = vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, chunk)
        code = lib.vp_lmhead_ce_fwd_bwd(X, W, y, None, None, N, H, V, T, -100, vp.VP_BF16, loss, lse, None, None,
                                        None, dX, dW, ws, nb, None)
        assert code == 4, (N, H, V, T, chunk, code)
        vc = int(rng.choice([0, 256, 512, 1000]))
        nb = vp.workspace_size(N, H, V, T, vp.VP_BF16, 1, vc)
        code = lib.vp_lmhead_ce_bwd(X, W, y, lse, None, None, N, H, V, T, -100, vp.VP_BF16, dX, dW, ws, nb, None)
        assert code == 4, (N, H, V, T, vc, code)


def test_dx_plan_choices(lib):
    """The dX GEMM's tile choice, host arithmetic only (cost in waves of
    128 x 256 tiles on the persistent grid: a 256-row wave counts 2, a 128-row
    wave 1.15; the lower cost wins, 256 rows on a tie)."""
    vp.set_gemm_variant(0)
    cases = [
        # rows, H, SMs -> tile rows, stream-K, cost
        # a V = 128256 token chunk: 576 tiles of 128 rows = 4 waves (4.6) against 288 of 256 rows = 2 waves (4)
        (4608, 4096, 148, 256, False, 4.0),
        # its 2560-row tail chunk: 320 tiles = 3 waves (3.45) against 160 = 2 waves (4)
        (2560, 4096, 148, 128, False, 3.45),
        # N = 8192 (V32k): 1024 tiles = 7 waves (8.05) against 512 = 4 waves (8)
        (8192, 4096, 148, 256, False, 8.0),
        # N = 16384, the split path's dX: 2048 = 14 waves (16.1) against 1024 = 7 waves (14)
        (16384, 4096, 148, 256, False, 14.0),
        # N = 32768, H = 5120 (20 column tiles): 5120 = 35 waves (40.25) against 2560 = 18 waves (36)
        (32768, 5120, 148, 256, False, 36.0),
        # MiniMind (H = 512, 2 column tiles): 64 tiles in one wave (1.15) against 32 (2); 32 tiles of
        # 256 rows are fewer than a quarter of the SMs, so no stream-K
        (4096, 512, 148, 128, False, 1.15),
        # 40 tiles of 256 rows (>= 148 / 4, < 148) and one wave (1.15) for 80 tiles' work (0.54):
        # stream-K over 256-row tiles, cost the work per CTA
        (2560, 1024, 148, 256, True, 80 / 148),
        # the same token chunk on 132 SMs: 576 tiles = 5 waves (5.75) against 288 = 3 waves (6)
        (4608, 4096, 132, 128, False, 5.75),
    ]
    for rows, H, sms, tile_rows, streamk, cost in cases:
        p = vp.dx_plan(rows, H, sms)
        assert (p["tile_rows"], p["streamk"]) == (tile_rows, streamk), (rows, H, sms, p)
        assert abs(p["cost"] - cost) < 1e-9, (rows, H, sms, p)
    # the shapes of the GPU test of the dX tile forms (test_gpu_ce.py), on 148 SMs: stream-K where
    # it expects the GEMM and its fix-up pass
    for rows, H, streamk in [(300, 264, False), (1100, 512, False), (77, 64, False), (2600, 1032, True),
                             (768, 4096, True), (700, 4104, True)]:
        assert vp.dx_plan(rows, H, 148)["streamk"] == streamk, (rows, H)
    # GEMM form 2 keeps 128-row tiles and no stream-K
    vp.set_gemm_variant(2)
    try:
        assert vp.dx_plan(8192, 4096, 148) == {"tile_rows": 128, "streamk": False, "cost": 1.15 * 7}
    finally:
        vp.set_gemm_variant(0)
    d, sk, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
    for args in [(0, 4096, 148), (4096, 0, 148), (4096, 4096, 0)]:
        assert lib.vp_test_dx_plan(*args, ctypes.byref(d), ctypes.byref(sk), ctypes.byref(c)) == 1
    assert lib.vp_test_dx_plan(4096, 4096, 148, None, ctypes.byref(sk), ctypes.byref(c)) == 1
