"""Python binding of libvp: vocab-parallel embedding and fused LM head +
vocab-parallel cross-entropy on one B300.

Argument marshalling only: every step of the path runs in libvp's CUDA
kernels; torch tensors supply device memory and the current stream.  There is
no fallback: without the built ``libvp.so`` every call raises.

    out = embed_fwd(ids, W, T)
    fwd = lmhead_ce_fwd(X, W, targets, T, ignore_index=-100)   # loss, lse, mean ...
    dX, dW = lmhead_ce_bwd(X, W, targets, fwd["lse"], T)
    out = lmhead_ce_fwd_bwd(X, W, targets, T)                   # both, probabilities saved
    loss = lmhead_ce(X, W, targets, T)                          # autograd wrapper
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["embed_fwd", "embed_fwd_sp", "embed_bwd", "embed_bwd_plan", "embed_bwd_planned", "lmhead_ce_fwd", "lmhead_ce_bwd", "lmhead_ce_fwd_bwd", "lmhead_ce",
           "lmhead_ce_shard_fwd", "lmhead_ce_merge_stats", "lmhead_ce_shard_bwd", "vocab_parallel_lmhead_ce", "workspace_size", "read_device_status",
           "test_gemm_bf16", "set_gemm_variant", "dx_plan", "set_wait_fault", "stage_timing_enable", "stage_timing_read", "VpError", "library_path", "VP_F32", "VP_BF16", "IGNORE_INDEX"]

VP_F32, VP_BF16 = 0, 1
IGNORE_INDEX = -100
_STATUS = {0: "VP_OK", 1: "VP_ERR_INVALID_ARG", 2: "VP_ERR_UNSUPPORTED", 3: "VP_ERR_WORKSPACE", 4: "VP_ERR_CUDA"}
DEV_STATUS_BITS = {0x1: "producer wait timed out", 0x2: "MMA wait timed out", 0x4: "epilogue wait timed out"}

_lib = None


class VpError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {_STATUS.get(code, code)}")
        self.code = code


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvp.so")


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libvp.so is not built ({path}); run `python -m vocab_lm_head_vp_b300.build`")
    L = ctypes.CDLL(path)
    P, I64, I32, SZ, U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_int
    L.vp_status_string.restype = ctypes.c_char_p
    L.vp_status_string.argtypes = [I32]
    L.vp_version.restype = ctypes.c_char_p
    L.vp_embed_fwd.restype = I32
    L.vp_embed_fwd.argtypes = [P, P, P, I64, I64, I64, I32, I32, P]
    L.vp_embed_fwd_sp.restype = I32
    L.vp_embed_fwd_sp.argtypes = [P, P, P, I64, I64, I64, I32, I32, I32, P]
    L.vp_embed_bwd_workspace_size.restype = SZ
    L.vp_embed_bwd_workspace_size.argtypes = [I64, I64, I64, I32, I32]
    L.vp_embed_bwd.restype = I32
    L.vp_embed_bwd.argtypes = [P, P, P, I64, I64, I64, I32, I32, I32, P, SZ, P]
    L.vp_embed_bwd_plan.restype = I32
    L.vp_embed_bwd_plan.argtypes = [P, I64, I64, I64, I32, P, SZ, P]
    L.vp_embed_bwd_planned.restype = I32
    L.vp_embed_bwd_planned.argtypes = [P, P, I64, I64, I64, I32, I32, I32, P, SZ, P]
    L.vp_lmhead_ce_workspace_size.restype = SZ
    L.vp_lmhead_ce_workspace_size.argtypes = [I64, I64, I64, I32, I32, I32, I64]
    L.vp_lmhead_ce_fwd.restype = I32
    L.vp_lmhead_ce_fwd.argtypes = [P, P, P, I64, I64, I64, I32, I64, I32, P, P, P, P, P, P, SZ, P]
    L.vp_lmhead_ce_bwd.restype = I32
    L.vp_lmhead_ce_bwd.argtypes = [P, P, P, P, P, P, I64, I64, I64, I32, I64, I32, P, P, P, SZ, P]
    L.vp_lmhead_ce_fwd_bwd.restype = I32
    L.vp_lmhead_ce_fwd_bwd.argtypes = [P, P, P, P, P, I64, I64, I64, I32, I64, I32, P, P, P, P, P, P, P, P, SZ, P]
    L.vp_lmhead_ce_fwd_keep.restype = I32
    L.vp_lmhead_ce_fwd_keep.argtypes = [P, P, P, I64, I64, I64, I32, I64, I32, P, P, P, P, P, P, SZ, P]
    L.vp_lmhead_ce_bwd_saved.restype = I32
    L.vp_lmhead_ce_bwd_saved.argtypes = [P, P, P, P, P, P, I64, I64, I64, I32, I64, I32, P, P, P, SZ, P]
    L.vp_lmhead_ce_shard_fwd.restype = I32
    L.vp_lmhead_ce_shard_fwd.argtypes = [P, P, P, I64, I64, I64, I32, I32, I64, I32, P, P, SZ, P]
    L.vp_lmhead_ce_merge_stats.restype = I32
    L.vp_lmhead_ce_merge_stats.argtypes = [P, P, I64, I64, I32, I64, P, P, P, P, P]
    L.vp_lmhead_ce_shard_bwd.restype = I32
    L.vp_lmhead_ce_shard_bwd.argtypes = [P, P, P, P, P, P, I64, I64, I64, I32, I32, I64, I32, P, P, P, SZ, P]
    L.vp_read_device_status.restype = I32
    L.vp_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
    L.vp_test_gemm_bf16.restype = I32
    L.vp_test_gemm_bf16.argtypes = [P, P, P, I64, I64, I64, U, U, P, P]
    L.vp_test_set_gemm_variant.restype = I32
    L.vp_test_set_gemm_variant.argtypes = [I32]
    L.vp_test_dx_plan.restype = I32
    L.vp_test_dx_plan.argtypes = [I64, I64, I32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                  ctypes.POINTER(ctypes.c_double)]
    L.vp_test_set_wait_fault.restype = I32
    L.vp_test_set_wait_fault.argtypes = [I32, ctypes.c_uint64]
    L.vp_lmhead_ce_fwd_noalloc.restype = I32
    L.vp_lmhead_ce_fwd_noalloc.argtypes = [P, P, P, I64, I64, I64, I32, I64, I32, P, P, P, P, P, P]
    L.vp_stage_timing_enable.restype = I32
    L.vp_stage_timing_enable.argtypes = [I32]
    L.vp_stage_timing_read.restype = I32
    L.vp_stage_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int32), I32]
    L.vp_stage_timing_dropped.restype = I32
    L.vp_stage_timing_dropped.argtypes = []
    L.vp_stage_name.restype = ctypes.c_char_p
    L.vp_stage_name.argtypes = [I32]
    _lib = L
    return L


def _check(fn, code):
    if code != 0:
        raise VpError(fn, code)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return VP_BF16
    if t.dtype == torch.float32:
        return VP_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or f32)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def workspace_size(N, H, V, T, dtype, pass_, vocab_chunk=0) -> int:
    code = dtype if isinstance(dtype, int) else (VP_BF16 if dtype == torch.bfloat16 else VP_F32)
    return int(_load().vp_lmhead_ce_workspace_size(N, H, V, T, code, pass_, int(vocab_chunk or 0)))


def _workspace(nbytes, device, workspace):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def embed_fwd(ids: torch.Tensor, W: torch.Tensor, T: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """out[n] = W[ids[n]] (zero row for ids outside [0, V)), gathered shard-wise."""
    _need(W, "W")
    _need(ids, "ids", torch.int64, W.device)
    V, H = W.shape
    N = ids.numel()
    if out is None:
        out = torch.empty((N, H), dtype=W.dtype, device=W.device)
    _need(out, "out", W.dtype, W.device)
    _check("vp_embed_fwd", _load().vp_embed_fwd(_ptr(ids), _ptr(W), _ptr(out), N, H, V, T, _dtype_code(W),
                                                _stream(W.device)))
    return out


def embed_fwd_sp(ids: torch.Tensor, W: torch.Tensor, T: int, rank: int, out: torch.Tensor | None = None):
    """Sequence-parallel embedding: rank's token rows [rank N/T, (rank+1) N/T)
    of the shard sum (the reduce-scatter of the shard outputs)."""
    _need(W, "W")
    _need(ids, "ids", torch.int64, W.device)
    V, H = W.shape
    N = ids.numel()
    if out is None:
        out = torch.empty((N // T, H), dtype=W.dtype, device=W.device)
    _need(out, "out", W.dtype, W.device)
    _check("vp_embed_fwd_sp", _load().vp_embed_fwd_sp(_ptr(ids), _ptr(W), _ptr(out), N, H, V, T, rank,
                                                      _dtype_code(W), _stream(W.device)))
    return out


def embed_bwd(ids: torch.Tensor, dOut: torch.Tensor, V: int, T: int, dW: torch.Tensor | None = None,
              accumulate: bool = False, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """dW[v] (+)= sum of dOut[n] over tokens with ids[n] = v (fp32 [V,H]);
    with accumulate=True it adds onto dW (the tied weight's LM-head gradient)."""
    _need(dOut, "dOut")
    _need(ids, "ids", torch.int64, dOut.device)
    N, H = dOut.shape
    dev = dOut.device
    if dW is None:
        if accumulate:
            raise ValueError("accumulate=True needs dW")
        dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    _need(dW, "dW", torch.float32, dev)
    L = _load()
    nb = int(L.vp_embed_bwd_workspace_size(N, H, V, T, _dtype_code(dOut)))
    if nb == 0:
        raise VpError("vp_embed_bwd_workspace_size", 1)
    ws = _workspace(nb, dev, workspace)
    _check("vp_embed_bwd", L.vp_embed_bwd(_ptr(ids), _ptr(dOut), _ptr(dW), N, H, V, T, _dtype_code(dOut),
                                          int(bool(accumulate)), _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(dev)))
    return dW


def embed_bwd_plan(ids: torch.Tensor, H: int, V: int, T: int, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """The id-only step of embed_bwd (the tokens grouped by id) into a
    workspace, for embed_bwd_planned later; returns the workspace."""
    _need(ids, "ids", torch.int64)
    N = ids.numel()
    L = _load()
    nb = int(L.vp_embed_bwd_workspace_size(N, H, V, T, VP_BF16))
    if nb == 0:
        raise VpError("vp_embed_bwd_workspace_size", 1)
    ws = _workspace(nb, ids.device, workspace)
    _check("vp_embed_bwd_plan", L.vp_embed_bwd_plan(_ptr(ids), N, H, V, T, _ptr(ws), ws.numel() * ws.element_size(),
                                                    _stream(ids.device)))
    return ws


def embed_bwd_planned(plan: torch.Tensor, dOut: torch.Tensor, V: int, T: int, dW: torch.Tensor | None = None,
                      accumulate: bool = False) -> torch.Tensor:
    """The sums of embed_bwd over a workspace that embed_bwd_plan prepared."""
    _need(dOut, "dOut")
    N, H = dOut.shape
    dev = dOut.device
    if dW is None:
        if accumulate:
            raise ValueError("accumulate=True needs dW")
        dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    _need(dW, "dW", torch.float32, dev)
    _check("vp_embed_bwd_planned", _load().vp_embed_bwd_planned(
        _ptr(dOut), _ptr(dW), N, H, V, T, _dtype_code(dOut), int(bool(accumulate)), _ptr(plan),
        plan.numel() * plan.element_size(), _stream(dev)))
    return dW


def lmhead_ce_fwd(X, W, targets, T, ignore_index=IGNORE_INDEX, shard_stats=False, workspace=None,
                  out=None, keep=False) -> dict:
    """Fused LM head + vocab-parallel CE forward.  Returns loss [N], lse [N],
    mean [1], n_bad [1] (int32) and, if asked, shard_stats [T,3,N].  With
    keep=True the tile probabilities stay in out["saved"] (about 2*N*V bytes)
    for lmhead_ce_bwd(..., saved=out["saved"]), which then skips the logit
    recompute."""
    _need(X, "X")
    _need(W, "W", X.dtype, X.device)
    _need(targets, "targets", torch.int64, X.device)
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if out is None:
        out = {"loss": torch.empty(N, dtype=torch.float32, device=dev),
               "lse": torch.empty(N, dtype=torch.float32, device=dev),
               "mean": torch.empty(1, dtype=torch.float32, device=dev),
               "n_bad": torch.empty(1, dtype=torch.int32, device=dev)}
        if shard_stats:
            out["shard_stats"] = torch.empty((T, 3, N), dtype=torch.float32, device=dev)
    ws_bytes = workspace_size(N, H, V, T, _dtype_code(X), 3 if keep else 0)
    if ws_bytes == 0:
        raise VpError("vp_lmhead_ce_workspace_size", 1)
    ws = _workspace(ws_bytes, dev, workspace)
    fn = _load().vp_lmhead_ce_fwd_keep if keep else _load().vp_lmhead_ce_fwd
    code = fn(
        _ptr(X), _ptr(W), _ptr(targets), N, H, V, T, ignore_index, _dtype_code(X), _ptr(out["loss"]),
        _ptr(out["lse"]), _ptr(out.get("mean")), _ptr(out.get("shard_stats")), _ptr(out.get("n_bad")),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(dev))
    _check("vp_lmhead_ce_fwd_keep" if keep else "vp_lmhead_ce_fwd", code)
    out["workspace"] = ws
    if keep:
        out["saved"] = ws
    return out


def lmhead_ce_bwd(X, W, targets, lse, T, ignore_index=IGNORE_INDEX, dloss=None, vocab_chunk=None,
                  workspace=None, dX=None, dW=None, dmean=None, saved=None):
    """Backward of dmean * loss_mean (dmean: a 1-element device tensor, default
    1) or of sum_n dloss[n] * loss[n]: (dX in X's dtype, dW in fp32).  With
    `saved` (from lmhead_ce_fwd(..., keep=True)) it uses the kept tile
    probabilities instead of recomputing the logits; the buffer is consumed."""
    _need(X, "X")
    _need(W, "W", X.dtype, X.device)
    _need(targets, "targets", torch.int64, X.device)
    _need(lse, "lse", torch.float32, X.device)
    if dloss is not None:
        _need(dloss, "dloss", torch.float32, X.device)
    if dmean is not None:
        _need(dmean, "dmean", torch.float32, X.device)
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if dX is None:
        dX = torch.empty_like(X)
    if dW is None:
        dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    _need(dX, "dX", X.dtype, dev)
    _need(dW, "dW", torch.float32, dev)
    if saved is not None:
        _check("vp_lmhead_ce_bwd_saved", _load().vp_lmhead_ce_bwd_saved(
            _ptr(X), _ptr(W), _ptr(targets), _ptr(lse), _ptr(dloss), _ptr(dmean), N, H, V, T, ignore_index,
            _dtype_code(X), _ptr(dX), _ptr(dW), _ptr(saved), saved.numel() * saved.element_size(), _stream(dev)))
        return dX, dW
    ws_bytes = workspace_size(N, H, V, T, _dtype_code(X), 1, vocab_chunk or 0)
    if ws_bytes == 0:
        raise VpError("vp_lmhead_ce_workspace_size", 1)
    ws = _workspace(ws_bytes, dev, workspace)
    code = _load().vp_lmhead_ce_bwd(
        _ptr(X), _ptr(W), _ptr(targets), _ptr(lse), _ptr(dloss), _ptr(dmean), N, H, V, T, ignore_index,
        _dtype_code(X),
        _ptr(dX), _ptr(dW), _ptr(ws), ws_bytes if workspace is None else ws.numel() * ws.element_size(),
        _stream(dev))
    _check("vp_lmhead_ce_bwd", code)
    return dX, dW


def lmhead_ce_fwd_bwd(X, W, targets, T, ignore_index=IGNORE_INDEX, dloss=None, shard_stats=False, token_chunk=None,
                      workspace=None, out=None, dmean=None) -> dict:
    """Forward and backward in one call (probabilities saved, no logit
    recompute).  Returns the forward's loss, lse, mean, n_bad (and
    shard_stats if asked) plus dX (X's dtype) and dW (fp32) of the mean loss,
    or of sum_n dloss[n] * loss[n] when dloss is given."""
    _need(X, "X")
    _need(W, "W", X.dtype, X.device)
    _need(targets, "targets", torch.int64, X.device)
    if dloss is not None:
        _need(dloss, "dloss", torch.float32, X.device)
    if dmean is not None:
        _need(dmean, "dmean", torch.float32, X.device)
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if out is None:
        out = {"loss": torch.empty(N, dtype=torch.float32, device=dev),
               "lse": torch.empty(N, dtype=torch.float32, device=dev),
               "mean": torch.empty(1, dtype=torch.float32, device=dev),
               "n_bad": torch.empty(1, dtype=torch.int32, device=dev),
               "dX": torch.empty_like(X),
               "dW": torch.empty((V, H), dtype=torch.float32, device=dev)}
        if shard_stats:
            out["shard_stats"] = torch.empty((T, 3, N), dtype=torch.float32, device=dev)
    _need(out["dX"], "dX", X.dtype, dev)
    _need(out["dW"], "dW", torch.float32, dev)
    if workspace is None:
        ws_bytes = workspace_size(N, H, V, T, _dtype_code(X), 2, token_chunk or 0)
        if ws_bytes == 0:
            raise VpError("vp_lmhead_ce_workspace_size", 1)
        ws = _workspace(ws_bytes, dev, None)
    else:
        # the library picks the largest token chunk the given bytes hold (VP_ERR_WORKSPACE if none)
        ws = workspace
        ws_bytes = ws.numel() * ws.element_size()
    code = _load().vp_lmhead_ce_fwd_bwd(
        _ptr(X), _ptr(W), _ptr(targets), _ptr(dloss), _ptr(dmean), N, H, V, T, ignore_index, _dtype_code(X),
        _ptr(out["loss"]),
        _ptr(out["lse"]), _ptr(out.get("mean")), _ptr(out.get("shard_stats")), _ptr(out.get("n_bad")),
        _ptr(out["dX"]), _ptr(out["dW"]), _ptr(ws), ws_bytes, _stream(dev))
    _check("vp_lmhead_ce_fwd_bwd", code)
    out["workspace"] = ws
    return out


def lmhead_ce_shard_fwd(X, W_t, targets, V, T, t, ignore_index=IGNORE_INDEX, workspace=None, stats=None):
    """Shard t's statistics [3, N] = (m_t, R_t = S_t - 1, z_y^(t)) from its own
    rows W_t = W[t V/T, (t+1) V/T) (the rank of a T-rank vocabulary)."""
    _need(X, "X")
    _need(W_t, "W_t", X.dtype, X.device)
    _need(targets, "targets", torch.int64, X.device)
    N, H = X.shape
    dev = X.device
    if stats is None:
        stats = torch.empty((3, N), dtype=torch.float32, device=dev)
    _need(stats, "stats", torch.float32, dev)
    nb = workspace_size(N, H, V // T, 1, _dtype_code(X), 0)
    if nb == 0:
        raise VpError("vp_lmhead_ce_workspace_size", 1)
    ws = _workspace(nb, dev, workspace)
    _check("vp_lmhead_ce_shard_fwd", _load().vp_lmhead_ce_shard_fwd(
        _ptr(X), _ptr(W_t), _ptr(targets), N, H, V, T, t, ignore_index, _dtype_code(X), _ptr(stats), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(dev)))
    return stats


def lmhead_ce_merge_stats(stats, targets, V, T, ignore_index=IGNORE_INDEX, out=None) -> dict:
    """Merge of the T shards' gathered statistics [T, 3, N] into loss, lse,
    mean and n_bad (the result vp_lmhead_ce_fwd gives for the whole W)."""
    _need(stats, "stats", torch.float32)
    _need(targets, "targets", torch.int64, stats.device)
    N = targets.numel()
    if tuple(stats.shape) != (T, 3, N):
        raise ValueError(f"stats must be [T, 3, N] = [{T}, 3, {N}], got {tuple(stats.shape)}")
    dev = stats.device
    if out is None:
        out = {"loss": torch.empty(N, dtype=torch.float32, device=dev),
               "lse": torch.empty(N, dtype=torch.float32, device=dev),
               "mean": torch.empty(1, dtype=torch.float32, device=dev),
               "n_bad": torch.empty(1, dtype=torch.int32, device=dev)}
    _check("vp_lmhead_ce_merge_stats", _load().vp_lmhead_ce_merge_stats(
        _ptr(stats), _ptr(targets), N, V, T, ignore_index, _ptr(out["loss"]), _ptr(out["lse"]), _ptr(out.get("mean")),
        _ptr(out.get("n_bad")), _stream(dev)))
    return out


def lmhead_ce_shard_bwd(X, W_t, targets, lse, V, T, t, ignore_index=IGNORE_INDEX, dloss=None, dmean=None,
                        vocab_chunk=None, workspace=None, dX_t=None, dW_t=None):
    """Shard t's backward: (dX_t, dW_t), both fp32.  dX_t is this shard's part of
    dX (sum it over the T shards); dW_t is complete for the shard's rows."""
    _need(X, "X")
    _need(W_t, "W_t", X.dtype, X.device)
    _need(targets, "targets", torch.int64, X.device)
    _need(lse, "lse", torch.float32, X.device)
    N, H = X.shape
    Vt = W_t.shape[0]
    dev = X.device
    if dX_t is None:
        dX_t = torch.empty((N, H), dtype=torch.float32, device=dev)
    if dW_t is None:
        dW_t = torch.empty((Vt, H), dtype=torch.float32, device=dev)
    _need(dX_t, "dX_t", torch.float32, dev)
    _need(dW_t, "dW_t", torch.float32, dev)
    nb = workspace_size(N, H, V // T, 1, _dtype_code(X), 1, vocab_chunk or 0)
    if nb == 0:
        raise VpError("vp_lmhead_ce_workspace_size", 1)
    ws = _workspace(nb, dev, workspace)
    _check("vp_lmhead_ce_shard_bwd", _load().vp_lmhead_ce_shard_bwd(
        _ptr(X), _ptr(W_t), _ptr(targets), _ptr(lse), _ptr(dloss), _ptr(dmean), N, H, V, T, t, ignore_index,
        _dtype_code(X), _ptr(dX_t), _ptr(dW_t), _ptr(ws), ws.numel() * ws.element_size(), _stream(dev)))
    return dX_t, dW_t


def vocab_parallel_lmhead_ce(X, W_t, targets, V, T, rank, group=None, ignore_index=IGNORE_INDEX, dmean=None):
    """One rank's step of the T-rank form ("Vocab Parallelism" sec. 5.3; the
    interview note's figure 2): the shard's statistics, one all-gather of them
    ([T, 3, N], rank order), the merge (every rank gets the same loss and lse),
    the shard's backward, and an all-reduce (SUM) of the fp32 dX parts.
    Returns (forward dict, dX fp32 [N, H], dW_t fp32 [V/T, H]).  The two
    collectives go through torch.distributed on `group`; everything else is
    libvp's kernels on this rank's device."""
    import torch.distributed as dist
    stats = lmhead_ce_shard_fwd(X, W_t, targets, V, T, rank, ignore_index)
    parts = [torch.empty_like(stats) for _ in range(T)]
    dist.all_gather(parts, stats, group=group)
    fwd = lmhead_ce_merge_stats(torch.stack(parts), targets, V, T, ignore_index)
    dX, dW_t = lmhead_ce_shard_bwd(X, W_t, targets, fwd["lse"], V, T, rank, ignore_index, dmean=dmean)
    dist.all_reduce(dX, group=group)
    return fwd, dX, dW_t


def read_device_status(workspace: torch.Tensor) -> int:
    """Synchronise the current stream and return the workspace's device status
    word (0 = no kernel gave up waiting)."""
    flags = ctypes.c_uint32(0)
    _check("vp_read_device_status", _load().vp_read_device_status(_ptr(workspace), ctypes.byref(flags),
                                                                  _stream(workspace.device)))
    return int(flags.value)


def test_gemm_bf16(A, B, a_mn_major=False, b_mn_major=False):
    """D = A * B^T (fp32) through the tcgen05 GEMM core.  A is [M,K] (or [K,M]
    when a_mn_major), B is [N,K] (or [K,N] when b_mn_major)."""
    _need(A, "A", torch.bfloat16)
    _need(B, "B", torch.bfloat16, A.device)
    M = A.shape[1] if a_mn_major else A.shape[0]
    K = A.shape[0] if a_mn_major else A.shape[1]
    N = B.shape[1] if b_mn_major else B.shape[0]
    D = torch.empty((M, N), dtype=torch.float32, device=A.device)
    ws = torch.zeros(256, dtype=torch.uint8, device=A.device)
    _check("vp_test_gemm_bf16", _load().vp_test_gemm_bf16(_ptr(A), _ptr(B), _ptr(D), M, N, K, int(a_mn_major),
                                                          int(b_mn_major), _ptr(ws), _stream(A.device)))
    return D, ws


def set_gemm_variant(variant) -> None:
    """tcgen05 GEMM form: 0 / False (default) one SM per logits and dX tile
    (dX tiles chosen per launch), dW^T on SM pairs; 1 / True SM pairs
    everywhere; 2 one SM per 128 x 256 tile everywhere, dW in the direct form;
    3 as 0 with the logits GEMMs in clusters that share W by TMA multicast."""
    _check("vp_test_set_gemm_variant", _load().vp_test_set_gemm_variant(int(variant)))


def dx_plan(rows: int, H: int, sms: int) -> dict:
    """How a bf16 dX GEMM over `rows` token rows and H columns would run on
    `sms` persistent CTAs (host arithmetic, no launch): tile rows (256 or
    128), whether stream-K, and the wave cost the choice is made by."""
    r, sk, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
    _check("vp_test_dx_plan", _load().vp_test_dx_plan(int(rows), int(H), int(sms), ctypes.byref(r),
                                                      ctypes.byref(sk), ctypes.byref(c)))
    return {"tile_rows": r.value, "streamk": bool(sk.value), "cost": c.value}


def set_wait_fault(mode: int, wait_ns: int = 0) -> None:
    """Diagnostic of the bounded waits in the tcgen05 GEMMs: mode 1 holds the
    TMA producer back, mode 2 the MMA issuer, 0 restores normal operation;
    wait_ns limits every wait (0: the default 1 s)."""
    _check("vp_test_set_wait_fault", _load().vp_test_set_wait_fault(int(mode), int(wait_ns)))


def stage_timing_enable(max_launches: int) -> None:
    """Record CUDA events around every kernel libvp launches (0 = stop)."""
    _check("vp_stage_timing_enable", _load().vp_stage_timing_enable(int(max_launches)))


def stage_timing_read() -> dict:
    """{stage name: (milliseconds, launches)} accumulated since enabling.

    Raises if some timed regions found every slot in use: the totals would be
    partial.
    """
    L = _load()
    dropped = L.vp_stage_timing_dropped()
    if dropped:
        raise RuntimeError(f"stage timing: {dropped} timed regions were not recorded (enable more slots)")
    n = 16
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    k = L.vp_stage_timing_read(ms, cnt, n)
    if k < 0:
        raise VpError("vp_stage_timing_read", 4)
    return {L.vp_stage_name(i).decode(): (float(ms[i]), int(cnt[i])) for i in range(k)}


class _LMHeadCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, W, targets, T, ignore_index, save_probs):
        out = lmhead_ce_fwd(X, W, targets, T, ignore_index, keep=save_probs)
        ctx.save_for_backward(X, W, targets, out["lse"])
        ctx.T, ctx.ignore_index = T, ignore_index
        ctx.saved_probs = out.get("saved")
        return out["mean"][0]

    @staticmethod
    def backward(ctx, grad):
        X, W, targets, lse = ctx.saved_tensors
        # the incoming gradient of the mean goes to the library as a device scalar
        dmean = grad.reshape(1)
        if dmean.dtype != torch.float32 or not dmean.is_contiguous():
            dmean = dmean.to(torch.float32).contiguous()
        dX, dW = lmhead_ce_bwd(X, W, targets, lse, ctx.T, ctx.ignore_index, dmean=dmean, saved=ctx.saved_probs)
        ctx.saved_probs = None
        return dX, dW.to(W.dtype), None, None, None, None


def lmhead_ce(X, W, targets, T, ignore_index=IGNORE_INDEX, save_probs=False):
    """Mean cross-entropy of the tied LM head over valid tokens, differentiable
    in X and W (autograd wrapper of lmhead_ce_fwd / lmhead_ce_bwd).
    save_probs=True keeps the tile probabilities (about 2*N*V bytes) from the
    forward to the backward, which then skips the logit recompute (6NHV flops
    instead of 8NHV); the default keeps only lse."""
    return _LMHeadCE.apply(X, W, targets, T, ignore_index, bool(save_probs))
