"""Float64 CPU oracle for vocab-parallel cross-entropy over a tied, vocab-sharded LM head.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) import this
module.  The product package ``vocab_lm_head_vp_b300`` never imports, links or
calls it, and shares no code with it: the CUDA path must stand on its own.

Everything here is the plain definition, written out in float64 NumPy, with no
blocking or fusion beyond what the definition states.  bf16 inputs enter as the
exact float64 values of their bf16 bit patterns.

Sources (page title, section):
  [VP-book]  MiniMind-tron book, ch. 5 "Vocab Parallelism":
             sec. 5.2.1 Vocab Parallel Embedding (shard ranges, masked lookup,
             the V=8 worked table), sec. 5.2.2 (embedding and LM head tied to
             one parameter), sec. 5.3.1 forward (max-shifted CE, the three
             [B,S] statistics), sec. 5.3.2 backward (p - onehot, local),
             sec. 5.3.3 ignore_index (mean over valid tokens).
  [VP-note]  "Vocab parallelism: how to split embedding and LM head" (interview
             note): figure 1 (id 5 on V=8, t=2), figure 2 (three all-reduces),
             key formulas (l = log sum e^(z-m) - (z_y - m), m = max_r m_r, ...,
             backward p - 1[j=y], LM-head dX all-reduced), NumPy t=4 simulation.
  [TP-gloss] LLM glossary "Tensor Parallelism": column-parallel linear
             Y^(r) = X W^(r) and its input-gradient partial sums.

Readings where the pages are silent (each also listed in the design notes):
  * a target outside [0, V) that is not ignore_index counts as ignored and is
    reported in ``n_bad`` (the pages' mask would silently give z_y = 0);
  * with every target ignored the mean is 0 / max(1, 0) = 0;
  * an embedding id outside [0, V) is masked by every shard, so its row is zero;
  * the embedding shard sum runs over t = 0..T-1 starting from +0.0, so a -0.0
    weight comes out as +0.0.

Parity: every public function is pinned by tests/test_oracle_pins.py (worked
examples from the pages, closed forms, invariants, a library routine, finite
differences); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


# --------------------------------------------------------------------------
# Shards  ([VP-book] sec. 5.1 "V % T == 0", sec. 5.2.1 rank t owns [tV/T,(t+1)V/T))
# --------------------------------------------------------------------------
def shard_bounds(V: int, T: int) -> list[tuple[int, int]]:
    """Vocab range [tV/T, (t+1)V/T) of each of the T shards; V % T must be 0."""
    if T <= 0 or V <= 0 or V % T != 0:
        raise ValueError(f"vocab-parallel split needs V % T == 0 (V={V}, T={T})")
    vs = V // T
    return [(t * vs, (t + 1) * vs) for t in range(T)]


# --------------------------------------------------------------------------
# Embedding  ([VP-book] sec. 5.2.1; [VP-note] figure 1)
# --------------------------------------------------------------------------
def embed_shard_partial(ids: np.ndarray, W: np.ndarray, V: int, T: int, t: int) -> np.ndarray:
    """Shard t's masked local lookup: ids outside [start, end) look up local
    row 0 and their output row is then set to zero."""
    start, end = shard_bounds(V, T)[t]
    ids = np.asarray(ids, dtype=np.int64)
    W_t = np.asarray(W, dtype=np.float64)[start:end]
    mask = (ids < start) | (ids >= end)
    local = ids - start
    local[mask] = 0
    out = W_t[local].copy()
    out[mask] = 0.0
    return out


def embed(ids: np.ndarray, W: np.ndarray, V: int, T: int) -> np.ndarray:
    """Sum of the T shard partials (the all-reduce of sec. 5.2.1), taken in
    order t = 0..T-1 from +0.0."""
    ids = np.asarray(ids, dtype=np.int64)
    acc = np.zeros((ids.shape[0], np.asarray(W).shape[1]), dtype=np.float64)
    for t in range(T):
        acc = acc + embed_shard_partial(ids, W, V, T, t)
    return acc


def embed_sp(ids: np.ndarray, W: np.ndarray, V: int, T: int, rank: int) -> np.ndarray:
    """Sequence parallelism on ([VP-book] sec. 5.2.1): the T shard partials are
    reduce-scattered along the token dimension, so rank r keeps token rows
    [r N/T, (r+1) N/T) of their sum (taken in order t = 0..T-1 from +0.0).
    N % T must be 0."""
    ids = np.asarray(ids, dtype=np.int64)
    N = ids.shape[0]
    if N % T != 0 or not 0 <= rank < T:
        raise ValueError(f"reduce-scatter over T={T} ranks needs N % T == 0 and 0 <= rank < T (N={N})")
    total = np.zeros((N, np.asarray(W).shape[1]), dtype=np.float64)
    for t in range(T):
        total = total + embed_shard_partial(ids, W, V, T, t)
    rows = N // T
    return total[rank * rows:(rank + 1) * rows]


# --------------------------------------------------------------------------
# Embedding backward  ([VP-book] sec. 5.2.1 masked lookup; sec. 5.2.2 the
# embedding and the LM head share one [V,H] parameter, so its gradient is the
# sum of both layers' gradients)
# --------------------------------------------------------------------------
def embed_shard_grad(ids: np.ndarray, dOut: np.ndarray, V: int, T: int, t: int) -> np.ndarray:
    """Gradient of shard t's masked local lookup with respect to its slice W_t,
    taking the lookup's steps backwards: the zeroing of masked output rows
    passes them no gradient, and the gather of local rows adds each remaining
    token's upstream row into local row id - start (token order)."""
    start, end = shard_bounds(V, T)[t]
    ids = np.asarray(ids, dtype=np.int64)
    g = np.array(dOut, dtype=np.float64)
    mask = (ids < start) | (ids >= end)
    local = ids - start
    local[mask] = 0
    g[mask] = 0.0                                   # backward of "output[mask] = 0"
    dW_t = np.zeros((end - start, g.shape[1]), dtype=np.float64)
    np.add.at(dW_t, local, g)                       # backward of "W_t[local]"
    return dW_t


def embed_backward(ids: np.ndarray, dOut: np.ndarray, V: int, T: int, dW0=None) -> np.ndarray:
    """Gradient of the summed shard outputs with respect to the tied weight
    W [V,H].  The forward's sum over shards hands every shard the same upstream
    rows dOut, so shard t's slice gradient fills rows [tV/T, (t+1)V/T).  With
    dW0 (the tied weight's other gradient, the LM head's) the two are added."""
    H = np.asarray(dOut).shape[1]
    dW = np.zeros((V, H), dtype=np.float64) if dW0 is None else np.array(dW0, dtype=np.float64)
    for t, (start, end) in enumerate(shard_bounds(V, T)):
        dW[start:end] += embed_shard_grad(ids, dOut, V, T, t)
    return dW


# --------------------------------------------------------------------------
# LM head logits  ([VP-book] sec. 5.2.2; [TP-gloss] column parallel)
# --------------------------------------------------------------------------
def logits(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Z = X W^T in float64 (the dense logits the method never materialises)."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def target_masks(y: np.ndarray, V: int, ignore_index: int = IGNORE_INDEX):
    """(valid, bad): valid = target in [0, V) and not ignore_index (an
    ignore_index inside [0, V) still marks the position as ignored);
    bad = out of range and not ignore_index."""
    y = np.asarray(y, dtype=np.int64)
    in_range = (y >= 0) & (y < V)
    return in_range & (y != ignore_index), (~in_range) & (y != ignore_index)


# --------------------------------------------------------------------------
# Dense cross-entropy  ([VP-book] sec. 5.3.1 CE(x,k) = -x_k + m + log sum e^(x_i - m);
# [VP-note] key formulas; [VP-book] sec. 5.3.3 L = sum_valid l / max(1, N_valid))
# --------------------------------------------------------------------------
def cross_entropy(Z: np.ndarray, y: np.ndarray, ignore_index: int = IGNORE_INDEX) -> dict:
    """Per-token loss, log-sum-exp, mean over valid tokens, and counts."""
    Z = np.asarray(Z, dtype=np.float64)
    n, V = Z.shape
    valid, bad = target_masks(y, V, ignore_index)
    m = Z.max(axis=1)
    s = np.exp(Z - m[:, None]).sum(axis=1)
    lse = m + np.log(s)
    z_y = Z[np.arange(n), np.where(valid, y, 0)]
    loss = np.where(valid, -z_y + m + np.log(s), 0.0)
    n_valid = int(valid.sum())
    return {"loss": loss, "lse": lse, "mean": float(loss.sum()) / max(1, n_valid),
            "n_valid": n_valid, "n_bad": int(bad.sum()), "z_y": np.where(valid, z_y, 0.0)}


# --------------------------------------------------------------------------
# Sharded forms ([VP-book] sec. 5.3.1; [VP-note] figure 2 and key formulas)
# --------------------------------------------------------------------------
def cross_entropy_three_reductions(Z: np.ndarray, y: np.ndarray, V: int, T: int,
                                   ignore_index: int = IGNORE_INDEX) -> dict:
    """The pages' T-rank formulation, ranks simulated in one process: local max
    then MAX over ranks; local sum of exp(z - m) with the global m, then SUM;
    local target logit (0 off-shard), then SUM."""
    Z = np.asarray(Z, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    n = Z.shape[0]
    bounds = shard_bounds(V, T)
    shards = [Z[:, a:b] for a, b in bounds]
    m = shards[0].max(axis=1)
    for zt in shards[1:]:
        m = np.maximum(m, zt.max(axis=1))
    s = np.zeros(n)
    for zt in shards:
        s = s + np.exp(zt - m[:, None]).sum(axis=1)
    z_y = np.zeros(n)
    for (a, b), zt in zip(bounds, shards):
        own = (y >= a) & (y < b)
        local = np.where(own, y - a, 0)
        z_y = z_y + np.where(own, zt[np.arange(n), local], 0.0)
    valid, bad = target_masks(y, V, ignore_index)
    loss = np.where(valid, np.log(s) - (z_y - m), 0.0)
    n_valid = int(valid.sum())
    return {"loss": loss, "lse": m + np.log(s), "mean": float(loss.sum()) / max(1, n_valid),
            "n_valid": n_valid, "n_bad": int(bad.sum())}


def shard_local_stats(Z: np.ndarray, y: np.ndarray, V: int, T: int,
                      ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """Per shard t and token n the triple (m_t, S_t, z_y^(t)): local max, sum of
    exp(z - m_t) over the shard, and the target logit if the (non-ignored)
    target is in the shard, else 0.  Returns an array [T, 3, N]."""
    Z = np.asarray(Z, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    n = Z.shape[0]
    out = np.zeros((T, 3, n))
    for t, (a, b) in enumerate(shard_bounds(V, T)):
        zt = Z[:, a:b]
        mt = zt.max(axis=1)
        out[t, 0] = mt
        out[t, 1] = np.exp(zt - mt[:, None]).sum(axis=1)
        own = (y >= a) & (y < b) & (y != ignore_index)
        out[t, 2] = np.where(own, zt[np.arange(n), np.where(own, y - a, 0)], 0.0)
    return out


def merge_local_stats(stats: np.ndarray) -> dict:
    """Merge of the per-shard triples: m = max_t m_t, S = sum_t S_t e^(m_t - m),
    z_y = sum_t z_y^(t); lse = m + log S."""
    m_t, s_t, zy_t = stats[:, 0], stats[:, 1], stats[:, 2]
    m = m_t.max(axis=0)
    s = (s_t * np.exp(m_t - m[None, :])).sum(axis=0)
    return {"lse": m + np.log(s), "z_y": zy_t.sum(axis=0), "m": m, "S": s}


# --------------------------------------------------------------------------
# Backward ([VP-book] sec. 5.3.2 dCE/dx_j = p_j - 1[j=k]; sec. 5.3.3 ignored
# positions get zero gradient; [VP-note] key formulas)
# --------------------------------------------------------------------------
def upstream_scale(y: np.ndarray, V: int, ignore_index: int = IGNORE_INDEX,
                   dloss: np.ndarray | None = None) -> np.ndarray:
    """g_n: d(mean loss)/d(l_n) = 1/max(1, N_valid) for valid n, else 0; a given
    per-token upstream gradient replaces it on valid n."""
    valid, _ = target_masks(y, V, ignore_index)
    if dloss is None:
        return valid / max(1, int(valid.sum()))
    return np.where(valid, np.asarray(dloss, dtype=np.float64), 0.0)


def grad_logits(Z: np.ndarray, y: np.ndarray, lse: np.ndarray, g: np.ndarray) -> np.ndarray:
    """dZ[n, j] = g_n (softmax_j(Z_n) - 1[j = y_n]); rows with g_n = 0 are zero."""
    Z = np.asarray(Z, dtype=np.float64)
    n, V = Z.shape
    p = np.exp(Z - np.asarray(lse, dtype=np.float64)[:, None])
    onehot = np.zeros_like(p)
    in_range = (np.asarray(y) >= 0) & (np.asarray(y) < V)
    rows = np.nonzero(in_range)[0]
    onehot[rows, np.asarray(y)[rows]] = 1.0
    # ignored rows carry g_n = 0, so their onehot term vanishes with them
    return np.asarray(g, dtype=np.float64)[:, None] * (p - onehot)


def lmhead_grads(X: np.ndarray, W: np.ndarray, dZ: np.ndarray):
    """Gradients of Z = X W^T: dX = dZ W (the column-parallel input gradient,
    summed over shards) and dW = dZ^T X."""
    dZ = np.asarray(dZ, dtype=np.float64)
    return dZ @ np.asarray(W, dtype=np.float64), dZ.T @ np.asarray(X, dtype=np.float64)


# --------------------------------------------------------------------------
# Whole path
# --------------------------------------------------------------------------
def lmhead_ce_forward(X, W, y, V: int, T: int, ignore_index: int = IGNORE_INDEX) -> dict:
    """Forward of the tied LM head + vocab-parallel CE: dense definition plus the
    per-shard triples (for checking the shard statistics output)."""
    Z = logits(X, W)
    out = cross_entropy(Z, y, ignore_index)
    out["shard_stats"] = shard_local_stats(Z, y, V, T, ignore_index)
    return out


def lmhead_ce_backward(X, W, y, V: int, ignore_index: int = IGNORE_INDEX,
                       dloss=None) -> dict:
    """dX, dW (and dZ) of the mean loss (or of sum_n dloss_n l_n)."""
    Z = logits(X, W)
    lse = cross_entropy(Z, y, ignore_index)["lse"]
    g = upstream_scale(y, V, ignore_index, dloss)
    dZ = grad_logits(Z, y, lse, g)
    dX, dW = lmhead_grads(X, W, dZ)
    return {"dX": dX, "dW": dW, "dZ": dZ, "lse": lse, "g": g}


def lmhead_ce_rows(X, W, y, rows, n_valid: int, ignore_index: int = IGNORE_INDEX,
                   w_chunk: int = 16384, with_dx: bool = True) -> dict:
    """Loss, lse and dX for selected token rows only, one row's logits at a time
    over vocab chunks (for workloads too large for the dense form).  ``n_valid``
    is the number of valid targets in the whole batch (it sets g = 1/n_valid).
    W may be float32 holding bf16 values; chunks are widened to float64.
    with_dx=False skips dX (the rows' loss and lse only)."""
    W = np.asarray(W)
    V, H = W.shape
    rows = np.asarray(rows, dtype=np.int64)
    Xr = np.asarray(X, dtype=np.float64)[rows]
    yr = np.asarray(y, dtype=np.int64)[rows]
    Zr = np.empty((len(rows), V))
    for a in range(0, V, w_chunk):
        Zr[:, a:a + w_chunk] = Xr @ np.asarray(W[a:a + w_chunk], dtype=np.float64).T
    ce = cross_entropy(Zr, yr, ignore_index)
    if not with_dx:
        return {"loss": ce["loss"], "lse": ce["lse"], "z_y": ce["z_y"]}
    valid, _ = target_masks(yr, V, ignore_index)
    g = valid / max(1, n_valid)
    dZ = grad_logits(Zr, yr, ce["lse"], g)
    dX = np.zeros((len(rows), H))
    for a in range(0, V, w_chunk):
        dX += dZ[:, a:a + w_chunk] @ np.asarray(W[a:a + w_chunk], dtype=np.float64)
    return {"loss": ce["loss"], "lse": ce["lse"], "dX": dX, "z_y": ce["z_y"], "dZ": dZ, "g": g}


def lmhead_ce_dw_rows(X, W, y, lse, vocab_rows, n_valid: int, ignore_index: int = IGNORE_INDEX,
                      return_dz: bool = False):
    """dW rows for selected vocab ids only ([VP-book] sec. 5.3.2): the logit
    gradient's columns dZ[:, v] = g (exp(Z[:, v] - lse) - 1[y = v]) for those
    ids, then dW[v, :] = sum_n dZ[n, v] X[n, :].  ``lse`` is every token's
    log-sum-exp, from this oracle (lmhead_ce_rows over all rows); ``n_valid``
    sets g = 1/n_valid on valid targets, 0 elsewhere.  return_dz=True returns
    (dW rows, those dZ columns [N, len(vocab_rows)], g) instead of dW rows."""
    W = np.asarray(W)
    V = W.shape[0]
    vr = np.asarray(vocab_rows, dtype=np.int64)
    X64 = np.asarray(X, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    Zv = X64 @ np.asarray(W[vr], dtype=np.float64).T                  # [N, len(vr)]
    valid, _ = target_masks(y, V, ignore_index)
    g = valid / max(1, n_valid)
    onehot = (y[:, None] == vr[None, :]) & valid[:, None]
    dZv = g[:, None] * (np.exp(Zv - np.asarray(lse, dtype=np.float64)[:, None]) - onehot)
    dW_rows = dZv.T @ X64
    return (dW_rows, dZv, g) if return_dz else dW_rows
