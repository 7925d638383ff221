"""Each pin set must catch a plausible mistake planted in the oracle: a dropped
term, a wrong sign, a transposed operand, an off-by-one shard edge, a wrong
normaliser.  Mistakes are planted in the oracle module (on the CPU) and undone
by monkeypatch after each test."""
import numpy as np
import pytest

import oracle.ref as ref
import pins


def _fails_some_pin():
    for pin in pins.ALL_PINS:
        try:
            pin(ref)
        except Exception:          # a wrong value or an impossible shape
            return pin.__name__
    return None


def _ce_drop_shift(Z, y, ignore_index=-100):
    r = _ORIG["cross_entropy"](Z, y, ignore_index)
    Z = np.asarray(Z, dtype=np.float64)
    m = Z.max(axis=1)
    r["loss"] = np.where(r["loss"] != 0.0, r["loss"] - m, 0.0)   # "+ m" dropped
    return r


def _grad_sign(Z, y, lse, g):
    Z = np.asarray(Z, dtype=np.float64)
    p = np.exp(Z - lse[:, None])
    onehot = np.zeros_like(p)
    rows = np.nonzero((y >= 0) & (y < Z.shape[1]))[0]
    onehot[rows, y[rows]] = 1.0
    return g[:, None] * (p + onehot)                               # wrong sign


def _grads_transposed(X, W, dZ):
    return dZ @ np.asarray(W, dtype=np.float64).T, dZ.T @ X         # W transposed


def _shard_off_by_one(V, T):
    vs = V // T
    if V % T:
        raise ValueError
    return [(t * vs, (t + 1) * vs + 1) for t in range(T)]            # ranges overlap


def _scale_by_n(y, V, ignore_index=-100, dloss=None):
    valid = (np.asarray(y) >= 0) & (np.asarray(y) < V)
    if dloss is None:
        return valid / len(y)                                          # N, not N_valid
    return np.where(valid, dloss, 0.0)


def _merge_no_rescale(stats):
    r = _ORIG["merge_local_stats"](stats)
    m = stats[:, 0].max(axis=0)
    s = stats[:, 1].sum(axis=0)                                       # e^(m_t - m) dropped
    r["lse"] = m + np.log(s)
    return r


def _embed_no_mask(ids, W, V, T, t):
    start, end = ref.shard_bounds(V, T)[t]
    W_t = np.asarray(W, dtype=np.float64)[start:end]
    local = np.clip(np.asarray(ids) - start, 0, end - start - 1)
    return W_t[local]                                                 # zeroing step dropped


def _embed_bwd_keep_masked(ids, dOut, V, T, t):
    start, end = ref.shard_bounds(V, T)[t]
    ids = np.asarray(ids, dtype=np.int64)
    local = np.where((ids < start) | (ids >= end), 0, ids - start)
    dW_t = np.zeros((end - start, np.asarray(dOut).shape[1]))
    np.add.at(dW_t, local, np.asarray(dOut, dtype=np.float64))     # masked rows not zeroed
    return dW_t


def _embed_bwd_assign(ids, dOut, V, T, t):
    start, end = ref.shard_bounds(V, T)[t]
    ids = np.asarray(ids, dtype=np.int64)
    keep = (ids >= start) & (ids < end)
    dW_t = np.zeros((end - start, np.asarray(dOut).shape[1]))
    dW_t[ids[keep] - start] = np.asarray(dOut, dtype=np.float64)[keep]   # repeats overwrite, not add
    return dW_t


def _embed_bwd_global_row(ids, dOut, V, T, t):
    start, end = ref.shard_bounds(V, T)[t]
    ids = np.asarray(ids, dtype=np.int64)
    keep = (ids >= start) & (ids < end)
    dW_t = np.zeros((end - start, np.asarray(dOut).shape[1]))
    np.add.at(dW_t, np.clip(ids[keep], 0, end - start - 1), np.asarray(dOut, dtype=np.float64)[keep])  # no "- start"
    return dW_t


def _embed_sp_wrong_slice(ids, W, V, T, rank):
    ids = np.asarray(ids, dtype=np.int64)
    rows = len(ids) // T
    if len(ids) % T:
        raise ValueError
    return ref.embed(ids, W, V, T)[(T - 1 - rank) * rows:(T - rank) * rows]   # ranks reversed


def _dw_rows_no_onehot(X, W, y, lse, vocab_rows, n_valid, ignore_index=-100):
    W = np.asarray(W)
    vr = np.asarray(vocab_rows, dtype=np.int64)
    X64 = np.asarray(X, dtype=np.float64)
    Zv = X64 @ np.asarray(W[vr], dtype=np.float64).T
    valid = (np.asarray(y) >= 0) & (np.asarray(y) < W.shape[0]) & (np.asarray(y) != ignore_index)
    g = valid / max(1, n_valid)
    return (g[:, None] * np.exp(Zv - np.asarray(lse)[:, None])).T @ X64      # the -1[y = v] term dropped


def _ce_lse_unshifted(Z, y, ignore_index=-100):
    r = _ORIG["cross_entropy"](Z, y, ignore_index)
    with np.errstate(over="ignore"):
        r["lse"] = np.log(np.exp(np.asarray(Z, dtype=np.float64)).sum(axis=1))   # max shift dropped
    return r


def _shard_stats_unshifted(Z, y, V, T, ignore_index=-100):
    out = _ORIG["shard_local_stats"](Z, y, V, T, ignore_index)
    Z = np.asarray(Z, dtype=np.float64)
    for t, (a, b) in enumerate(ref.shard_bounds(V, T)):
        out[t, 0] = 0.0
        with np.errstate(over="ignore"):
            out[t, 1] = np.exp(Z[:, a:b]).sum(axis=1)                   # local max not subtracted
    return out


_ORIG = {k: getattr(ref, k) for k in ("cross_entropy", "merge_local_stats", "shard_local_stats")}

MUTANTS = {
    "ce_drop_max_term": ("cross_entropy", _ce_drop_shift),
    "grad_sign": ("grad_logits", _grad_sign),
    "grads_transposed": ("lmhead_grads", _grads_transposed),
    "shard_off_by_one": ("shard_bounds", _shard_off_by_one),
    "mean_scale_over_N": ("upstream_scale", _scale_by_n),
    "merge_no_rescale": ("merge_local_stats", _merge_no_rescale),
    "ce_lse_unshifted": ("cross_entropy", _ce_lse_unshifted),
    "shard_stats_unshifted": ("shard_local_stats", _shard_stats_unshifted),
    "embed_no_mask": ("embed_shard_partial", _embed_no_mask),
    "embed_bwd_keep_masked_rows": ("embed_shard_grad", _embed_bwd_keep_masked),
    "embed_bwd_assign_not_add": ("embed_shard_grad", _embed_bwd_assign),
    "embed_bwd_global_row": ("embed_shard_grad", _embed_bwd_global_row),
    "embed_sp_wrong_slice": ("embed_sp", _embed_sp_wrong_slice),
    "dw_rows_no_onehot": ("lmhead_ce_dw_rows", _dw_rows_no_onehot),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(ref, attr, fn)
    caught = _fails_some_pin()
    assert caught is not None, f"planted mistake {name} passed every pin"
