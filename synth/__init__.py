"""Seeded synthetic inputs for the vocab-parallel LM head + cross-entropy path.

This module only draws random numbers and rounds them to the storage type.  It
holds none of the method's arithmetic (no logits, no softmax, no gather), so
that both the CUDA path and the float64 oracle can consume the very same
inputs without sharing any computation.

Workloads (sizes of the tiled vocab-parallel LM head, "Vocab Parallelism",
MiniMind-tron book ch. 5, sec. 5.1-5.3):

  name      N       H     V       T  dtype  X        W                targets
  tiny      6       64    16      4  f32    N(0,1)   0.625*N(0,1)     uniform
  minimind  4096    512   6400    2  bf16   N(0,1)   N(0,0.02^2)      uniform
  v32k      8192    4096  32000   4  bf16   N(0,1)   N(0,0.02^2)      Zipf(1.1)
  v128k     16384   4096  128256  8  bf16   N(0,1)   N(0,0.02^2)      Zipf(1.1)
  v152k     32768   5120  151936  8  bf16   N(0,1)   N(0,0.02^2)      Zipf(1.1), 10% ignored

Draw order per workload (one ``numpy.random.default_rng(seed)`` stream):
X, then W, then targets, then the ignored positions.  bf16 values are rounded
from float32 with round-to-nearest-even on the host.

The tiny workload scales W so that logits have standard deviation 5, the
spread of the NumPy t=4 simulation on the interview note "Vocab parallelism:
how to split embedding and LM head" (code section): std(z) = 0.625*sqrt(64) = 5.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    H: int
    V: int
    T: int
    dtype: str            # "f32" or "bf16": storage/compute type of X and W
    w_std: float          # standard deviation of W entries
    targets: str          # "uniform" or "zipf"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.N


WORKLOADS = {
    "tiny": Workload("tiny", 6, 64, 16, 4, "f32", 0.625, "uniform", seed=1000),
    "minimind": Workload("minimind", 4096, 512, 6400, 2, "bf16", 0.02, "uniform", seed=1001),
    "v32k": Workload("v32k", 8192, 4096, 32000, 4, "bf16", 0.02, "zipf", seed=1002),
    "v128k": Workload("v128k", 16384, 4096, 128256, 8, "bf16", 0.02, "zipf", seed=1003),
    "v152k": Workload("v152k", 32768, 5120, 151936, 8, "bf16", 0.02, "zipf",
                      ignore_frac=0.1, seed=1004),
}


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Inputs here are finite normals, so no NaN handling is needed."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def zipf_ids(rng: np.random.Generator, n: int, V: int, s: float) -> np.ndarray:
    """Truncated Zipf(s) on ranks k = 1..V, P(k) ~ k^-s, id = k - 1 (inverse CDF)."""
    k = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-s))
    cdf /= cdf[-1]
    u = rng.random(n)
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, V - 1).astype(np.int64)


@dataclasses.dataclass
class Inputs:
    """One workload's inputs.  For bf16 workloads ``X``/``W`` are float32 arrays
    holding exactly the bf16 values and ``X_bits``/``W_bits`` are the raw bf16
    bit patterns; for f32 workloads the bits fields are None."""
    wl: Workload
    X: np.ndarray
    W: np.ndarray
    targets: np.ndarray
    X_bits: np.ndarray | None
    W_bits: np.ndarray | None


def _normal(rng, shape, std, dtype_bits):
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if dtype_bits:
        bits = round_to_bf16_bits(a)
        return bf16_bits_to_f32(bits), bits
    return a, None


def make_inputs(wl: Workload | str, *, N: int | None = None, seed: int | None = None,
                uniform_targets: bool = False) -> Inputs:
    """Draw X [N,H], W [V,H] and targets [N] for a workload.

    ``N`` overrides the token count (a smaller sample of the same distribution),
    ``seed`` the stream seed (e.g. one per rank), ``uniform_targets`` forces
    uniform ids (used to measure the gather without Zipf repeats)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    if N is not None:
        wl = dataclasses.replace(wl, N=N)
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    bf = wl.dtype == "bf16"
    X, Xb = _normal(rng, (wl.N, wl.H), 1.0, bf)
    W, Wb = _normal(rng, (wl.V, wl.H), wl.w_std, bf)
    if wl.targets == "zipf" and not uniform_targets:
        y = zipf_ids(rng, wl.N, wl.V, wl.zipf_s)
    else:
        y = rng.integers(0, wl.V, wl.N, dtype=np.int64)
    if wl.ignore_frac > 0:
        k = int(math.floor(wl.ignore_frac * wl.N))
        pos = rng.choice(wl.N, size=k, replace=False)
        y[pos] = IGNORE_INDEX
    return Inputs(wl, X, W, y, Xb, Wb)


def small_case(N: int, H: int, V: int, T: int, dtype: str, seed: int,
               w_std: float | None = None, targets: str = "uniform",
               ignore_frac: float = 0.0) -> Inputs:
    """An ad-hoc case with the same value distributions (parity tests over
    several tiles with ragged tails).  Default W scale keeps logits ~N(0, 1.6^2)."""
    if w_std is None:
        w_std = 1.6 / math.sqrt(H)
    wl = Workload(f"case_{N}x{H}x{V}", N, H, V, T, dtype, w_std, targets,
                  ignore_frac=ignore_frac, seed=seed)
    return make_inputs(wl)


def page_t4_simulation():
    """The seeded setup of the NumPy t=4 simulation on the interview note
    "Vocab parallelism: how to split embedding and LM head" (code section):
    n=6 tokens, V=16, t=4, ``default_rng(0)``, logits 5*N(0,1) drawn first,
    then targets uniform on [0, 16).  Returns (z [6,16] float64, y [6] int64)."""
    rng = np.random.default_rng(0)
    z = rng.standard_normal((6, 16)) * 5
    y = rng.integers(0, 16, 6)
    return z, y.astype(np.int64)
