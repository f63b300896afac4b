"""Seeded synthetic input generators.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds no arithmetic of the optimizer itself: it only draws activations X,
gradients G, weights W and test matrices with the shapes and spectra of the
workloads described in "Dobb: Shard-Local Preconditioning in Block-Diagonal
Eigenbases" (thelatestinai.com page, Table 1 caption; Figure 2 caption;
Table 6 notation).

Conventions
-----------
* A weight matrix W is m x n with y = W x (Table 6 notation): n is the input
  axis that is split into B blocks of width k = n / B.
* Activations X are stored row-major N x n: one row per token.
* Gradients are G = D X / N with D ~ N(0, 1) of shape m x N: the mean over
  tokens of g_i x_i^T for the layer y = W x (Table 6: x_i, g_i).
* bf16 inputs are produced by rounding the fp32 draw to nearest even; every
  consumer (CUDA path and oracle) sees the same rounded values.

Effective rank (Figure 2 caption) is exp(-sum p_i log p_i) as a fraction of
the dimension, p_i the normalised eigenvalues (or singular values).  The
spectra below are solved by bisection so that the drawn covariance has the
requested effective rank.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "entropy_rank_fraction",
    "geometric_spectrum",
    "power_law_spectrum",
    "haar_orthogonal",
    "matrix_with_singular_values",
    "activations",
    "ActivationStream",
    "gradients",
    "gradients_fp32",
    "weights",
    "round_bf16_np",
    "spd_with_gap",
    "ModelShapes",
    "gpt2_small_shapes",
    "gpt2_xl_shapes",
    "llama3_8b_shapes",
    "single_matrix_shapes",
    "layer_rank_schedule",
]


# ---------------------------------------------------------------------------
# spectra
# ---------------------------------------------------------------------------

def entropy_rank_fraction(values: np.ndarray) -> float:
    """exp(H(p)) / len(p) for p = values / sum(values); used only to solve
    the spectra of the generators below."""
    v = np.asarray(values, dtype=np.float64)
    p = v / v.sum()
    p = p[p > 0]
    return float(np.exp(-(p * np.log(p)).sum()) / len(v))


def _bisect(fn, lo, hi, target, increasing, iters=200):
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        val = fn(mid)
        if (val < target) == increasing:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def geometric_spectrum(n: int, target: float) -> np.ndarray:
    """lambda_i = r**i (i = 0..n-1), r in (0, 1) chosen so that the entropy
    effective rank fraction equals `target` (eigenvalues decaying
    geometrically, as the single-matrix workload prescribes)."""
    if not 0.0 < target < 1.0:
        raise ValueError("target effective rank must lie in (0, 1)")
    idx = np.arange(n, dtype=np.float64)

    def frac(r):
        return entropy_rank_fraction(np.exp(idx * math.log(r)))

    r = _bisect(frac, 1e-12, 1.0 - 1e-15, target, increasing=True)
    return np.exp(idx * math.log(r))


def power_law_spectrum(n: int, target: float) -> np.ndarray:
    """sigma_i proportional to i**(-alpha), alpha solved by bisection so that
    the entropy effective rank fraction of sigma equals `target`."""
    idx = np.arange(1, n + 1, dtype=np.float64)

    def frac(alpha):
        return entropy_rank_fraction(idx ** (-alpha))

    alpha = _bisect(frac, 0.0, 50.0, target, increasing=False)
    return idx ** (-alpha)


# ---------------------------------------------------------------------------
# random matrices
# ---------------------------------------------------------------------------

def haar_orthogonal(n: int, rng: np.random.Generator) -> np.ndarray:
    """Haar-distributed orthogonal matrix: QR of a Gaussian matrix with the
    signs of R's diagonal folded into Q (Mezzadri 2007)."""
    z = rng.standard_normal((n, n))
    q, r = np.linalg.qr(z)
    d = np.sign(np.diag(r))
    d[d == 0] = 1.0
    return q * d[None, :]


def matrix_with_singular_values(sigma: np.ndarray, rng: np.random.Generator,
                                m: Optional[int] = None) -> np.ndarray:
    """Y = U diag(sigma) V^T with U, V Haar random (square when m is None)."""
    n = len(sigma)
    m = n if m is None else m
    u = haar_orthogonal(m, rng)[:, :n]
    v = haar_orthogonal(n, rng)
    return (u * sigma[None, :]) @ v.T


def round_bf16_np(x: np.ndarray) -> np.ndarray:
    """Round an fp32 array to bfloat16 (nearest, ties to even), returned as
    fp32 holding bf16-representable values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = ((u + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(x)
    out = rounded.astype(np.uint32).view(np.float32).copy()
    out[nan] = np.nan
    return out


def activations(N: int, n: int, target: float, rng: np.random.Generator,
                dtype: str = "f32") -> np.ndarray:
    """X = Z diag(sqrt(lambda)) Q^T: N tokens x n features, Gaussian with a
    column covariance Q diag(lambda) Q^T of geometric spectrum at the given
    effective rank fraction and Haar eigenvectors.  The spectrum is scaled so
    that the mean eigenvalue is 1 (unit average feature variance)."""
    lam = geometric_spectrum(n, target)
    lam = lam * (n / lam.sum())
    q = haar_orthogonal(n, rng)
    z = rng.standard_normal((N, n))
    x = (z * np.sqrt(lam)[None, :]) @ q.T
    x = x.astype(np.float32)
    if dtype == "bf16":
        x = round_bf16_np(x)
    return x


class ActivationStream:
    """Activations of one matrix input step after step: a fixed column
    covariance Q diag(lambda) Q^T (geometric spectrum at the target effective
    rank, mean eigenvalue 1) and fresh Gaussian tokens at every draw, as a
    layer sees during training.  Q is Haar, or a shared Haar basis of the
    same width with rows permuted and sign-flipped (cheap distinct bases for
    many matrices of one width).  Draws are computed in fp32."""

    def __init__(self, n: int, target: float, rng: np.random.Generator,
                 shared_basis: Optional[np.ndarray] = None):
        lam = geometric_spectrum(n, target)
        lam = lam * (n / lam.sum())
        if shared_basis is None:
            q = haar_orthogonal(n, rng)
        else:
            perm = rng.permutation(n)
            flip = rng.choice(np.array([-1.0, 1.0]), size=n)
            q = shared_basis[perm] * flip[:, None]
        self.n = n
        self.mix = (np.sqrt(lam)[:, None] * q.T).astype(np.float32)   # diag(sqrt lam) Q^T

    def draw(self, N: int, rng: np.random.Generator, dtype: str = "f32") -> np.ndarray:
        z = rng.standard_normal((N, self.n), dtype=np.float32)
        x = z @ self.mix
        if dtype == "bf16":
            x = round_bf16_np(x)
        return np.ascontiguousarray(x, dtype=np.float32)


def gradients_fp32(m: int, X: np.ndarray, rng: np.random.Generator,
                   dtype: str = "f32") -> np.ndarray:
    """`gradients` evaluated in fp32 (the generator for model-sized runs)."""
    N = X.shape[0]
    d = rng.standard_normal((m, N), dtype=np.float32)
    g = (d @ np.asarray(X, dtype=np.float32)) / np.float32(N)
    if dtype == "bf16":
        g = round_bf16_np(g)
    return np.ascontiguousarray(g, dtype=np.float32)


def gradients(m: int, X: np.ndarray, rng: np.random.Generator,
              dtype: str = "f32") -> np.ndarray:
    """G = D X / N with D ~ N(0, 1) of shape m x N (tokens as columns)."""
    N = X.shape[0]
    d = rng.standard_normal((m, N))
    g = (d @ X.astype(np.float64)) / N
    g = g.astype(np.float32)
    if dtype == "bf16":
        g = round_bf16_np(g)
    return g


def weights(m: int, n: int, rng: np.random.Generator, dtype: str = "f32",
            std: float = 0.02) -> np.ndarray:
    w = (rng.standard_normal((m, n)) * std).astype(np.float32)
    if dtype == "bf16":
        w = round_bf16_np(w)
    return w


def spd_with_gap(k: int, rng: np.random.Generator, cond: float = 1e6,
                 min_rel_gap: float = 1e-3, max_tries: int = 100):
    """SPD block Q diag(lambda) Q^T with Haar Q and eigenvalues log-spaced on
    [1/cond, 1] (jittered, resampled until every relative gap between
    neighbours is at least `min_rel_gap`).  Returns (A, lambda, Q) in fp64."""
    for _ in range(max_tries):
        logs = np.linspace(0.0, -math.log(cond), k)
        if k > 2:
            h = math.log(cond) / (k - 1)
            logs[1:-1] += rng.uniform(-0.25 * h, 0.25 * h, size=k - 2)
        lam = np.exp(logs)
        gaps = np.abs(np.diff(lam)) / lam[:-1] if k > 1 else np.array([1.0])
        if gaps.min() >= min_rel_gap:
            q = haar_orthogonal(k, rng)
            a = (q * lam[None, :]) @ q.T
            a = 0.5 * (a + a.T)
            return a, lam, q
    raise RuntimeError("could not draw a spectrum with the requested gap")


# ---------------------------------------------------------------------------
# parameter sets (matrix shapes, m x n with n the blocked input axis)
# ---------------------------------------------------------------------------

@dataclass
class ModelShapes:
    name: str
    shapes: List[tuple]                 # (m, n) per matrix
    kinds: List[str] = field(default_factory=list)
    layer: List[int] = field(default_factory=list)

    @property
    def num_params(self) -> int:
        return int(sum(m * n for m, n in self.shapes))


def single_matrix_shapes(m: int = 768, n: int = 768) -> ModelShapes:
    return ModelShapes("single", [(m, n)], ["w"], [0])


def gpt2_small_shapes() -> ModelShapes:
    """12 layers x {q, k, v, o: 768x768; fc: 3072x768; proj: 768x3072}."""
    shapes, kinds, layer = [], [], []
    for li in range(12):
        for kind, (m, n) in (("q", (768, 768)), ("k", (768, 768)), ("v", (768, 768)),
                             ("o", (768, 768)), ("fc", (3072, 768)), ("proj", (768, 3072))):
            shapes.append((m, n)); kinds.append(kind); layer.append(li)
    return ModelShapes("gpt2-small", shapes, kinds, layer)


def gpt2_xl_shapes(include_embedding: bool = True) -> ModelShapes:
    """48 layers, d = 1600, MLP 6400, plus the tied 50257 x 1600 token
    embedding / head (1,554,971,200 parameters in total)."""
    shapes, kinds, layer = [], [], []
    for li in range(48):
        for kind, (m, n) in (("q", (1600, 1600)), ("k", (1600, 1600)), ("v", (1600, 1600)),
                             ("o", (1600, 1600)), ("fc", (6400, 1600)), ("proj", (1600, 6400))):
            shapes.append((m, n)); kinds.append(kind); layer.append(li)
    if include_embedding:
        shapes.append((50257, 1600)); kinds.append("wte"); layer.append(48)
    return ModelShapes("gpt2-xl", shapes, kinds, layer)


def llama3_8b_shapes() -> ModelShapes:
    """32 layers x {q, o: 4096x4096; k, v: 1024x4096; gate, up: 14336x4096;
    down: 4096x14336} plus 128256 x 4096 embedding and head."""
    shapes, kinds, layer = [], [], []
    for li in range(32):
        for kind, (m, n) in (("q", (4096, 4096)), ("k", (1024, 4096)), ("v", (1024, 4096)),
                             ("o", (4096, 4096)), ("gate", (14336, 4096)), ("up", (14336, 4096)),
                             ("down", (4096, 14336))):
            shapes.append((m, n)); kinds.append(kind); layer.append(li)
    shapes.append((128256, 4096)); kinds.append("embed"); layer.append(32)
    shapes.append((128256, 4096)); kinds.append("head"); layer.append(32)
    return ModelShapes("llama3-8b", shapes, kinds, layer)


def layer_rank_schedule(layer: int, num_layers: int, lo: float = 0.10,
                        hi: float = 0.40) -> float:
    """Effective-rank target varying linearly with depth from lo to hi."""
    if num_layers <= 1:
        return lo
    t = min(max(layer / (num_layers - 1), 0.0), 1.0)
    return lo + (hi - lo) * t
