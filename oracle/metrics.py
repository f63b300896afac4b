"""Measurements and parity rules used with the oracle.

TEST INFRASTRUCTURE ONLY (see `oracle/__init__.py`).

* `effective_rank` - [Dobb, Figure 2 caption]: exp(-sum p_i log p_i) as a
  fraction of the dimension, p_i the normalised eigenvalues (or singular
  values, [Dobb, Table 1 caption]).
* `orthogonality` - [Dobb, Table 1 caption]: ||O||_* / (sqrt(min(m, n)) ||O||_F),
  equal to 1 exactly when all singular values are equal.  Pinned by the
  printed Table 1(a) values.
* eigen residuals, sign agreement and parameter parity implement the
  comparison rules between the oracle and a second implementation.
"""
from __future__ import annotations

import math
from typing import Dict

import numpy as np

from .dobb import round_to_bf16

__all__ = [
    "effective_rank",
    "orthogonality",
    "eig_residuals",
    "sign_agreement",
    "w_rel_error",
    "bf16_parity",
]


def effective_rank(values: np.ndarray) -> float:
    v = np.abs(np.asarray(values, dtype=np.float64))
    p = v / v.sum()
    nz = p[p > 0]
    return float(math.exp(-(nz * np.log(nz)).sum()) / len(v))


def orthogonality(O: np.ndarray) -> float:
    O = np.asarray(O, dtype=np.float64)
    sv = np.linalg.svd(O, compute_uv=False)
    fro = math.sqrt(float((sv ** 2).sum()))
    return float(sv.sum() / (math.sqrt(min(O.shape)) * fro))


def eig_residuals(A: np.ndarray, Q: np.ndarray, lam: np.ndarray) -> Dict[str, float]:
    """Residuals of a claimed eigendecomposition A = Q diag(lam) Q^T, all in
    fp64: ||A Q - Q Lambda||_F / ||A||_F, ||Q^T Q - I||_F and the
    reconstruction ||Q Lambda Q^T - A||_F / ||A||_F."""
    A = np.asarray(A, dtype=np.float64)
    Q = np.asarray(Q, dtype=np.float64)
    lam = np.asarray(lam, dtype=np.float64)
    fro = np.linalg.norm(A)
    fro = fro if fro > 0 else 1.0
    k = A.shape[0]
    return {
        "residual": float(np.linalg.norm(A @ Q - Q * lam[None, :]) / fro),
        "orth": float(np.linalg.norm(Q.T @ Q - np.eye(k))),
        "recon": float(np.linalg.norm((Q * lam[None, :]) @ Q.T - A) / fro),
    }


def sign_agreement(C_ref: np.ndarray, S_test: np.ndarray, k: int,
                   band: float = 1e-5) -> Dict[str, float]:
    """Score a sign matrix against exact coefficients C_ref (same basis).

    Per column block b, RMS_b = RMS(C_ref[:, block b]).  A disagreement
    sign(C_ref) != S_test is tolerated only where |C_ref| < band * RMS_b.
    Returns the number of disagreements, the number outside the band, and the
    fraction of disagreeing entries."""
    C = np.asarray(C_ref, dtype=np.float64)
    S = np.asarray(S_test, dtype=np.float64)
    m, n = C.shape
    B = n // k
    Cb = C.reshape(m, B, k)
    rms = np.sqrt((Cb ** 2).mean(axis=(0, 2)))
    thr = (band * rms)[None, :, None]
    dis = np.sign(Cb) != S.reshape(m, B, k)
    outside = dis & (np.abs(Cb) >= thr)
    return {
        "disagree": int(dis.sum()),
        "outside_band": int(outside.sum()),
        "fraction": float(dis.sum()) / max(C.size, 1),
    }


def w_rel_error(W_test: np.ndarray, W_ref: np.ndarray) -> float:
    """max_ij |W_test - W_ref| / max_ij |W_ref| (normwise max relative)."""
    W_ref = np.asarray(W_ref, dtype=np.float64)
    d = np.abs(np.asarray(W_test, dtype=np.float64) - W_ref).max() if W_ref.size else 0.0
    scale = np.abs(W_ref).max() if W_ref.size else 1.0
    return float(d / (scale if scale > 0 else 1.0))


def bf16_parity(W_test_bf16: np.ndarray, W_exact: np.ndarray, tol: float = 1e-5) -> Dict[str, int]:
    """Score bf16 parameters against the exact (unrounded, fp64) result.

    A second implementation computes a pre-rounding value y within
    tol * max|W_exact| of the exact result and rounds it to bf16; rounding is
    monotone, so every acceptable output lies in
    [round_to_bf16(W_exact - band), round_to_bf16(W_exact + band)],
    band = tol * max|W_exact|.  Returns counts of outputs equal to the
    rounded exact value, other outputs inside that interval, and violations."""
    We = np.asarray(W_exact, dtype=np.float64)
    Wt = np.asarray(W_test_bf16, dtype=np.float64)
    band = tol * (float(np.abs(We).max()) if We.size else 1.0)
    lo = round_to_bf16(We - band)
    hi = round_to_bf16(We + band)
    eq = Wt == round_to_bf16(We)
    inside = (Wt >= lo) & (Wt <= hi)
    return {"exact": int(eq.sum()), "tolerated": int((~eq & inside).sum()),
            "violations": int((~inside).sum())}
