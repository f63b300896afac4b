"""Shared helpers of the GPU parity tests: build seeded inputs, run the CUDA
path through the C ABI and the fp64 oracle on the same inputs, and score the
results with the oracle's parity rules.

Tolerances (the bar every GPU test applies):
  * block moments A: relative Frobenius error <= 1e-5 per block;
  * eigen-blocks: ||Q Lambda Q^T - A||_F / ||A||_F <= 1e-5 and
    ||A Q - Q Lambda||_F / ||A||_F <= 1e-5 (fp64 evaluation against the
    oracle's A), ||Q^T Q - I||_F <= 1e-5 * sqrt(k) (k columns, each
    normalised to fp32 rounding), eigenvalues within 1e-5 ||A||_F of the
    oracle's (Weyl's bound for a 1e-5 backward error);
  * signs: disagreements with sign(C_ref) only where |C_ref| < 1e-5 RMS(C_b)
    and in fewer than 1e-4 of the entries, C_ref computed in fp64 with the
    GPU's own basis (the basis of an ill-conditioned block is determined
    only to fp32 accuracy, so the sign check must not depend on it);
  * parameters: fp32 W within 1e-5 max relative error; bf16 W bitwise equal
    to the rounded fp64 result except where that result lies within
    1e-5 max|W| of a rounding midpoint (oracle.metrics.bf16_parity), both
    computed from the GPU's signs at the tolerated entries.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from block_eigenbasis_preconditioning_gb300 import inputs as I
from oracle import dobb as O
from oracle import metrics as MX

TOL_A = 1e-5
TOL_EIG = 1e-5
TOL_SIGN_BAND = 1e-5
TOL_SIGN_FRAC = 1e-4
TOL_W = 1e-5

TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device="cuda", dtype=TORCH[dtype]).contiguous()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def make_problem(shapes, N, eff, seed, param_dtype="f32", act_dtype="f32"):
    """Seeded inputs for a list of (m, n): X (N x n), G = D X / N, W."""
    rng = np.random.default_rng(seed)
    Xs, Gs, Ws = [], [], []
    for (m, n) in shapes:
        X = I.activations(N, n, eff, rng, dtype=act_dtype)
        Xs.append(X)
        Gs.append(I.gradients(m, X, rng, dtype=param_dtype))
        Ws.append(I.weights(m, n, rng, dtype=param_dtype))
    return Xs, Gs, Ws


def make_output_side_problem(shapes, N, eff, seed, param_dtype="f32", act_dtype="f32"):
    """Seeded inputs of the output-gradient side for a list of (m, n):
    output gradients D (N x m) with a geometric-spectrum covariance, input
    activations X (N x n), G = D^T X / N (a linear layer's weight gradient)
    and W."""
    rng = np.random.default_rng(seed)
    Ds, Gs, Ws = [], [], []
    for (m, n) in shapes:
        D = I.activations(N, m, eff, rng, dtype=act_dtype)
        X = I.activations(N, n, 0.5, rng)
        g = (D.astype(np.float64).T @ X.astype(np.float64) / N).astype(np.float32)
        Ds.append(D)
        Gs.append(I.round_bf16_np(g) if param_dtype == "bf16" else g)
        Ws.append(I.weights(m, n, rng, dtype=param_dtype))
    return Ds, Gs, Ws


def check_moments(opt, orc, matrices=None):
    worst = 0.0
    for i in (matrices if matrices is not None else range(len(orc.shapes))):
        Ag = to_np(opt.tensor("moments", i))
        Ar = orc.A[i]
        for b in range(Ar.shape[0]):
            fro = np.linalg.norm(Ar[b])
            err = np.linalg.norm(Ag[b] - Ar[b]) / (fro if fro > 0 else 1.0)
            worst = max(worst, err)
            assert np.array_equal(Ag[b], Ag[b].T), "A must stay exactly symmetric"
    assert worst <= TOL_A, f"block moments relative error {worst:.3e}"
    return worst


def check_bases(opt, A_ref_list, matrices=None):
    """Eigen residuals of the GPU bases against fp64 reference moments."""
    worst = {"residual": 0.0, "orth": 0.0, "recon": 0.0, "lam": 0.0}
    for i in (matrices if matrices is not None else range(len(A_ref_list))):
        Q = to_np(opt.tensor("bases", i))
        lam = to_np(opt.tensor("eigvals", i))
        Ar = A_ref_list[i]
        for b in range(Ar.shape[0]):
            k = Ar.shape[1]
            r = MX.eig_residuals(Ar[b], Q[b], lam[b])
            assert r["residual"] <= TOL_EIG, f"matrix {i} block {b}: residual {r['residual']:.3e}"
            assert r["recon"] <= TOL_EIG, f"matrix {i} block {b}: reconstruction {r['recon']:.3e}"
            assert r["orth"] <= TOL_EIG * max(1.0, np.sqrt(k)), f"orthogonality {r['orth']:.3e}"
            lam_ref = np.sort(np.linalg.eigvalsh(0.5 * (Ar[b] + Ar[b].T)))[::-1]
            fro = np.linalg.norm(Ar[b])
            dl = np.abs(lam[b] - lam_ref).max() / (fro if fro > 0 else 1.0)
            assert dl <= TOL_EIG, f"eigenvalues off by {dl:.3e} ||A||"
            assert np.all(np.diff(lam[b]) <= 0), "eigenvalues must be sorted descending"
            for key in ("residual", "orth", "recon"):
                worst[key] = max(worst[key], r[key])
            worst["lam"] = max(worst["lam"], dl)
    return worst


def check_update(W_prev, M_prev, G, Q_gpu, S_gpu, W_gpu, M_gpu, beta1, lr, s, param_dtype, k,
                 basis_dtype="f32", side="input"):
    """Score one matrix's update against the oracle run with the GPU basis
    (rounded by the oracle itself when the basis is stored in bf16).  All
    matrices in the caller's (m, n) layout; side "output" scores Dobb-G (row
    blocks: the sign band is taken per row block of C)."""
    ref = O.update_from_bases(W_prev, M_prev, G, Q_gpu, beta1, lr, s, param_dtype,
                              basis_dtype=basis_dtype, side=side)
    # momentum
    dm = np.abs(M_gpu - ref["M"]).max() / max(np.abs(ref["M"]).max(), 1e-30)
    assert dm <= 1e-6, f"momentum relative error {dm:.3e}"
    # signs
    if side == "output":
        sa = MX.sign_agreement(ref["C"].T, np.asarray(S_gpu).T, k, TOL_SIGN_BAND)
    else:
        sa = MX.sign_agreement(ref["C"], S_gpu, k, TOL_SIGN_BAND)
    assert sa["outside_band"] == 0, f"{sa['outside_band']} sign flips outside the band"
    assert sa["fraction"] < TOL_SIGN_FRAC, f"sign disagreement fraction {sa['fraction']:.2e}"
    # parameters, scored with the GPU's signs at the tolerated entries
    ref2 = O.update_from_bases(W_prev, M_prev, G, Q_gpu, beta1, lr, s, "f32", S_override=S_gpu,
                               basis_dtype=basis_dtype, side=side)
    if param_dtype == "f32":
        e = MX.w_rel_error(W_gpu, ref2["W"])
        assert e <= TOL_W, f"W max relative error {e:.3e}"
        return {"sign": sa, "w_err": e, "m_err": dm}
    res = MX.bf16_parity(W_gpu, ref2["W"], TOL_W)
    assert res["violations"] == 0, f"bf16 W: {res}"
    return {"sign": sa, "bf16": res, "m_err": dm}


def l2_update_error_bound(M_new, Q, k, m):
    """Frobenius bound on the error of a Dobb-l2 U computed in fp32 (the
    tolerance is derived from the arithmetic, not chosen).  The projection's
    k-term fp32 dot products have |C~ - C|_ij <= g (|M| |Q|)_ij, g = k u /
    (1 - k u), u = 2^-24; normalising column j to norm sqrt(m) moves it by at
    most 2 sqrt(m) ||e_j|| / ||c_j||; with Q_b orthonormal ||dU_b||_F equals
    ||dS_b||_F.  Columns with little momentum energy dominate, as tiny |C|
    entries do for the sign."""
    u = 2.0 ** -24
    g = k * u / (1 - k * u)
    Mn = np.abs(np.asarray(M_new, dtype=np.float64))
    B = Q.shape[0]
    tot = 0.0
    for b in range(B):
        sl = slice(b * k, (b + 1) * k)
        C = np.asarray(M_new, dtype=np.float64)[:, sl] @ Q[b]
        E = g * (Mn[:, sl] @ np.abs(Q[b]))
        cn = np.linalg.norm(C, axis=0)
        en = np.linalg.norm(E, axis=0)
        ok = cn > 0
        tot += float(((2 * math.sqrt(m) * en[ok] / cn[ok]) ** 2).sum())
        # plus the rounding of the normalisation and the reconstruction
        tot += (8 * k * u) ** 2 * m * k
    return math.sqrt(tot)


def check_update_l2(W_prev, M_prev, G, Q_gpu, W_gpu, M_gpu, beta1, lr, s, param_dtype,
                    basis_dtype="f32", side="input"):
    """Score a Dobb-l2 update (column l2 normalisation) against the oracle run
    with the GPU basis.  The normalised coefficients are continuous, so W is
    compared directly, in Frobenius norm, within lr s times the fp32 bound of
    `l2_update_error_bound` (plus, for bf16 parameters, half a bf16 quantum per
    entry, 2^-8 |W|).  Side "output" (Dobb-G) normalises the rows of C: the
    bound is that of the transposed problem."""
    ref = O.update_from_bases(W_prev, M_prev, G, Q_gpu, beta1, lr, s, "f32",
                              basis_dtype=basis_dtype, norm="l2", side=side)
    dm = np.abs(M_gpu - ref["M"]).max() / max(np.abs(ref["M"]).max(), 1e-30)
    assert dm <= 1e-6, f"momentum relative error {dm:.3e}"
    Mt = ref["M"].T if side == "output" else ref["M"]
    m = Mt.shape[0]
    k = Q_gpu.shape[1]
    bound = lr * s * l2_update_error_bound(Mt, Q_gpu, k, m)
    if param_dtype == "bf16":
        bound += float(np.linalg.norm(2.0 ** -8 * np.abs(ref["W"])))
    err = float(np.linalg.norm(np.asarray(W_gpu, dtype=np.float64) - ref["W"]))
    assert err <= bound, f"W error {err:.3e} above the fp32 bound {bound:.3e}"
    return err, bound
