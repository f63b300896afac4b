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


def moment_tolerance(N):
    """Tolerance of fp32 block moments accumulated over N tokens: max(1e-5,
    N u / 2), u = 2^-24.  Each of the N additions into an fp32 accumulator
    may lose up to u of the partial sum (N u relative on the diagonal, whose
    terms are all positive); an accumulator that truncates loses half of that
    on average, which is what a sum on the tensor cores shows (1.1e-5 at
    N = 4096).  Small N keeps the fixed 1e-5, which the per-token moment tests
    (ragged N up to 300) use; at N = 4096 a block missing one token (2.4e-4)
    still fails."""
    return max(TOL_A, N * 2.0 ** -24 / 2)


def check_moments(opt, orc, matrices=None, N=None):
    """GPU block moments against the oracle's, relative Frobenius per block,
    within TOL_A, or within `moment_tolerance(N)` when the token count of the
    accumulations is given."""
    tol = moment_tolerance(N) if N is not None else TOL_A
    worst = 0.0
    for i in (matrices if matrices is not None else range(len(orc.shapes))):
        Ag = to_np(opt.tensor("moments", i))
        Ar = orc.A[i]
        for b in range(Ar.shape[0]):
            fro = np.linalg.norm(Ar[b])
            err = np.linalg.norm(Ag[b] - Ar[b]) / (fro if fro > 0 else 1.0)
            worst = max(worst, err)
            assert np.array_equal(Ag[b], Ag[b].T), "A must stay exactly symmetric"
            assert err <= tol, f"matrix {i} block {b}: moments relative error {err:.3e} > {tol:.3e}"
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


def l2_update_entry_bound(M_new, Q, lr_s):
    """Per-entry bound on |U_gpu - U| * lr s for a Dobb-l2 update computed in
    fp32 (a tolerance derived from the arithmetic, not chosen), for the
    registered (input-side) layout: M_new m x n, Q (B, k, k).

    * C = M_b Q_b from an fp32 momentum (one rounding, u |M|) by k-term fp32
      dot products: |C~ - C|_ij <= (g_k + u) (|M_b| |Q_b|)_ij = E_ij,
      g_k = k u / (1 - k u), u = 2^-24.
    * S_j = sqrt(m) c_j / ||c_j||; to first order
      |dS_ij| <= sqrt(m) (E_ij + |C_ij| ||E_j|| / ||c_j||) / ||c_j||, capped at
      2 sqrt(m) (both sides lie in [-sqrt(m), sqrt(m)]), plus eta |S_ij| for
      the fp32 column sum of squares over the m rows, its square root and the
      division, eta = (m + 8) u.
    * U_b = S_b Q_b^T by k-term fp32 dot products:
      |dU| <= |dS| |Q_b|^T + g_k |S_b| |Q_b|^T.
    Returns lr s |dU| bound (m x n) and the exact U."""
    u = 2.0 ** -24
    M_new = np.asarray(M_new, dtype=np.float64)
    m, n = M_new.shape
    B, k, _ = Q.shape
    g = k * u / (1 - k * u)
    eta = (m + 8) * u
    out = np.empty_like(M_new)
    U = np.empty_like(M_new)
    for b in range(B):
        sl = slice(b * k, (b + 1) * k)
        Qb = np.asarray(Q[b], dtype=np.float64)
        C = M_new[:, sl] @ Qb
        E = (g + u) * (np.abs(M_new[:, sl]) @ np.abs(Qb))
        cn = np.linalg.norm(C, axis=0)
        en = np.linalg.norm(E, axis=0)
        safe = np.where(cn > 0, cn, 1.0)
        S = np.where(cn > 0, math.sqrt(m) * C / safe, 0.0)
        dS = math.sqrt(m) * (E + np.abs(C) * (en / safe)) / safe
        dS = np.minimum(np.where(cn > 0, dS, 2 * math.sqrt(m)), 2 * math.sqrt(m)) + eta * np.abs(S)
        out[:, sl] = lr_s * (dS @ np.abs(Qb).T + g * (np.abs(S) @ np.abs(Qb).T))
        U[:, sl] = S @ Qb.T
    return out, U


def bf16_parity_entrywise(W_test_bf16, W_exact, band):
    """bf16 parameters against the exact result with a per-entry band: the
    pre-rounding value lies within band_ij of W_exact_ij and is rounded once
    (monotone), so the output must lie in
    [round(W_exact - band), round(W_exact + band)]."""
    We = np.asarray(W_exact, dtype=np.float64)
    Wt = np.asarray(W_test_bf16, dtype=np.float64)
    lo = O.round_to_bf16(We - band)
    hi = O.round_to_bf16(We + band)
    return int((~((Wt >= lo) & (Wt <= hi))).sum())


def check_update_l2(W_prev, M_prev, G, Q_gpu, W_gpu, M_gpu, beta1, lr, s, param_dtype,
                    basis_dtype="f32", side="input"):
    """Score a Dobb-l2 update (column l2 normalisation) against the oracle run
    with the GPU basis, entry by entry: every W entry within lr s times the
    per-entry fp32 bound of `l2_update_entry_bound` (plus the final rounding
    of the parameter: one fp32 rounding, or a bf16 rounding of a value inside
    that band).  Side "output" (Dobb-G) normalises the rows of C: the bound is
    that of the transposed problem, transposed back."""
    ref = O.update_from_bases(W_prev, M_prev, G, Q_gpu, beta1, lr, s, "f32",
                              basis_dtype=basis_dtype, norm="l2", side=side)
    dm = np.abs(M_gpu - ref["M"]).max() / max(np.abs(ref["M"]).max(), 1e-30)
    assert dm <= 1e-6, f"momentum relative error {dm:.3e}"
    Mt = ref["M"].T if side == "output" else ref["M"]
    Qb = O.basis_for_update(Q_gpu, basis_dtype)
    band, U = l2_update_entry_bound(Mt, Qb, lr * s)
    if side == "output":
        band, U = band.T, U.T
    Wg = np.asarray(W_gpu, dtype=np.float64)
    if param_dtype == "bf16":
        bad = bf16_parity_entrywise(Wg, ref["W"], band)
        assert bad == 0, f"{bad} bf16 W entries outside the per-entry fp32 band"
    else:
        u = 2.0 ** -24
        err = np.abs(Wg - ref["W"])
        # one rounding of the fused W - (lr s) U, and lr s itself rounded to fp32
        lim = band + u * np.abs(ref["W"]) + u * lr * s * np.abs(U)
        bad = int((err > lim).sum())
        assert bad == 0, (f"{bad} W entries outside the per-entry bound "
                          f"(worst ratio {float((err / lim).max()):.3g})")
    err = np.abs(Wg - ref["W"]).max()
    return float(err), float(band.max())
