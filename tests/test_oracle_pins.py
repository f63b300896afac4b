"""Pins of the fp64 oracle against facts fixed outside the oracle itself:
values printed on the pages, closed forms, brute force on tiny inputs,
invariants of the method, and an independent library routine (LAPACK)."""
import itertools
import math
import os

import numpy as np
import pytest

from block_eigenbasis_preconditioning_gb300 import inputs as I
from oracle import dobb as O
from oracle import metrics as MX

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_table1a():
    rows = []
    with open(os.path.join(GOLDEN, "table1a_orthogonality.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(v) for v in line.split()])
    return rows


# --------------------------------------------------------------------------
# Table 1(a): the orthogonality metric on the power-law construction
# --------------------------------------------------------------------------

def test_table1a_orthogonality_metric():
    rows = _load_table1a()
    rng = np.random.default_rng(0)
    for eff, orth_y, orth_sign in rows:
        sigma = I.power_law_spectrum(768, eff)
        Y = I.matrix_with_singular_values(sigma, rng)
        # the drawn matrix has the prescribed effective rank
        assert abs(MX.effective_rank(np.linalg.svd(Y, compute_uv=False)) - eff) < 1e-6
        # printed to three digits: the metric of Y depends only on sigma
        assert abs(MX.orthogonality(Y) - orth_y) <= 5e-4 + 1e-9
        # sign(Y) depends on the random singular vectors: agree within 0.012
        assert abs(MX.orthogonality(np.sign(Y)) - orth_sign) <= 0.012


def test_orthogonality_equals_one_iff_equal_singular_values():
    rng = np.random.default_rng(1)
    Q = I.haar_orthogonal(50, rng)
    assert abs(MX.orthogonality(Q) - 1.0) < 1e-12
    assert abs(MX.orthogonality(3.0 * Q[:, :20]) - 1.0) < 1e-12
    Y = I.matrix_with_singular_values(np.array([2.0, 1.0, 1.0]), rng)
    assert MX.orthogonality(Y) < 1.0 - 1e-3


# --------------------------------------------------------------------------
# eigensolver pins
# --------------------------------------------------------------------------

def test_sym_schur2_closed_form():
    rng = np.random.default_rng(2)
    for _ in range(200):
        a, b, d = rng.standard_normal(3) * rng.uniform(0.1, 10, 3)
        A = np.array([[a, b], [b, d]])
        c, s = O.sym_schur2(A, 0, 1)
        J = np.array([[c, s], [-s, c]])
        Bm = J.T @ A @ J
        assert abs(Bm[0, 1]) <= 1e-14 * np.abs(A).max()
        assert abs(c * c + s * s - 1.0) < 1e-15
        lam, V, _ = O.jacobi_eigh(A)
        closed = np.array([(a + d) / 2 + math.sqrt(((a - d) / 2) ** 2 + b * b),
                           (a + d) / 2 - math.sqrt(((a - d) / 2) ** 2 + b * b)])
        assert np.allclose(np.sort(lam)[::-1], closed, rtol=0, atol=1e-13 * np.abs(A).max())
        # the closed-form eigenvector of the larger root is (b, lambda_+ - a)
        v = np.array([b, closed[0] - a])
        if np.linalg.norm(v) > 1e-8:
            v /= np.linalg.norm(v)
            lam_c, V_c = O.canonicalize(lam, V)
            assert abs(abs(V_c[:, 0] @ v) - 1.0) < 1e-12


def _charpoly_brute_force(A):
    """det(A - x I) expanded over all permutations (Leibniz), as a
    polynomial in x with coefficients from low to high degree."""
    n = A.shape[0]
    total = np.zeros(n + 1)
    for perm in itertools.permutations(range(n)):
        inv = sum(1 for i in range(n) for j in range(i + 1, n) if perm[i] > perm[j])
        poly = np.array([1.0])
        for i in range(n):
            j = perm[i]
            entry = np.array([A[i, j], -1.0]) if i == j else np.array([A[i, j]])
            poly = np.convolve(poly, entry)
        padded = np.zeros(n + 1)
        padded[:len(poly)] = poly
        total += (-1) ** inv * padded
    return total


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_jacobi_matches_characteristic_polynomial_roots(k):
    rng = np.random.default_rng(10 + k)
    for _ in range(20):
        Z = rng.standard_normal((k, k))
        A = Z + Z.T
        coeffs = _charpoly_brute_force(A)
        roots = np.sort(np.real(np.roots(coeffs[::-1])))
        lam, V, _ = O.jacobi_eigh(A)
        assert np.allclose(np.sort(lam), roots, atol=1e-9 * max(1.0, np.abs(A).max()))
        r = MX.eig_residuals(A, V, lam)
        assert r["residual"] < 1e-13 and r["orth"] < 1e-13


@pytest.mark.parametrize("k", [8, 24, 40])
def test_jacobi_agrees_with_lapack(k):
    rng = np.random.default_rng(k)
    X = I.activations(4 * k, k, 0.3, rng)
    A = X.T.astype(np.float64) @ X / (4 * k)
    lam_j, V_j, sweeps = O.jacobi_eigh(A)
    lam_l, V_l = O.lapack_eigh(A)
    lam_j, V_j = O.canonicalize(lam_j, V_j)
    lam_l, V_l = O.canonicalize(lam_l, V_l)
    fro = np.linalg.norm(A)
    # Weyl: eigenvalues of two backward-stable solvers agree to O(eps ||A||)
    assert np.abs(lam_j - lam_l).max() <= 1e-13 * fro
    for lam, V in ((lam_j, V_j), (lam_l, V_l)):
        r = MX.eig_residuals(A, V, lam)
        assert r["residual"] < 1e-13 and r["orth"] < 1e-13 and r["recon"] < 1e-13
    # eigenvectors of well separated eigenvalues agree up to the sign fix
    gaps = np.minimum(np.abs(np.diff(lam_l, prepend=np.inf)), np.abs(np.diff(lam_l, append=-np.inf)))
    ok = gaps > 1e-6 * fro
    assert ok.sum() >= k // 2
    assert np.abs(np.abs((V_j * V_l).sum(axis=0))[ok] - 1.0).max() < 1e-8
    assert 1 <= sweeps <= 20


def test_refresh_bases_routes_agree():
    rng = np.random.default_rng(3)
    A = np.stack([I.spd_with_gap(16, rng, cond=1e4)[0] for _ in range(3)])
    Qj, lj = O.refresh_bases(A, "jacobi")
    Ql, ll = O.refresh_bases(A, "lapack")
    assert np.abs(lj - ll).max() < 1e-13
    assert np.abs(Qj - Ql).max() < 1e-9       # distinct eigenvalues, canonical signs
    for b in range(3):
        assert np.all(np.diff(lj[b]) <= 0)


# --------------------------------------------------------------------------
# update pins
# --------------------------------------------------------------------------

def _rand_case(rng, m=12, n=8, B=2):
    k = n // B
    M = rng.standard_normal((m, n))
    G = rng.standard_normal((m, n))
    W = rng.standard_normal((m, n)) * 0.02
    Q = np.stack([I.haar_orthogonal(k, rng) for _ in range(B)])
    return M, G, W, Q


def test_identity_basis_gives_sign_of_momentum():
    rng = np.random.default_rng(4)
    M, G, W, _ = _rand_case(rng)
    Q = np.broadcast_to(np.eye(4), (2, 4, 4)).copy()
    r = O.update_from_bases(W, M, G, Q, 0.9, 0.02, 1.5)
    Mn = 0.9 * M + G
    assert np.array_equal(r["U"], np.sign(Mn))
    assert np.array_equal(r["W"], W - 0.02 * 1.5 * np.sign(Mn))


def test_update_norm_is_sqrt_nnz():
    rng = np.random.default_rng(5)
    M, G, W, Q = _rand_case(rng, m=33, n=24, B=3)
    r = O.update_from_bases(W, M, G, Q, 0.95, 0.02, 1.0)
    k = 8
    for b in range(3):
        Ub = r["U"][:, b * k:(b + 1) * k]
        Sb = r["S"][:, b * k:(b + 1) * k]
        assert abs((Ub ** 2).sum() - np.count_nonzero(Sb)) < 1e-10 * Ub.size
    # exact zeros in C: the norm counts only nonzero signs
    M2 = M.copy()
    M2[0, :] = 0.0
    G2 = G.copy()
    G2[0, :] = 0.0
    r2 = O.update_from_bases(W, M2, G2, Q, 0.95, 0.02, 1.0)
    assert np.count_nonzero(r2["S"]) == 33 * 24 - 24
    assert abs((r2["U"] ** 2).sum() - (33 * 24 - 24)) < 1e-9


def test_table9_rms_identity():
    """[Dobb, Table 9]: a Dobb raw update O with ||O||_F^2 = n scaled by
    s = tau sqrt(max(m, n)) has RMS tau sqrt(max(m, n) / m).  With U the
    unscaled sign reconstruction, O = U / sqrt(m)."""
    rng = np.random.default_rng(6)
    for (m, n, B) in ((40, 24, 3), (16, 48, 4)):
        M, G, W, Q = _rand_case(rng, m=m, n=n, B=B)
        U = O.update_from_bases(W, M, G, Q, 0.95, 1.0, 1.0)["U"]
        Ob = U / math.sqrt(m)
        assert abs((Ob ** 2).sum() - n) < 1e-9 * n
        tau = 0.2
        s = tau * math.sqrt(max(m, n))
        rms = math.sqrt(((s * Ob) ** 2).mean())
        assert abs(rms - tau * math.sqrt(max(m, n) / m)) < 1e-12


def test_invariances():
    rng = np.random.default_rng(7)
    M, G, W, Q = _rand_case(rng, m=20, n=12, B=3)
    base = O.update_from_bases(W, M, G, Q, 0.95, 0.02, 1.0)["U"]
    # column sign flips and permutations of every Q_b
    Q2 = Q.copy()
    for b in range(3):
        flips = rng.choice([-1.0, 1.0], size=4)
        perm = rng.permutation(4)
        Q2[b] = (Q[b] * flips[None, :])[:, perm]
    U2 = O.update_from_bases(W, M, G, Q2, 0.95, 0.02, 1.0)["U"]
    assert np.abs(U2 - base).max() < 1e-12
    # positive scaling of the momentum
    U3 = O.update_from_bases(W, 3.7 * M, 3.7 * G, Q, 0.95, 0.02, 1.0)["U"]
    assert np.abs(U3 - base).max() < 1e-12
    # positive scaling of the second moment leaves the canonical basis unchanged
    A = np.stack([I.spd_with_gap(4, rng, cond=100.0)[0] for _ in range(2)])
    Qa, la = O.refresh_bases(A, "jacobi")
    Qb, lb = O.refresh_bases(5.0 * A, "jacobi")
    assert np.abs(Qa - Qb).max() < 1e-12 and np.abs(5.0 * la - lb).max() < 1e-12


# --------------------------------------------------------------------------
# Dobb-G: output-gradient basis ([Dobb, Tables 9, 12, 13])
# --------------------------------------------------------------------------

def test_dobb_g_table9_norm():
    """[Dobb, Table 9]: Dobb-G's raw update has ||O||_F^2 = m with RMS
    tau sqrt(max(m, n) / n) at s = tau sqrt(max(m, n)): O = U / sqrt(n)."""
    rng = np.random.default_rng(61)
    for (m, n, B) in ((24, 40, 3), (48, 16, 4)):
        k = m // B
        M, G, W = rng.standard_normal((3, m, n))
        Q = np.stack([I.haar_orthogonal(k, rng) for _ in range(B)])
        U = O.update_from_bases(W, M, G, Q, 0.95, 1.0, 1.0, side="output")["U"]
        Ob = U / math.sqrt(n)
        assert abs((Ob ** 2).sum() - m) < 1e-9 * m
        tau = 0.2
        rms = math.sqrt(((tau * math.sqrt(max(m, n)) * Ob) ** 2).mean())
        assert abs(rms - tau * math.sqrt(max(m, n) / n)) < 1e-12


@pytest.mark.parametrize("norm", ["sign", "l2"])
def test_dobb_g_is_dobb_on_the_transpose(norm):
    """Row blocks of W with bases applied from the left are the column blocks
    of W^T: Dobb-G(W, M, G) = Dobb(W^T, M^T, G^T)^T with the same bases."""
    rng = np.random.default_rng(62)
    m, n, B = 18, 10, 3
    k = m // B
    M, G, W = rng.standard_normal((3, m, n))
    Q = np.stack([I.haar_orthogonal(k, rng) for _ in range(B)])
    rg = O.update_from_bases(W, M, G, Q, 0.9, 0.05, 1.3, side="output", norm=norm)
    rd = O.update_from_bases(W.T, M.T, G.T, Q, 0.9, 0.05, 1.3, side="input", norm=norm)
    for key in ("M", "C", "S", "U", "W"):
        assert np.abs(rg[key] - rd[key].T).max() < 1e-12, key


def test_dobb_g_identity_basis_and_moments():
    rng = np.random.default_rng(63)
    m, n, B, N = 12, 7, 3, 50
    M, G, W = rng.standard_normal((3, m, n))
    I4 = np.broadcast_to(np.eye(4), (B, 4, 4)).copy()
    r = O.update_from_bases(W, M, G, I4, 0.5, 0.1, 1.0, side="output")
    assert np.array_equal(r["U"], np.sign(0.5 * M + G))
    # moments of the output gradients: blocks along m
    orc = O.DobbOracle([(m, n)], B, beta2=0.0, refresh_period=0, side="output")
    D = rng.standard_normal((N, m))
    orc.accumulate([D])
    for b in range(B):
        Db = D[:, b * 4:(b + 1) * 4]
        assert np.abs(orc.A[0][b] - Db.T @ Db / N).max() < 1e-12


# --------------------------------------------------------------------------
# Dobb-l2: column l2 normalisation ([Dobb, Tables 9 and 11])
# --------------------------------------------------------------------------

def test_l2_table9_norm_and_nonzero_columns():
    """[Dobb, Table 9]: Dobb-l2's raw update has ||O||_F^2 = n (O = U / sqrt(m));
    with zero columns in C only the nonzero ones count."""
    rng = np.random.default_rng(51)
    for (m, n, B) in ((40, 24, 3), (16, 48, 4)):
        M, G, W, Q = _rand_case(rng, m=m, n=n, B=B)
        U = O.update_from_bases(W, M, G, Q, 0.95, 1.0, 1.0, norm="l2")["U"]
        assert abs((U ** 2).sum() / m - n) < 1e-9 * n
        # a zero column of C (zero momentum column and Q = I) stays zero
        Q2 = np.broadcast_to(np.eye(n // B), (B, n // B, n // B)).copy()
        M2, G2 = M.copy(), G.copy()
        M2[:, 1] = 0.0
        G2[:, 1] = 0.0
        U2 = O.update_from_bases(W, M2, G2, Q2, 0.95, 1.0, 1.0, norm="l2")["U"]
        assert np.all(U2[:, 1] == 0.0) and abs((U2 ** 2).sum() / m - (n - 1)) < 1e-9 * n


def test_l2_identity_basis_closed_form_and_invariances():
    rng = np.random.default_rng(52)
    m, n, B = 20, 12, 3
    M, G, W, Q = _rand_case(rng, m=m, n=n, B=B)
    Mn = 0.9 * M + G
    I4 = np.broadcast_to(np.eye(4), (B, 4, 4)).copy()
    U = O.update_from_bases(W, M, G, I4, 0.9, 0.02, 1.0, norm="l2")["U"]
    assert np.abs(U - math.sqrt(m) * Mn / np.linalg.norm(Mn, axis=0)[None, :]).max() < 1e-12
    base = O.update_from_bases(W, M, G, Q, 0.9, 0.02, 1.0, norm="l2")["U"]
    Q2 = Q.copy()
    for b in range(B):
        Q2[b] = (Q[b] * rng.choice([-1.0, 1.0], size=4)[None, :])[:, rng.permutation(4)]
    assert np.abs(O.update_from_bases(W, M, G, Q2, 0.9, 0.02, 1.0, norm="l2")["U"] - base).max() < 1e-12
    assert np.abs(O.update_from_bases(W, 2.5 * M, 2.5 * G, Q, 0.9, 0.02, 1.0, norm="l2")["U"]
                  - base).max() < 1e-12


def test_l2_brute_force_tiny_step():
    rng = np.random.default_rng(53)
    m, n, B = 3, 4, 2
    k = n // B
    M, G, W, Q = _rand_case(rng, m=m, n=n, B=B)
    beta1, lr, s = 0.8, 0.1, 1.5
    W_exp = W.copy()
    for b in range(B):
        C = [[sum((beta1 * M[i, b * k + l] + G[i, b * k + l]) * Q[b, l, j] for l in range(k))
              for j in range(k)] for i in range(m)]
        nrm = [math.sqrt(sum(C[i][j] ** 2 for i in range(m))) for j in range(k)]
        for i in range(m):
            for l in range(k):
                u = sum(math.sqrt(m) * C[i][j] / nrm[j] * Q[b, l, j] for j in range(k))
                W_exp[i, b * k + l] -= lr * s * u
    r = O.update_from_bases(W, M, G, Q, beta1, lr, s, norm="l2")
    assert np.abs(r["W"] - W_exp).max() < 1e-12


# --------------------------------------------------------------------------
# orthogonal-iteration refresh ([Dobb, Table 15] principal, Table 16 Cholesky QR)
# --------------------------------------------------------------------------

def test_cholesky_qr_is_the_positive_diagonal_householder_qr():
    rng = np.random.default_rng(31)
    for k in (2, 5, 40):
        T = rng.standard_normal((k, k)) + 3 * np.eye(k)
        Q, R = O.cholesky_qr(T)
        Qh, Rh = np.linalg.qr(T)                    # Householder (LAPACK geqrf)
        d = np.sign(np.diag(Rh))
        Qh, Rh = Qh * d[None, :], Rh * d[:, None]
        assert np.abs(Q - Qh).max() < 1e-10 and np.abs(R - Rh).max() < 1e-10
        assert np.all(np.diag(R) > 0) and np.allclose(np.tril(R, -1), 0)


def test_cholesky_qr_two_by_two_by_hand():
    a, b, c, d = 3.0, 1.0, -2.0, 4.0
    T = np.array([[a, b], [c, d]])
    r11 = math.hypot(a, c)
    q1 = np.array([a, c]) / r11
    r12 = q1 @ np.array([b, d])
    w = np.array([b, d]) - r12 * q1
    r22 = np.linalg.norm(w)
    Q, R = O.cholesky_qr(T)
    assert np.allclose(Q[:, 0], q1, atol=1e-14) and np.allclose(Q[:, 1], w / r22, atol=1e-14)
    assert np.allclose(R, [[r11, r12], [0.0, r22]], atol=1e-14)


def test_orthogonal_iteration_fixed_point_and_convergence():
    rng = np.random.default_rng(32)
    k = 12
    A = np.stack([I.spd_with_gap(k, rng, cond=50.0)[0] for _ in range(2)])
    Qe, le = O.refresh_bases(A, "lapack")
    # exact eigenvectors (descending, PSD) are a fixed point, eigenvalues the quotients
    Q1, l1 = O.orthogonal_iteration(A, Qe, 1)
    assert np.abs(Q1 - Qe).max() < 1e-10 and np.abs(l1 - le).max() < 1e-10 * le.max()
    # from a generic start, many steps converge to the eigenvectors (up to sign)
    Q0 = np.stack([I.haar_orthogonal(k, rng) for _ in range(2)])
    Qn, ln = O.orthogonal_iteration(A, Q0, 3000)
    for b in range(2):
        assert np.abs(np.abs(Qn[b].T @ Qe[b]) - np.eye(k)).max() < 1e-8
        assert np.abs(ln[b] - le[b]).max() < 1e-10 * le[b].max()
    # one step is one QR of A Q0
    Qs, _ = O.orthogonal_iteration(A, Q0, 1)
    Qr, _ = O.cholesky_qr(0.5 * (A[0] + A[0].T) @ Q0[0])
    assert np.abs(Qs[0] - Qr).max() < 1e-14


# --------------------------------------------------------------------------
# bf16 basis storage ([Dobb, Table 18]: the principal precision setting)
# --------------------------------------------------------------------------

def test_bf16_basis_identity_and_invariances():
    rng = np.random.default_rng(41)
    M, G, W, Q = _rand_case(rng, m=20, n=12, B=3)
    # the identity is exact in bf16: U = sign(M) as with the fp32 basis
    I4 = np.broadcast_to(np.eye(4), (3, 4, 4)).copy()
    r = O.update_from_bases(W, M, G, I4, 0.95, 0.02, 1.0, basis_dtype="bf16")
    assert np.array_equal(r["U"], np.sign(0.95 * M + G))
    # column sign flips and permutations of Q_b still leave U unchanged
    base = O.update_from_bases(W, M, G, Q, 0.95, 0.02, 1.0, basis_dtype="bf16")["U"]
    Q2 = Q.copy()
    for b in range(3):
        Q2[b] = (Q[b] * rng.choice([-1.0, 1.0], size=4)[None, :])[:, rng.permutation(4)]
    U2 = O.update_from_bases(W, M, G, Q2, 0.95, 0.02, 1.0, basis_dtype="bf16")["U"]
    assert np.abs(U2 - base).max() < 1e-12


def test_bf16_basis_brute_force_with_torch_rounding():
    """Hand loops with the basis rounded by torch's bf16 conversion (Q chosen
    exactly representable in fp32, so torch's fp32 -> bf16 rounding is the
    single rounding the oracle applies)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(42)
    m, n, B = 3, 4, 2
    k = n // B
    M = rng.standard_normal((m, n))
    G = rng.standard_normal((m, n))
    W = rng.standard_normal((m, n))
    Q = np.stack([np.linalg.qr(rng.standard_normal((k, k)))[0] for _ in range(B)])
    Q = Q.astype(np.float32).astype(np.float64)
    Qb = torch.from_numpy(Q.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    beta1, lr, s = 0.9, 0.05, 2.0
    W_exp = np.zeros((m, n))
    for i in range(m):
        for b in range(B):
            cols = range(b * k, (b + 1) * k)
            mn = [beta1 * M[i, c] + G[i, c] for c in cols]
            sg = [math.copysign(1.0, sum(mn[l] * Qb[b, l, j] for l in range(k))) for j in range(k)]
            for l in range(k):
                u = sum(sg[j] * Qb[b, l, j] for j in range(k))
                W_exp[i, b * k + l] = W[i, b * k + l] - lr * s * u
    r = O.update_from_bases(W, M, G, Q, beta1, lr, s, basis_dtype="bf16")
    assert np.abs(r["W"] - W_exp).max() < 1e-12
    assert not np.array_equal(Qb, Q)  # the rounding did act


def test_bf16_basis_update_within_rounding_bound():
    """With the same signs, |U_bf16 - U_f32| <= ||S_b||_F ||bf16(Q_b) - Q_b||_2
    per block, and each basis entry moves by at most half a bf16 quantum,
    i.e. 2^-8 of its size (8 significant bits)."""
    rng = np.random.default_rng(43)
    M, G, W, Q = _rand_case(rng, m=40, n=24, B=3)
    r32 = O.update_from_bases(W, M, G, Q, 0.95, 0.02, 1.0)
    r16 = O.update_from_bases(W, M, G, Q, 0.95, 0.02, 1.0, S_override=r32["S"], basis_dtype="bf16")
    Qb = O.basis_for_update(Q, "bf16")
    assert np.all(np.abs(Qb - Q) <= 2.0 ** -8 * np.abs(Q))
    k = 8
    for b in range(3):
        sl = slice(b * k, (b + 1) * k)
        bound = np.linalg.norm(r32["S"][:, sl]) * np.linalg.norm(Qb[b] - Q[b], 2)
        assert np.linalg.norm(r16["U"][:, sl] - r32["U"][:, sl]) <= bound * (1 + 1e-12)
        assert np.linalg.norm(r16["U"][:, sl] - r32["U"][:, sl]) > 0


def test_ema_linearity_block_diagonal():
    """Block moments are the diagonal blocks of the full moment's EMA, and
    the EMA is linear (averaging replicas' EMAs = EMA of averaged moments)."""
    rng = np.random.default_rng(8)
    n, B, k = 12, 3, 4
    Xs = [rng.standard_normal((7, n)) for _ in range(4)]
    Ablk = np.zeros((B, k, k))
    Afull = np.zeros((1, n, n))
    for X in Xs:
        Ablk = O.block_moment_ema(Ablk, X, 0.9, B)
        Afull = O.block_moment_ema(Afull, X, 0.9, 1)
    for b in range(B):
        assert np.abs(Ablk[b] - Afull[0][b * k:(b + 1) * k, b * k:(b + 1) * k]).max() < 1e-14
    # explicit EMA sum
    ref = sum((1 - 0.9) * 0.9 ** (len(Xs) - 1 - i) * (X.T @ X) / 7 for i, X in enumerate(Xs))
    assert np.abs(Afull[0] - ref).max() < 1e-13
    # replica averaging commutes with the EMA
    r1 = [rng.standard_normal((7, n)) for _ in range(3)]
    r2 = [rng.standard_normal((7, n)) for _ in range(3)]
    A1 = np.zeros((B, k, k)); A2 = np.zeros((B, k, k)); Am = np.zeros((B, k, k))
    for x1, x2 in zip(r1, r2):
        A1 = O.block_moment_ema(A1, x1, 0.99, B)
        A2 = O.block_moment_ema(A2, x2, 0.99, B)
        Am = 0.99 * Am + 0.01 * 0.5 * (O.block_moment_ema(np.zeros((B, k, k)), x1, 0.0, B)
                                       + O.block_moment_ema(np.zeros((B, k, k)), x2, 0.0, B))
    assert np.abs(0.5 * (A1 + A2) - Am).max() < 1e-14


# --------------------------------------------------------------------------
# brute force: the whole step on a 3 x 4 matrix with B = 2 (k = 2)
# --------------------------------------------------------------------------

def _eig2_closed(a, c, d):
    """Eigenpairs of [[a, c], [c, d]] from the closed form (descending)."""
    mid, rad = (a + d) / 2.0, math.sqrt(((a - d) / 2.0) ** 2 + c * c)
    out = []
    for lam in (mid + rad, mid - rad):
        if abs(c) > 0:
            v = [c, lam - a]
        else:
            v = [1.0, 0.0] if abs(lam - a) <= abs(lam - d) else [0.0, 1.0]
        nrm = math.sqrt(v[0] ** 2 + v[1] ** 2)
        out.append((lam, [v[0] / nrm, v[1] / nrm]))
    return out


def brute_force_steps(Xs, Gs, W0, beta1, beta2, T, lr, s):
    """Pure-Python loops, closed-form 2x2 eigenvectors; m = 3, n = 4, B = 2."""
    m, n, B, k = 3, 4, 2, 2
    A = [[[0.0] * k for _ in range(k)] for _ in range(B)]
    Q = [[[1.0 if i == j else 0.0 for j in range(k)] for i in range(k)] for _ in range(B)]
    M = [[0.0] * n for _ in range(m)]
    W = [list(r) for r in W0]
    hist = []
    for t, (X, G) in enumerate(zip(Xs, Gs)):
        N = len(X)
        for b in range(B):
            for i in range(k):
                for j in range(k):
                    acc = 0.0
                    for tok in range(N):
                        acc += X[tok][b * k + i] * X[tok][b * k + j]
                    A[b][i][j] = beta2 * A[b][i][j] + (1 - beta2) * acc / N
        if T > 0 and t % T == 0:
            for b in range(B):
                pairs = _eig2_closed(A[b][0][0], A[b][0][1], A[b][1][1])
                for j, (_, v) in enumerate(pairs):
                    Q[b][0][j], Q[b][1][j] = v[0], v[1]
        for i in range(m):
            for j in range(n):
                M[i][j] = beta1 * M[i][j] + G[i][j]
        for i in range(m):
            for b in range(B):
                S = []
                for j in range(k):
                    c = sum(M[i][b * k + l] * Q[b][l][j] for l in range(k))
                    S.append(0.0 if c == 0 else math.copysign(1.0, c))
                for l in range(k):
                    u = sum(S[j] * Q[b][l][j] for j in range(k))
                    W[i][b * k + l] -= lr * s * u
        hist.append(([r[:] for r in M], [r[:] for r in W],
                     [[row[:] for row in A[b]] for b in range(B)]))
    return hist


def _tiny_inputs(seed=11, steps=4):
    rng = np.random.default_rng(seed)
    Xs = [rng.standard_normal((5, 4)) * np.array([3.0, 1.0, 0.5, 2.0]) for _ in range(steps)]
    Gs = [rng.standard_normal((3, 4)) for _ in range(steps)]
    W0 = rng.standard_normal((3, 4)) * 0.02
    return Xs, Gs, W0


def _run_oracle(Xs, Gs, W0, beta1, beta2, T, lr, s):
    orc = O.DobbOracle([(3, 4)], B=2, beta1=beta1, beta2=beta2, refresh_period=T,
                       scale_s=s, eig_method="jacobi")
    W = W0.copy()
    hist = []
    for X, G in zip(Xs, Gs):
        orc.accumulate([X])
        W = orc.step([W], [G], lr)[0]
        hist.append((orc.M[0].copy(), W.copy(), orc.A[0].copy()))
    return hist


def _max_diff(h1, h2):
    d = 0.0
    for (m1, w1, a1), (m2, w2, a2) in zip(h1, h2):
        for x, y in ((m1, m2), (w1, w2), (a1, a2)):
            d = max(d, np.abs(np.array(x) - np.array(y)).max())
    return d


@pytest.mark.parametrize("T", [1, 2, 0])
def test_brute_force_tiny_step(T):
    Xs, Gs, W0 = _tiny_inputs()
    bf = brute_force_steps(Xs, Gs, W0, 0.9, 0.95, T, 0.05, 1.3)
    orc = _run_oracle(Xs, Gs, W0, 0.9, 0.95, T, 0.05, 1.3)
    assert _max_diff(bf, orc) < 1e-12


# --------------------------------------------------------------------------
# planted mistakes in the oracle must be caught by the pins above
# --------------------------------------------------------------------------

def _blockwise(Mat, Q, fn):
    Mat = np.asarray(Mat, dtype=np.float64)
    Bn, k, _ = Q.shape
    out = np.empty_like(Mat)
    for b in range(Bn):
        out[:, b * k:(b + 1) * k] = fn(Mat[:, b * k:(b + 1) * k], Q[b])
    return out


def _mut_project_transposed(M, Q):
    return _blockwise(M, Q, lambda Mb, Qb: Mb @ Qb.T)


def _mut_reconstruct_untransposed(S, Q):
    return _blockwise(S, Q, lambda Sb, Qb: Sb @ Qb)


def _mut_ema_dropped_weight(A, X, beta2, B):
    X = np.asarray(X, dtype=np.float64)
    k = X.shape[1] // B
    return np.stack([beta2 * A[b] + X[:, b * k:(b + 1) * k].T @ X[:, b * k:(b + 1) * k] / len(X)
                     for b in range(B)])


def _mut_momentum_dampened(M, G, beta1):
    return beta1 * np.asarray(M, float) + (1 - beta1) * np.asarray(G, float)


def _mut_sign_flipped(C):
    return -np.sign(C)


@pytest.mark.parametrize("name,mutant", [
    ("project", _mut_project_transposed),
    ("reconstruct", _mut_reconstruct_untransposed),
    ("block_moment_ema", _mut_ema_dropped_weight),
    ("momentum", _mut_momentum_dampened),
    ("sign", _mut_sign_flipped),
])
def test_planted_mistakes_are_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(O, name, mutant)
    Xs, Gs, W0 = _tiny_inputs()
    bf = brute_force_steps(Xs, Gs, W0, 0.9, 0.95, 1, 0.05, 1.3)
    orc = _run_oracle(Xs, Gs, W0, 0.9, 0.95, 1, 0.05, 1.3)
    assert _max_diff(bf, orc) > 1e-6


# --------------------------------------------------------------------------
# Table 1 direction: sign normalisation in the block eigenbasis raises the
# orthogonality of low-effective-rank updates
# --------------------------------------------------------------------------

@pytest.mark.parametrize("B", [1, 4])
def test_sign_normalisation_raises_orthogonality(B):
    rng = np.random.default_rng(20 + B)
    n, N = 128, 512
    X = I.activations(N, n, 0.15, rng).astype(np.float64)
    G = I.gradients(96, X, rng).astype(np.float64)
    A = O.block_moment_ema(np.zeros((B, n // B, n // B)), X, 0.0, B)
    Q, _ = O.refresh_bases(A, "lapack")
    r = O.update_from_bases(np.zeros_like(G), np.zeros_like(G), G, Q, 0.95, 1.0, 1.0)
    assert MX.orthogonality(r["U"]) > MX.orthogonality(G) + 0.1


# --------------------------------------------------------------------------
# rounding and parity rules
# --------------------------------------------------------------------------

def test_round_to_bf16_matches_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_to_bf16(x.astype(np.float64)), ref)
    # ties go to even
    one = 1.0
    assert O.round_to_bf16(np.array([one + 2.0 ** -8]))[0] == 1.0
    assert O.round_to_bf16(np.array([one + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
    # double rounding through fp32 would differ here: fp64 just above a midpoint
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert O.round_to_bf16(np.array([v]))[0] == 1.0 + 2.0 ** -7


def test_parity_rules_detect_planted_errors():
    rng = np.random.default_rng(12)
    C = rng.standard_normal((64, 32))
    S = np.sign(C)
    assert MX.sign_agreement(C, S, 8)["disagree"] == 0
    S2 = S.copy()
    S2[3, 5] *= -1
    res = MX.sign_agreement(C, S2, 8)
    assert res["disagree"] == 1 and res["outside_band"] == 1
    C3 = C.copy()
    C3[3, 5] = 1e-9
    res = MX.sign_agreement(C3, S2 * 0 + np.sign(C3) * np.where(np.arange(C3.size).reshape(C3.shape) == 3 * 32 + 5, -1, 1), 8)
    assert res["disagree"] == 1 and res["outside_band"] == 0
    W = rng.standard_normal((50, 50)) * 0.02
    Wb = O.round_to_bf16(W)
    assert MX.bf16_parity(Wb, W)["violations"] == 0
    Wbad = Wb.copy()
    Wbad[0, 0] = O.round_to_bf16(np.array([Wb[0, 0] * (1 + 2 ** -6)]))[0]
    assert MX.bf16_parity(Wbad, W)["violations"] == 1
    # a value whose exact result sits on a rounding midpoint may round either way
    x = np.array([1.0 + 2.0 ** -8, 0.5])
    assert MX.bf16_parity(np.array([1.0 + 2.0 ** -7, 0.5]), x)["violations"] == 0
    assert MX.bf16_parity(np.array([1.0, 0.5]), x)["violations"] == 0
    # tiny entries: any value reachable from within the normwise band is accepted
    y = np.array([1e-6, 0.08])
    ok = O.round_to_bf16(np.array([1e-6 + 5e-7, 0.08]))
    assert MX.bf16_parity(ok, y)["violations"] == 0
    bad = O.round_to_bf16(np.array([1e-6 + 2e-6, 0.08]))
    assert MX.bf16_parity(bad, y)["violations"] == 1
    assert MX.w_rel_error(W, W) == 0.0


# --------------------------------------------------------------------------
# input generators produce what they claim (checked with the oracle metric)
# --------------------------------------------------------------------------

def test_generators_hit_target_effective_rank():
    for n, tgt in ((768, 0.15), (768, 0.20), (400, 0.40)):
        lam = I.geometric_spectrum(n, tgt)
        assert abs(MX.effective_rank(lam) - tgt) < 1e-9
    rng = np.random.default_rng(13)
    Q = I.haar_orthogonal(64, rng)
    assert np.abs(Q.T @ Q - np.eye(64)).max() < 1e-12
    a, lam, q = I.spd_with_gap(200, rng, cond=1e6)
    gaps = -np.diff(lam) / lam[:-1]
    assert gaps.min() >= 1e-3 and abs(lam[0] / lam[-1] - 1e6) < 1e-3 * 1e6
    assert MX.eig_residuals(a, q, lam)["residual"] < 1e-12


# --------------------------------------------------------------------------
# the parity rules themselves, pinned by hand-computed values
# --------------------------------------------------------------------------

def test_w_rel_error_reports_known_offsets():
    """max_ij |W_test - W_ref| / max_ij |W_ref|: the largest offset (not the
    sum or the mean), over the largest |entry| of the reference (not of the
    tested matrix, not a Frobenius norm, with the sign of the entry dropped)."""
    W = np.array([[2.0, -3.0], [1.0, 0.0]])
    one = W.copy()
    one[1, 1] += 0.006
    assert MX.w_rel_error(one, W) == pytest.approx(0.002, rel=1e-12)
    two = W.copy()
    two[0, 0] += 0.003
    two[1, 0] -= 0.0015
    assert MX.w_rel_error(two, W) == pytest.approx(0.001, rel=1e-12)       # max, not sum / mean
    at_max = W.copy()
    at_max[0, 1] -= 0.3                                                      # |W_test| max 3.3
    assert MX.w_rel_error(at_max, W) == pytest.approx(0.1, rel=1e-12)       # reference's max
    assert MX.w_rel_error(-W, -W) == 0.0
    neg = -W
    neg[0, 0] += 0.03
    assert MX.w_rel_error(neg, -W) == pytest.approx(0.01, rel=1e-12)
    # homogeneous of degree 0: scaling both sides leaves it unchanged
    assert MX.w_rel_error(7.0 * one, 7.0 * W) == pytest.approx(0.002, rel=1e-12)


def test_eig_residuals_closed_forms_flag_wrong_decompositions():
    """Hand-derived residuals of wrong decompositions of A = diag(l1, l2):
    a basis rotated by theta gives ||AQ - Q Lambda||_F = ||Q Lambda Q^T - A||_F
    = sqrt(2) |l1 - l2| |sin theta| and zero orthogonality error; permuted
    eigenvalues, a scaled column and a sheared basis each move the residual
    they must move, by the amount computed by hand."""
    l1, l2 = 3.0, 1.0
    A = np.diag([l1, l2])
    fro = math.sqrt(l1 ** 2 + l2 ** 2)
    exact = MX.eig_residuals(A, np.eye(2), np.array([l1, l2]))
    assert exact == {"residual": 0.0, "orth": 0.0, "recon": 0.0}
    th = 0.01
    c, s = math.cos(th), math.sin(th)
    Qr = np.array([[c, -s], [s, c]])
    r = MX.eig_residuals(A, Qr, np.array([l1, l2]))
    want = math.sqrt(2) * abs(l1 - l2) * abs(s) / fro
    assert r["residual"] == pytest.approx(want, rel=1e-9)
    assert r["recon"] == pytest.approx(want, rel=1e-9)
    assert r["orth"] < 1e-15
    # permuted eigenvalues, exact basis
    A3 = np.diag([1.0, 2.0, 3.0])
    r = MX.eig_residuals(A3, np.eye(3), np.array([2.0, 1.0, 3.0]))
    assert r["residual"] == pytest.approx(math.sqrt(2) / math.sqrt(14), rel=1e-12)
    assert r["recon"] == pytest.approx(math.sqrt(2) / math.sqrt(14), rel=1e-12)
    assert r["orth"] == 0.0
    # a column scaled by (1 + e): orthogonality error 2e + e^2, reconstruction l1 (2e + e^2)
    e = 1e-3
    Qs = np.diag([1.0 + e, 1.0])
    r = MX.eig_residuals(A, Qs, np.array([l1, l2]))
    assert r["orth"] == pytest.approx(2 * e + e * e, rel=1e-9)
    assert r["recon"] == pytest.approx(l1 * (2 * e + e * e) / fro, rel=1e-9)
    assert r["residual"] == 0.0
    # a sheared basis: Q^T Q - I = [[0, d], [d, d^2]]
    d = 1e-2
    Qh = np.array([[1.0, d], [0.0, 1.0]])
    r = MX.eig_residuals(A, Qh, np.array([l1, l2]))
    assert r["orth"] == pytest.approx(math.sqrt(2 * d * d + d ** 4), rel=1e-9)
    # || A Q - Q Lambda || = || [[0, (l1 - l2) d], [0, 0]] ||
    assert r["residual"] == pytest.approx(abs(l1 - l2) * d / fro, rel=1e-9)
    # scale invariance of the relative residuals; orth does not see A at all
    r10 = MX.eig_residuals(10 * A, Qr, 10 * np.array([l1, l2]))
    assert r10["residual"] == pytest.approx(math.sqrt(2) * abs(l1 - l2) * abs(s) / fro, rel=1e-9)
    # a random exact decomposition passes, a perturbed one fails in proportion
    rng = np.random.default_rng(5)
    a, lam, q = I.spd_with_gap(40, rng, cond=1e3)
    assert MX.eig_residuals(a, q, lam)["residual"] < 1e-13
    qp = q.copy()
    qp[:, 7] += 1e-4 * q[:, 8]
    rp = MX.eig_residuals(a, qp, lam)
    assert rp["residual"] == pytest.approx(1e-4 * abs(lam[8] - lam[7]) / np.linalg.norm(a), rel=1e-6)
    assert rp["orth"] == pytest.approx(1e-4 * math.sqrt(2 + 1e-8), rel=1e-6)


def test_l2_entrywise_bound_holds_for_fp32_and_catches_a_planted_error():
    """The per-entry Dobb-l2 tolerance of the GPU tests is derived from fp32
    arithmetic: an fp32 evaluation of the update (numpy float32, a different
    summation order than the GPU's) lies inside it, and one entry moved by
    1 % of the update's RMS does not."""
    import parity_util as PU
    rng = np.random.default_rng(41)
    m, n, B = 300, 192, 2
    k = n // B
    X = I.activations(4 * k, n, 0.3, rng)
    A = O.block_moment_ema(np.zeros((B, k, k)), X, 0.0, B)
    Q, _ = O.refresh_bases(A, "lapack")
    W = I.weights(m, n, rng)
    G = I.gradients(m, X, rng)
    lr, s = 0.02, 1.5
    ref = O.update_from_bases(W, np.zeros((m, n)), G, Q, 0.9, lr, s, "f32", norm="l2")
    # fp32 evaluation
    M32 = (np.float32(0.9) * np.zeros((m, n), np.float32) + G.astype(np.float32))
    W32 = W.astype(np.float32).copy()
    for b in range(B):
        sl = slice(b * k, (b + 1) * k)
        Q32 = Q[b].astype(np.float32)
        C = M32[:, sl] @ Q32
        nrm = np.sqrt((C * C).sum(axis=0, dtype=np.float32))
        S = C * (np.float32(math.sqrt(m)) / nrm)[None, :]
        W32[:, sl] = W32[:, sl] - np.float32(lr * s) * (S @ Q32.T)
    W64 = W32.astype(np.float64)
    err, bmax = PU.check_update_l2(W, np.zeros((m, n)), G, Q, W64, M32.astype(np.float64), 0.9, lr,
                                   s, "f32")
    assert 0 < err <= bmax
    # the worst-case bound sits near 2.5e-3 of the update's RMS here: a 1 %
    # error in one entry is caught
    bad = W64.copy()
    bad[17, 40] += 1e-2 * lr * s * math.sqrt((ref["U"] ** 2).mean())
    with pytest.raises(AssertionError):
        PU.check_update_l2(W, np.zeros((m, n)), G, Q, bad, M32.astype(np.float64), 0.9, lr, s, "f32")
    # bf16 parameters: the rounded fp32 result passes, one bf16 ulp off does not
    Wb = O.round_to_bf16(W)
    ref_b = O.update_from_bases(Wb, np.zeros((m, n)), G, Q, 0.9, lr, s, "f32", norm="l2")
    out = O.round_to_bf16(Wb + (W64 - W.astype(np.float32).astype(np.float64)))
    PU.check_update_l2(Wb, np.zeros((m, n)), G, Q, out, M32.astype(np.float64), 0.9, lr, s, "bf16")
    worse = out.copy()
    worse[3, 5] = O.round_to_bf16(np.array([out[3, 5] * (1 + 2 ** -6)]))[0]
    with pytest.raises(AssertionError):
        PU.check_update_l2(Wb, np.zeros((m, n)), G, Q, worse, M32.astype(np.float64), 0.9, lr, s,
                           "bf16")
    assert ref_b["W"].shape == (m, n)
