"""Plain fp64 CPU oracle of one Dobb optimizer step.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  Shares no code with
the CUDA implementation.

Source.  "Dobb: Shard-Local Preconditioning in Block-Diagonal Eigenbases"
(arXiv 2610.39412; abstract on paperdot.bitmofang.com and fugumt.com, tables
on thelatestinai.com).  Cited below as [Dobb, <section>].  The pages give the
method only in words (Abstract) and through table captions; the step written
out here is:

  per weight matrix W (m x n, y = W x, [Dobb, Table 6 notation]), n split into
  B column blocks of width k = n / B:
    A_b <- beta2 A_b + (1 - beta2) X_b^T X_b / N        (block second moment)
    every T steps: Q_b, Lambda_b with A_b = Q_b Lambda_b Q_b^T   (complete basis)
    M   <- beta1 M + G                                 (momentum)
    C_b  = M_b Q_b ; S_b = sign(C_b) ; U_b = S_b Q_b^T  (project, sign, reconstruct)
    W   <- W - lr * s * U

  [Dobb, Abstract]: "approximates the input-activation second moment with
  diagonal blocks and tracks a complete basis within each block ... projects
  momentum into these bases, applies sign normalization to the coefficients,
  and reconstructs the update".  [Dobb, Table 3 caption]: n^2/B second-moment
  entries per matrix.  [Dobb, Table 13]: the l_inf (sign) normalisation in the
  activation second-moment basis is Dobb.  [Dobb, Table 15]: the exact
  eigendecomposition refresh.  [Dobb, Table 21 footnote a]: the moment
  reduction runs behind the backward pass and the refresh inside the optimizer
  call, so the order within a step is accumulate -> refresh (if due) -> update.

Readings where the pages are silent (each one is also listed in the design
notes of the repository):
  * t counts steps from 0; the basis is refreshed when t % T == 0, after that
    step's moments were accumulated; T == 0 means "never automatically".
  * A starts at 0, Q at I, M at 0; no bias correction and no momentum
    dampening (sign and eigenvectors are invariant to positive scaling).
  * sign(0) = 0.
  * bf16 parameters: the fp64 result is rounded once to bf16, nearest-even.

Pins (tests/test_oracle_*.py): the 2x2 closed form and brute-force
characteristic-polynomial roots (k <= 4) pin `jacobi_eigh`; LAPACK agreement,
orthogonality and residuals pin both eigen routes; Q = I gives U = sign(M);
||U_b||_F^2 = nnz(S_b); invariance under column sign flips / permutations of
Q_b and positive scaling of M; EMA linearity; a pure-Python brute-force step
on a 3 x 4 matrix with B = 2 (k = 2, closed-form eigenvectors) pins the whole
update including operand orientation.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "block_width",
    "block_moment_ema",
    "sym_schur2",
    "jacobi_eigh",
    "lapack_eigh",
    "canonicalize",
    "refresh_bases",
    "cholesky_qr",
    "orthogonal_iteration",
    "momentum",
    "project",
    "sign",
    "reconstruct",
    "l2_normalize_columns",
    "project_left",
    "reconstruct_left",
    "normalize",
    "apply_update",
    "round_to_bf16",
    "basis_for_update",
    "update_from_bases",
    "DobbOracle",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def block_width(n: int, B: int) -> int:
    """k = n / B; the input axis must split evenly ([Dobb, Table 3 caption])."""
    if B <= 0 or n % B != 0:
        raise ValueError(f"n={n} is not divisible by B={B}")
    return n // B


# ---------------------------------------------------------------------------
# (1) block second moment with EMA          [Dobb, Abstract; Table 3 caption]
# ---------------------------------------------------------------------------

def block_moment_ema(A: np.ndarray, X: np.ndarray, beta2: float, B: int) -> np.ndarray:
    """A has shape (B, k, k); X is N x n (tokens x input features).
    Returns A_b <- beta2 A_b + (1 - beta2) X_b^T X_b / N for every block."""
    X = _f64(X)
    N, n = X.shape
    k = block_width(n, B)
    out = np.empty((B, k, k), dtype=np.float64)
    for b in range(B):
        Xb = X[:, b * k:(b + 1) * k]
        out[b] = beta2 * _f64(A[b]) + (1.0 - beta2) * (Xb.T @ Xb) / N
    return out


# ---------------------------------------------------------------------------
# (2) exact eigendecomposition of each block               [Dobb, Table 15]
# ---------------------------------------------------------------------------

def sym_schur2(A: np.ndarray, p: int, q: int) -> Tuple[float, float]:
    """Cosine/sine of the Jacobi rotation J(p, q) that zeroes B[p, q] of
    B = J^T A J (Golub & Van Loan, Matrix Computations, 2x2 symmetric Schur
    decomposition).  J has J[p,p] = J[q,q] = c, J[p,q] = s, J[q,p] = -s."""
    apq = A[p, q]
    if apq == 0.0:
        return 1.0, 0.0
    tau = (A[q, q] - A[p, p]) / (2.0 * apq)
    if tau >= 0.0:
        t = 1.0 / (tau + math.sqrt(1.0 + tau * tau))
    else:
        t = -1.0 / (-tau + math.sqrt(1.0 + tau * tau))
    c = 1.0 / math.sqrt(1.0 + t * t)
    return c, t * c


def _off(A: np.ndarray) -> float:
    """Frobenius norm of the off-diagonal part, summed directly (the
    difference ||A||_F^2 - ||diag A||^2 cancels catastrophically)."""
    return float(np.linalg.norm(A - np.diag(np.diag(A))))


def jacobi_eigh(A: np.ndarray, tol: float = 1e-15, max_sweeps: int = 60):
    """Cyclic-by-row Jacobi (Golub & Van Loan, "Jacobi methods") in fp64.

    Sweeps over every pair p < q in row order, applying the rotation from
    `sym_schur2` to A (both sides) and accumulating V, until
    off(A) <= tol * ||A||_F.  Returns (eigenvalues, V, sweeps) unsorted."""
    A = _f64(A).copy()
    n = A.shape[0]
    V = np.eye(n)
    fro = math.sqrt(float((A * A).sum()))
    sweeps = 0
    while sweeps < max_sweeps and _off(A) > tol * fro:
        sweeps += 1
        for p in range(n - 1):
            for q in range(p + 1, n):
                c, s = sym_schur2(A, p, q)
                if s == 0.0:
                    continue
                # A <- J^T A J, J = identity except the (p, q) 2x2 rotation
                ap, aq = A[p, :].copy(), A[q, :].copy()
                A[p, :] = c * ap - s * aq
                A[q, :] = s * ap + c * aq
                ap, aq = A[:, p].copy(), A[:, q].copy()
                A[:, p] = c * ap - s * aq
                A[:, q] = s * ap + c * aq
                vp, vq = V[:, p].copy(), V[:, q].copy()
                V[:, p] = c * vp - s * vq
                V[:, q] = s * vp + c * vq
    return np.diag(A).copy(), V, sweeps


def lapack_eigh(A: np.ndarray):
    """LAPACK symmetric eigensolver (numpy.linalg.eigh), used to cross-check
    `jacobi_eigh` and for blocks too large for the Python-loop Jacobi."""
    lam, V = np.linalg.eigh(_f64(A))
    return lam, V


def canonicalize(lam: np.ndarray, V: np.ndarray):
    """Sort eigenpairs by descending eigenvalue and flip each eigenvector so
    that its largest-magnitude entry is positive.  U is invariant to both
    choices, so this only makes the oracle's own output deterministic."""
    order = np.argsort(-lam, kind="stable")
    lam = lam[order]
    V = V[:, order].copy()
    idx = np.argmax(np.abs(V), axis=0)
    sgn = np.sign(V[idx, np.arange(V.shape[1])])
    sgn[sgn == 0] = 1.0
    return lam, V * sgn[None, :]


def refresh_bases(A: np.ndarray, method: str = "auto", jacobi_max_k: int = 48):
    """Complete orthonormal eigenbasis of every block: A has shape (B, k, k);
    returns Q (B, k, k) with column j the j-th eigenvector (descending
    eigenvalue) and Lambda (B, k)."""
    A = _f64(A)
    Bn, k, _ = A.shape
    Q = np.empty_like(A)
    lam = np.empty((Bn, k))
    for b in range(Bn):
        Ab = 0.5 * (A[b] + A[b].T)
        use_jacobi = method == "jacobi" or (method == "auto" and k <= jacobi_max_k)
        if use_jacobi:
            l, V, _ = jacobi_eigh(Ab)
        else:
            l, V = lapack_eigh(Ab)
        lam[b], Q[b] = canonicalize(l, V)
    return Q, lam


def cholesky_qr(T: np.ndarray):
    """QR factorisation through the Gram matrix ([Dobb, Table 16]: the
    "Cholesky" QR routine): R = chol(T^T T) upper triangular with positive
    diagonal, Q = T R^{-1}.  Mathematically the QR factorisation of T whose R
    has a positive diagonal."""
    T = _f64(T)
    L = np.linalg.cholesky(T.T @ T)          # T^T T = L L^T, L lower
    Q = np.linalg.solve(L, T.T).T            # Q^T = L^{-1} T^T
    return Q, L.T


def orthogonal_iteration(A: np.ndarray, Q0: np.ndarray, steps: int = 1):
    """Refresh by orthogonal (subspace) iteration started from the current
    basis ([Dobb, Table 15]: "k = 1" orthogonal-iteration steps per refresh is
    the principal setting; Table 16: Cholesky QR).  For every block,
    `steps` times: T = A_b Q_b, Q_b = T R^{-1} with R = chol(T^T T).
    Returns Q (B, k, k) and the Rayleigh quotients diag(Q_b^T A_b Q_b)."""
    A = _f64(A)
    Q = _f64(Q0).copy()
    Bn, k, _ = A.shape
    lam = np.empty((Bn, k))
    for b in range(Bn):
        Ab = 0.5 * (A[b] + A[b].T)
        for _ in range(steps):
            Q[b], _ = cholesky_qr(Ab @ Q[b])
        lam[b] = np.einsum("ij,ij->j", Q[b], Ab @ Q[b])
    return Q, lam


# ---------------------------------------------------------------------------
# (3) momentum, project, sign, reconstruct, apply   [Dobb, Abstract; Table 9]
# ---------------------------------------------------------------------------

def momentum(M: np.ndarray, G: np.ndarray, beta1: float) -> np.ndarray:
    """M <- beta1 M + G (no dampening; Nesterov off, [Dobb, Table 19])."""
    return beta1 * _f64(M) + _f64(G)


def project(M: np.ndarray, Q: np.ndarray) -> np.ndarray:
    """C_b = M_b Q_b for every column block b: coefficients of the momentum
    rows in the block eigenbasis.  M is m x n, Q is (B, k, k)."""
    M = _f64(M)
    Bn, k, _ = Q.shape
    C = np.empty_like(M)
    for b in range(Bn):
        C[:, b * k:(b + 1) * k] = M[:, b * k:(b + 1) * k] @ _f64(Q[b])
    return C


def sign(C: np.ndarray) -> np.ndarray:
    """l_inf normalisation of the coefficients, sign(0) = 0 ([Dobb, Table 13])."""
    return np.sign(_f64(C))


def l2_normalize_columns(C: np.ndarray) -> np.ndarray:
    """Column l2 normalisation of the coefficients, "Dobb-l2" ([Dobb, Table 11];
    Table 9 gives its raw update the same ||O||_F^2 = n as Dobb's sign).  Each
    column of C (over all m rows) is scaled to l2 norm sqrt(m), so that with
    O = U / sqrt(m) as for the sign update every nonzero column of O has unit
    norm; a zero column stays zero."""
    C = _f64(C)
    m = C.shape[0]
    nrm = np.sqrt((C ** 2).sum(axis=0))
    scale = np.where(nrm > 0, math.sqrt(m) / np.where(nrm > 0, nrm, 1.0), 0.0)
    return C * scale[None, :]


def normalize(C: np.ndarray, norm: str = "sign") -> np.ndarray:
    """The coefficient normalisation: "sign" (Dobb, l_inf) or "l2" (Dobb-l2)."""
    if norm == "sign":
        return sign(C)
    if norm == "l2":
        return l2_normalize_columns(C)
    raise ValueError(f"norm {norm!r}")


def reconstruct(S: np.ndarray, Q: np.ndarray) -> np.ndarray:
    """U_b = S_b Q_b^T: map the normalised coefficients back to the input
    axis; U = [U_1 ... U_B] along the columns."""
    S = _f64(S)
    Bn, k, _ = Q.shape
    U = np.empty_like(S)
    for b in range(Bn):
        U[:, b * k:(b + 1) * k] = S[:, b * k:(b + 1) * k] @ _f64(Q[b]).T
    return U


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bfloat16 (8 significant bits, fp32 exponent
    range), nearest with ties to even, in one rounding; returns fp64."""
    x = _f64(x)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0.0)
    _, e = np.frexp(x[fin])                 # x = f * 2**e, 0.5 <= |f| < 1
    qexp = np.maximum(e - 8, -133)          # quantum 2**(e-8); subnormal floor
    r = np.rint(np.ldexp(x[fin], -qexp))    # round half to even
    vals = np.ldexp(r, qexp)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    vals[np.abs(vals) > bf16_max] = np.copysign(np.inf, vals[np.abs(vals) > bf16_max])
    out[fin] = vals
    return out


def apply_update(W: np.ndarray, U: np.ndarray, lr: float, s: float,
                 param_dtype: str = "f32") -> np.ndarray:
    """W <- W - lr * s * U.  With bf16 parameters the exact result is rounded
    once to bf16 (the parameter storage format)."""
    out = _f64(W) - lr * s * _f64(U)
    if param_dtype == "bf16":
        out = round_to_bf16(out)
    return out


def basis_for_update(Q: np.ndarray, basis_dtype: str = "f32") -> np.ndarray:
    """The block bases the update multiplies with.  "bf16": the stored basis
    is bfloat16 ([Dobb, Table 18]: fp32 moment accumulation with a bf16
    basis is the principal setting, 6 n^2 / B bytes per matrix), i.e. every
    entry of Q rounded once to bf16; the products themselves stay exact here.
    "f32": Q as given."""
    if basis_dtype == "bf16":
        return round_to_bf16(Q)
    if basis_dtype != "f32":
        raise ValueError(f"basis_dtype {basis_dtype!r}")
    return _f64(Q)


def project_left(M: np.ndarray, Q: np.ndarray) -> np.ndarray:
    """Output-gradient side ("Dobb-G", [Dobb, Tables 12-13]): C_b = Q_b^T M_b
    for every row block b (k = m / B rows): coefficients of the momentum
    columns in the block eigenbasis of the output-gradient second moment."""
    M = _f64(M)
    Bn, k, _ = Q.shape
    C = np.empty_like(M)
    for b in range(Bn):
        C[b * k:(b + 1) * k, :] = _f64(Q[b]).T @ M[b * k:(b + 1) * k, :]
    return C


def reconstruct_left(S: np.ndarray, Q: np.ndarray) -> np.ndarray:
    """U_b = Q_b S_b for every row block b (the mirror of `reconstruct`)."""
    S = _f64(S)
    Bn, k, _ = Q.shape
    U = np.empty_like(S)
    for b in range(Bn):
        U[b * k:(b + 1) * k, :] = _f64(Q[b]) @ S[b * k:(b + 1) * k, :]
    return U


def update_from_bases(W, M, G, Q, beta1: float, lr: float, s: float,
                      param_dtype: str = "f32", S_override: Optional[np.ndarray] = None,
                      basis_dtype: str = "f32", norm: str = "sign", side: str = "input"):
    """One update of a single matrix with given block bases Q (B, k, k).
    Returns dict with the new M, C, S, U and W.  `S_override` substitutes a
    given sign matrix (used to score a second implementation's signs at the
    entries where the sign is numerically undetermined).  `basis_dtype`
    selects the stored precision of the basis (see `basis_for_update`), `norm`
    the coefficient normalisation (see `normalize`), `side` the axis the
    blocks and bases live on: "input" (Dobb: column blocks, bases of the
    activation second moment) or "output" (Dobb-G: row blocks, bases of the
    output-gradient second moment, applied from the left; the normalisation
    then runs over the rows of C^T, i.e. the columns of the transposed
    problem)."""
    Qu = basis_for_update(Q, basis_dtype)
    Mn = momentum(M, G, beta1)
    if side == "output":
        C = project_left(Mn, Qu)
        S = normalize(C.T, norm).T if S_override is None else _f64(S_override)
        U = reconstruct_left(S, Qu)
    elif side == "input":
        C = project(Mn, Qu)
        S = normalize(C, norm) if S_override is None else _f64(S_override)
        U = reconstruct(S, Qu)
    else:
        raise ValueError(f"side {side!r}")
    Wn = apply_update(W, U, lr, s, param_dtype)
    return {"M": Mn, "C": C, "S": S, "U": U, "W": Wn}


# ---------------------------------------------------------------------------
# the stateful optimizer (all matrices of a model)
# ---------------------------------------------------------------------------

@dataclass
class DobbOracle:
    """State and schedule of the optimizer over a list of matrices.

    shapes: list of (m, n); B blocks per matrix; beta1, beta2; refresh period
    T (0 = never automatic); update scale s; parameter dtype "f32" / "bf16".
    """
    shapes: Sequence[Tuple[int, int]]
    B: int
    beta1: float = 0.95
    beta2: float = 0.99
    refresh_period: int = 10
    scale_s: float = 1.0
    param_dtype: str = "f32"
    eig_method: str = "auto"
    basis_dtype: str = "f32"
    refresh_method: str = "eigh"   # "eigh" (exact) or "orth" (orthogonal iteration)
    orth_steps: int = 1
    norm: str = "sign"             # "sign" (Dobb) or "l2" (Dobb-l2)
    side: str = "input"            # "input" (Dobb) or "output" (Dobb-G)

    def __post_init__(self):
        self.t = 0
        self.A: List[np.ndarray] = []
        self.Q: List[np.ndarray] = []
        self.lam: List[np.ndarray] = []
        self.M: List[np.ndarray] = []
        for (m, n) in self.shapes:
            k = block_width(m if self.side == "output" else n, self.B)
            self.A.append(np.zeros((self.B, k, k)))
            self.Q.append(np.broadcast_to(np.eye(k), (self.B, k, k)).copy())
            self.lam.append(np.zeros((self.B, k)))
            self.M.append(np.zeros((m, n)))

    def accumulate(self, X_list: Sequence[np.ndarray]) -> None:
        """X: input activations (N x n), or for side "output" the output
        gradients (N x m)."""
        for i, X in enumerate(X_list):
            if X is None:
                continue
            self.A[i] = block_moment_ema(self.A[i], X, self.beta2, self.B)

    def refresh(self) -> None:
        for i in range(len(self.shapes)):
            if self.refresh_method == "orth":
                self.Q[i], self.lam[i] = orthogonal_iteration(self.A[i], self.Q[i], self.orth_steps)
            else:
                self.Q[i], self.lam[i] = refresh_bases(self.A[i], self.eig_method)

    def step(self, W_list, G_list, lr: float, keep_parts: bool = False):
        """Refresh if due, then update every matrix.  Returns the new W list
        (and the per-matrix parts when keep_parts)."""
        if self.refresh_period > 0 and self.t % self.refresh_period == 0:
            self.refresh()
        out_W, parts = [], []
        for i, (W, G) in enumerate(zip(W_list, G_list)):
            r = update_from_bases(W, self.M[i], G, self.Q[i], self.beta1, lr,
                                  self.scale_s, self.param_dtype, basis_dtype=self.basis_dtype,
                                  norm=self.norm, side=self.side)
            self.M[i] = r["M"]
            out_W.append(r["W"])
            if keep_parts:
                parts.append(r)
        self.t += 1
        return (out_W, parts) if keep_parts else out_W
