"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the
same seeded inputs, phase by phase and over whole multi-step runs."""
import math

import numpy as np
import pytest
import torch

from block_eigenbasis_preconditioning_gb300 import inputs as I
from oracle import dobb as O
from oracle import metrics as MX

from parity_util import (TOL_A, check_bases, check_moments, check_update, check_update_l2,
                         make_output_side_problem, make_problem, to_dev, to_np)

pytestmark = pytest.mark.gpu


def _dobb(*a, **k):
    from block_eigenbasis_preconditioning_gb300 import Dobb
    return Dobb(*a, **k)


# --------------------------------------------------------------------------
# (a1) block moments
# --------------------------------------------------------------------------

@pytest.mark.parametrize("act", ["f32", "bf16"])
@pytest.mark.parametrize("shapes,B,N", [
    ([(24, 96), (33, 64)], 2, 100),      # k = 48 / 32, ragged token tail
    ([(8, 130)], 2, 37),                 # k = 65: crosses one 64 tile
    ([(5, 7)], 7, 3),                    # k = 1
    ([(40, 400)], 1, 70),                # k = 400: 7 x 7 tiles
    ([(16, 392), (12, 600)], 2, 300),    # k = 196 / 300, odd blocks 4 columns off: 2-3 slices
    ([(24, 384)], 2, 200),               # k = 192 alone: two slices in one unit, two accumulators
])
def test_moments_match_oracle(act, shapes, B, N):
    Xs, _, _ = make_problem(shapes, N, 0.3, seed=1, act_dtype=act)
    opt = _dobb(shapes, B, beta2=0.9, refresh_period=0, act_dtype=act)
    orc = O.DobbOracle(shapes, B, beta2=0.9, refresh_period=0)
    for rep in range(3):
        Xd = [to_dev(x, act) for x in Xs]
        opt.accumulate(Xd)
        orc.accumulate(Xs)
        torch.cuda.synchronize()
        check_moments(opt, orc)
        Xs = [x[::-1].copy() for x in Xs]


def test_moments_skip_null_and_flag_nonfinite():
    shapes = [(8, 32), (8, 32)]
    Xs, _, _ = make_problem(shapes, 16, 0.5, seed=2)
    opt = _dobb(shapes, 2, refresh_period=0)
    orc = O.DobbOracle(shapes, 2, refresh_period=0)
    opt.accumulate([to_dev(Xs[0], "f32"), None])
    orc.accumulate([Xs[0], None])
    check_moments(opt, orc)
    assert np.all(opt.block_flags() == 0)
    bad = Xs[1].copy()
    bad[3, 20] = np.nan
    opt.accumulate([None, to_dev(bad, "f32")])
    flags = opt.block_flags()
    assert flags[opt.block_offset(1) + 1] & 1 and flags[opt.block_offset(1)] == 0
    # refresh keeps the previous basis (identity) for the non-finite block
    opt.refresh()
    f2 = opt.block_flags()
    assert f2[opt.block_offset(1) + 1] & 4
    Q = to_np(opt.tensor("bases", 1))
    assert np.array_equal(Q[1], np.eye(16))


# --------------------------------------------------------------------------
# (a2) eigen refresh
# --------------------------------------------------------------------------

@pytest.mark.parametrize("solver", ["default", "one-cta"])
@pytest.mark.parametrize("k", [1, 2, 3, 5, 16, 48, 64, 100, 128, 168, 169, 192, 400, 448])
def test_refresh_on_spd_blocks_with_gaps(k, solver):
    """Both eigensolvers (by default the grid solver for k >= 64 and one CTA
    per block below; "one-cta" forces the latter) on SPD blocks with gaps."""
    rng = np.random.default_rng(k)
    B = 2
    shapes = [(4, B * k)]
    opt = _dobb(shapes, B, refresh_period=0)
    if solver == "one-cta":
        opt.set_eig_grid(0)
    A = np.stack([I.spd_with_gap(k, rng, cond=1e6)[0] if k > 1 else np.array([[0.7]])
                  for _ in range(B)])
    opt.tensor("moments", 0).copy_(torch.from_numpy(A.astype(np.float32)).view(B, k, k))
    A32 = A.astype(np.float32).astype(np.float64)
    opt.refresh()
    torch.cuda.synchronize()
    check_bases(opt, [A32])
    assert np.all(opt.block_flags() == 0)
    chk = opt.check_bases()
    assert chk[:, 0].max() <= 1e-5 and chk[:, 2].max() <= 1e-5


def test_refresh_on_a_1600_wide_stress_block():
    """Refresh-stress shape at B = 4 / B = 1 (k = 1600): one SPD block with
    every relative eigenvalue gap >= 1e-3 and condition number 1e6, solved
    from the identity by one CTA."""
    k = 1600
    rng = np.random.default_rng(1600)
    opt = _dobb([(4, k)], 1, refresh_period=0)
    A = I.spd_with_gap(k, rng, cond=1e6)[0]
    opt.tensor("moments", 0).copy_(torch.from_numpy(A.astype(np.float32)).view(1, k, k))
    A32 = A.astype(np.float32).astype(np.float64)
    opt.refresh()
    torch.cuda.synchronize()
    check_bases(opt, [A32[None]])
    assert np.all(opt.block_flags() == 0)


@pytest.mark.parametrize("k,eff", [(192, 0.15), (100, 0.10), (64, 0.40)])
def test_refresh_on_accumulated_moments(k, eff):
    """Blocks of a low-effective-rank activation moment (ill-conditioned)."""
    B = 2
    shapes = [(16, B * k)]
    Xs, _, _ = make_problem(shapes, 1024, eff, seed=3)
    opt = _dobb(shapes, B, beta2=0.0, refresh_period=0)
    opt.accumulate([to_dev(Xs[0], "f32")])
    opt.refresh()
    torch.cuda.synchronize()
    A_gpu = to_np(opt.tensor("moments", 0))
    check_bases(opt, [A_gpu])
    orc = O.DobbOracle(shapes, B, beta2=0.0, refresh_period=0)
    orc.accumulate(Xs)
    check_moments(opt, orc)


@pytest.mark.parametrize("n,B,eff", [(1600, 16, 0.3), (3200, 8, 0.2)])
def test_refresh_cold_then_warm_on_every_block(n, B, eff):
    """Every block of two wide matrices (k = 100 / 400), refreshed from the
    identity and again from the previous basis after the moments moved with a
    second batch of the same distribution.  A solver that ends on a sweep of a
    B carrying the rounding of earlier sweeps misses the tolerance on a few
    blocks only, so all of them are scored."""
    shapes = [(8, n), (8, n)]
    rng = np.random.default_rng(11)
    X = [I.activations(4096, n, eff, rng, dtype="bf16") for _ in shapes]
    opt = _dobb(shapes, B, beta2=0.9, refresh_period=0, act_dtype="bf16")
    for half in (slice(0, 2048), slice(2048, 4096)):
        opt.accumulate([to_dev(np.ascontiguousarray(x[half]), "bf16") for x in X])
        opt.refresh()
        torch.cuda.synchronize()
        check_bases(opt, [to_np(opt.tensor("moments", i)) for i in range(len(shapes))])
        assert np.all(opt.block_flags() == 0)


# --------------------------------------------------------------------------
# (a3 - a7) the update, with the GPU's own basis
# --------------------------------------------------------------------------

@pytest.mark.parametrize("pdt", ["f32", "bf16"])
@pytest.mark.parametrize("shapes,B", [
    ([(37, 96)], 2),            # k = 48, ragged rows
    ([(1, 24), (17, 24)], 3),   # m = 1, k = 8
    ([(130, 200)], 2),          # k = 100
    ([(200, 400)], 1),          # k = 400
    ([(9, 15)], 5),             # k = 3 (odd)
])
def test_update_matches_oracle_with_gpu_basis(pdt, shapes, B):
    # at least 4 k tokens: a full-rank moment, so no column of C is exactly 0
    N = max(256, 4 * max(n // B for _, n in shapes))
    Xs, Gs, Ws = make_problem(shapes, N, 0.2, seed=4, param_dtype=pdt)
    opt = _dobb(shapes, B, beta1=0.9, beta2=0.95, refresh_period=1, scale_s=1.5, param_dtype=pdt)
    Wd = [to_dev(w, pdt) for w in Ws]
    Gd = [to_dev(g, pdt) for g in Gs]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Ws]
    M_prev = [np.zeros(s) for s in shapes]
    W_prev = [to_np(w) for w in Wd]
    opt.accumulate([to_dev(x, "f32") for x in Xs])
    opt.step(Wd, Gd, 0.02, signs=Sd)
    torch.cuda.synchronize()
    for i, (m, n) in enumerate(shapes):
        Q = to_np(opt.tensor("bases", i))
        check_update(W_prev[i], M_prev[i], to_np(Gd[i]), Q, to_np(Sd[i]), to_np(Wd[i]),
                     to_np(opt.tensor("momentum", i)), 0.9, 0.02, 1.5, pdt, n // B)
    # ||U_b||_F^2 equals the number of nonzero signs (orthonormal Q_b)
    st = opt.block_stats()
    for i, (m, n) in enumerate(shapes):
        k = n // B
        S = to_np(Sd[i])
        for b in range(B):
            nnz = np.count_nonzero(S[:, b * k:(b + 1) * k])
            assert abs(st[opt.block_offset(i) + b, 0] - nnz) <= 1e-4 * max(nnz, 1)


@pytest.mark.parametrize("pdt", ["f32", "bf16"])
@pytest.mark.parametrize("shapes,B", [
    ([(37, 96)], 2),            # k = 48, tensor cores
    ([(130, 200)], 2),          # k = 100, tensor cores
    ([(200, 400)], 1),          # k = 400, tensor cores
    ([(9, 15)], 5),             # k = 3, FP32 path
])
def test_update_with_bf16_basis_matches_oracle(pdt, shapes, B):
    """[Dobb, Table 18] bf16 basis storage: the update multiplies with the
    basis rounded once to bf16; scored against the oracle with the GPU's
    basis, rounded by the oracle."""
    N = max(256, 4 * max(n // B for _, n in shapes))
    Xs, Gs, Ws = make_problem(shapes, N, 0.2, seed=14, param_dtype=pdt)
    opt = _dobb(shapes, B, beta1=0.9, beta2=0.95, refresh_period=1, scale_s=1.5, param_dtype=pdt,
                basis_dtype="bf16")
    Wd = [to_dev(w, pdt) for w in Ws]
    Gd = [to_dev(g, pdt) for g in Gs]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Ws]
    W_prev = [to_np(w) for w in Wd]
    opt.accumulate([to_dev(x, "f32") for x in Xs])
    opt.step(Wd, Gd, 0.02, signs=Sd)
    torch.cuda.synchronize()
    for i, (m, n) in enumerate(shapes):
        Q = to_np(opt.tensor("bases", i))
        check_update(W_prev[i], np.zeros((m, n)), to_np(Gd[i]), Q, to_np(Sd[i]), to_np(Wd[i]),
                     to_np(opt.tensor("momentum", i)), 0.9, 0.02, 1.5, pdt, n // B, basis_dtype="bf16")
    # the rounding acts: the fp32-basis update differs somewhere
    Q = to_np(opt.tensor("bases", 0))
    m, n = shapes[0]
    r32 = O.update_from_bases(W_prev[0], np.zeros((m, n)), to_np(Gd[0]), Q, 0.9, 0.02, 1.5, "f32")
    assert np.abs(r32["W"] - to_np(Wd[0])).max() > 0


def test_identity_basis_gives_sign_of_momentum():
    shapes = [(33, 40)]
    _, Gs, Ws = make_problem(shapes, 8, 0.5, seed=5)
    opt = _dobb(shapes, 4, beta1=0.5, refresh_period=0, scale_s=2.0)
    Wd, Gd = [to_dev(Ws[0], "f32")], [to_dev(Gs[0], "f32")]
    W0 = to_np(Wd[0])
    opt.step(Wd, Gd, 0.01)
    torch.cuda.synchronize()
    expect = W0 - 0.01 * 2.0 * np.sign(Gs[0].astype(np.float64))
    assert MX.w_rel_error(to_np(Wd[0]), expect) <= 1e-6


def test_nonfinite_gradient_is_flagged():
    shapes = [(16, 32)]
    _, Gs, Ws = make_problem(shapes, 8, 0.5, seed=6)
    G = Gs[0].copy()
    G[2, 30] = np.inf
    opt = _dobb(shapes, 2, refresh_period=0)
    opt.step([to_dev(Ws[0], "f32")], [to_dev(G, "f32")], 0.01)
    f = opt.block_flags()
    assert f[1] & 2 and not f[0] & 2


# --------------------------------------------------------------------------
# whole runs: single fp32 768 x 768 matrix, B = 4 (k = 192), 10 steps,
# refresh every 5, beta1 0.95, beta2 0.99, lr 0.02, s 1, seed 0
# --------------------------------------------------------------------------

def _run(shapes, B, N, eff, steps, T, pdt, adt, seed, beta1=0.95, beta2=0.99, lr=0.02, s=1.0):
    rng = np.random.default_rng(seed)
    opt = _dobb(shapes, B, beta1=beta1, beta2=beta2, refresh_period=T, scale_s=s,
                param_dtype=pdt, act_dtype=adt)
    orc = O.DobbOracle(shapes, B, beta1=beta1, beta2=beta2, refresh_period=0, scale_s=s,
                       param_dtype=pdt)
    Ws = [I.weights(m, n, rng, dtype=pdt) for (m, n) in shapes]
    Wd = [to_dev(w, pdt) for w in Ws]
    for t in range(steps):
        Xs = [I.activations(N, n, eff, rng, dtype=adt) for (m, n) in shapes]
        Gs = [I.gradients(m, X, rng, dtype=pdt) for (m, n), X in zip(shapes, Xs)]
        Gd = [to_dev(g, pdt) for g in Gs]
        Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Wd]
        W_prev = [to_np(w) for w in Wd]
        M_prev = [m.copy() for m in orc.M]
        opt.accumulate([to_dev(x, adt) for x in Xs])
        orc.accumulate(Xs)
        opt.step(Wd, Gd, lr, signs=Sd)
        torch.cuda.synchronize()
        check_moments(opt, orc)
        if T > 0 and t % T == 0:
            # the eigensolver is scored on the moments it was given; the
            # moments themselves were scored against the oracle just above
            check_bases(opt, [to_np(opt.tensor("moments", i)) for i in range(len(shapes))])
        for i, (m, n) in enumerate(shapes):
            Q = to_np(opt.tensor("bases", i))
            check_update(W_prev[i], M_prev[i], to_np(Gd[i]), Q, to_np(Sd[i]), to_np(Wd[i]),
                         to_np(opt.tensor("momentum", i)), beta1, lr, s, pdt, n // B)
            orc.M[i] = O.momentum(M_prev[i], to_np(Gd[i]), beta1)
    return opt


def test_single_matrix_ten_steps():
    _run([(768, 768)], 4, 1024, 0.15, steps=10, T=5, pdt="f32", adt="f32", seed=0)


def test_small_model_bf16_mixed_shapes():
    shapes = [(96, 64), (256, 64), (64, 256)]
    _run(shapes, 4, 512, 0.2, steps=4, T=2, pdt="bf16", adt="bf16", seed=7)


# --------------------------------------------------------------------------
# checkpoint / resume is bitwise
# --------------------------------------------------------------------------

def test_checkpoint_resume_bitwise():
    shapes = [(64, 96), (32, 48)]
    rng = np.random.default_rng(8)
    seq = []
    for t in range(8):
        Xs = [I.activations(64, n, 0.3, rng) for (m, n) in shapes]
        Gs = [I.gradients(m, X, rng) for (m, n), X in zip(shapes, Xs)]
        seq.append((Xs, Gs))
    W0 = [I.weights(m, n, rng) for (m, n) in shapes]

    def run(opt, W, ts):
        for t in ts:
            Xs, Gs = seq[t]
            opt.accumulate([to_dev(x, "f32") for x in Xs])
            opt.step(W, [to_dev(g, "f32") for g in Gs], 0.02)

    a = _dobb(shapes, 2, refresh_period=3)
    Wa = [to_dev(w, "f32") for w in W0]
    run(a, Wa, range(5))
    buf, t = a.get_state()
    W_mid = [w.clone() for w in Wa]
    run(a, Wa, range(5, 8))
    b = _dobb(shapes, 2, refresh_period=3)
    b.set_state(buf, t)
    run(b, W_mid, range(5, 8))
    torch.cuda.synchronize()
    for x, y in zip(Wa, W_mid):
        assert torch.equal(x, y)
    assert torch.equal(a.tensor("momentum"), b.tensor("momentum"))
    assert torch.equal(a.tensor("bases"), b.tensor("bases"))


# --------------------------------------------------------------------------
# tensor-core update kernel vs FFMA kernel vs oracle
# --------------------------------------------------------------------------

@pytest.mark.parametrize("pdt", ["f32", "bf16"])
@pytest.mark.parametrize("shapes,B", [
    ([(300, 1600), (200, 6400)], 16),   # k = 100 and 400 (GPT-2 XL blocks), ragged rows
    ([(129, 896)], 2),                  # k = 448 (largest tensor-core width)
    ([(257, 512)], 4),                  # k = 128
    ([(64, 48), (5, 20)], 4),           # k = 12 and 5 (5: FFMA-only remainder)
])
def test_tensor_core_and_ffma_paths_agree(pdt, shapes, B):
    """Both update kernels, run on the same inputs and the same basis, meet
    the oracle's sign and parameter rules with their own signs."""
    N = max(512, 4 * max(n // B for _, n in shapes))
    Xs, Gs, Ws = make_problem(shapes, N, 0.15, seed=21, param_dtype=pdt)
    bases = None
    for path in ("auto", "ffma"):
        opt = _dobb(shapes, B, beta1=0.95, beta2=0.99, refresh_period=1, param_dtype=pdt)
        opt.set_step_path(path)
        Wd = [to_dev(w, pdt) for w in Ws]
        Gd = [to_dev(g, pdt) for g in Gs]
        Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Ws]
        opt.accumulate([to_dev(x, "f32") for x in Xs])
        W_prev = [to_np(w) for w in Wd]
        opt.step(Wd, Gd, 0.02, signs=Sd)
        torch.cuda.synchronize()
        assert opt.device_error() == 0
        Q = [to_np(opt.tensor("bases", i)) for i in range(len(shapes))]
        if bases is None:
            bases = Q
        for i, (m, n) in enumerate(shapes):
            assert np.array_equal(Q[i], bases[i])  # the same refresh kernel
            check_update(W_prev[i], np.zeros((m, n)), to_np(Gd[i]), Q[i], to_np(Sd[i]),
                         to_np(Wd[i]), to_np(opt.tensor("momentum", i)), 0.95, 0.02, 1.0,
                         pdt, n // B)


def test_tensor_core_update_matches_oracle_multi_step():
    """GPT-2 XL block shapes (k = 100, 400), bf16 parameters, three steps,
    each scored against the oracle run with the GPU basis and GPU signs."""
    shapes = [(256, 1600), (160, 6400)]
    _run(shapes, 16, 1024, 0.2, steps=3, T=2, pdt="bf16", adt="bf16", seed=22)


# --------------------------------------------------------------------------
# (f1) orthogonal-iteration refresh ([Dobb, Table 15] principal, Table 16)
# --------------------------------------------------------------------------

def _orth_case(k, B, cond, seed):
    rng = np.random.default_rng(seed)
    A = np.stack([I.spd_with_gap(k, rng, cond=cond)[0] if k > 1 else np.array([[0.7]])
                  for _ in range(B)]).astype(np.float32).astype(np.float64)
    Q0 = np.stack([I.haar_orthogonal(k, rng) for _ in range(B)]).astype(np.float32).astype(np.float64)
    return A, Q0


def _load(opt, A, Q0, k, B):
    opt.tensor("moments", 0).copy_(torch.from_numpy(A.astype(np.float32)).view(B, k, k))
    opt.tensor("bases", 0).copy_(torch.from_numpy(Q0.astype(np.float32)).view(B, k, k))


@pytest.mark.parametrize("k", [1, 3, 31, 48, 65, 100, 130, 400])
def test_orth_refresh_is_one_cholesky_qr_step(k):
    """One step: Q = T R^{-1}, T = A Q0.  Scored by what fixes the QR factor of
    T: orthonormal columns, Q^T T upper triangular with a positive diagonal
    (backward stable, independent of kappa(T)), and the forward error against
    the fp64 oracle within the fp32 perturbation bound ~ kappa k eps."""
    B, cond = 2, 50.0
    A, Q0 = _orth_case(k, B, cond, seed=100 + k)
    opt = _dobb([(4, B * k)], B, refresh_period=0, refresh="orth", orth_steps=1)
    _load(opt, A, Q0, k, B)
    opt.refresh()
    torch.cuda.synchronize()
    Q = to_np(opt.tensor("bases", 0))
    lam = to_np(opt.tensor("eigvals", 0))
    Qr, lr = O.orthogonal_iteration(A, Q0, 1)
    assert np.all(opt.block_flags() == 0)
    for b in range(B):
        T = A[b] @ Q0[b]
        R = Q[b].T @ T
        assert np.linalg.norm(Q[b].T @ Q[b] - np.eye(k)) <= 1e-5 * max(1.0, np.sqrt(k))
        assert np.linalg.norm(np.tril(R, -1)) <= 1e-5 * np.linalg.norm(T)
        assert np.all(np.diag(R) > 0)
        assert np.linalg.norm(Q[b] - Qr[b]) <= 20 * cond * k * 2.0 ** -24
        assert np.abs(lam[b] - lr[b]).max() <= 1e-5 * np.abs(lr[b]).max()


def test_orth_refresh_converges_to_the_eigenbasis():
    k, B = 48, 2
    A, Q0 = _orth_case(k, B, 20.0, seed=7)
    opt = _dobb([(4, B * k)], B, refresh_period=0, refresh="orth", orth_steps=400)
    _load(opt, A, Q0, k, B)
    opt.refresh()
    torch.cuda.synchronize()
    Q = to_np(opt.tensor("bases", 0))
    lam = to_np(opt.tensor("eigvals", 0))
    Qe, le = O.refresh_bases(A, "lapack")
    for b in range(B):
        assert np.abs(np.abs(Q[b].T @ Qe[b]) - np.eye(k)).max() <= 1e-4
        assert np.abs(lam[b] - le[b]).max() <= 1e-5 * le[b].max()


def test_orth_refresh_shifted_pass_on_ill_conditioned_blocks():
    """kappa(A) = 1e6: the fp32 Gram matrix of T = A Q0 is not positive
    definite, so shifted passes come first (each lowers kappa by ~0.1 at
    k = 100); the factor is still orthonormal and Q^T T upper triangular to
    fp32 level."""
    k, B = 100, 2
    A, Q0 = _orth_case(k, B, 1e6, seed=8)
    opt = _dobb([(4, B * k)], B, refresh_period=0, refresh="orth", orth_steps=1)
    _load(opt, A, Q0, k, B)
    opt.refresh()
    torch.cuda.synchronize()
    Q = to_np(opt.tensor("bases", 0))
    assert np.all(opt.block_flags() == 0)
    st = opt.block_stats()
    assert np.all(st[:, 3] >= 1.0)  # shifted passes were taken
    for b in range(B):
        T = A[b] @ Q0[b]
        assert np.linalg.norm(Q[b].T @ Q[b] - np.eye(k)) <= 1e-5 * np.sqrt(k)
        assert np.linalg.norm(np.tril(Q[b].T @ T, -1)) <= 1e-4 * np.linalg.norm(T)


@pytest.mark.parametrize("k", [64, 100, 400])
def test_orth_grid_and_one_cta_forms_agree(k):
    """Blocks at least 64 wide run the orthogonal iteration on the grid
    (batched tile products, a Cholesky factorisation per block, the
    triangular solve split by 64-row panels); the one-CTA form runs the same
    steps in one CTA per block.  Three steps from a Haar start: both match the
    fp64 oracle to the fp32 perturbation bound, and their Rayleigh quotients
    agree."""
    B, cond, steps = 3, 50.0, 3
    A, Q0 = _orth_case(k, B, cond, seed=300 + k)
    Qr, lr = O.orthogonal_iteration(A, Q0, steps)
    out = []
    for grid in (True, False):
        opt = _dobb([(4, B * k)], B, refresh_period=0, refresh="orth", orth_steps=steps)
        if not grid:
            opt.set_eig_grid(0)
        _load(opt, A, Q0, k, B)
        opt.refresh()
        torch.cuda.synchronize()
        assert np.all(opt.block_flags() == 0)
        Q = to_np(opt.tensor("bases", 0))
        lam = to_np(opt.tensor("eigvals", 0))
        for b in range(B):
            assert np.linalg.norm(Q[b].T @ Q[b] - np.eye(k)) <= 1e-5 * np.sqrt(k)
            assert np.linalg.norm(Q[b] - Qr[b]) <= 20 * cond * k * 2.0 ** -24 * steps
            assert np.abs(lam[b] - lr[b]).max() <= 1e-5 * np.abs(lr[b]).max()
        out.append((Q, lam))
    assert np.abs(out[0][1] - out[1][1]).max() <= 2e-5 * np.abs(out[1][1]).max()


def test_orth_grid_hands_ill_conditioned_blocks_to_the_shifted_passes():
    """A batch mixing well- and ill-conditioned 100-wide blocks on the grid:
    the well-conditioned blocks finish there (no shifted pass), the others
    (Gram matrix of T not positive definite in fp32) are redone from their
    old basis by the one-CTA shifted passes; every block ends orthonormal with
    Q^T T upper triangular."""
    k, B = 100, 4
    rng = np.random.default_rng(9)
    conds = [50.0, 1e6, 50.0, 1e6]
    A = np.stack([I.spd_with_gap(k, rng, cond=c)[0] for c in conds]).astype(np.float32).astype(np.float64)
    Q0 = np.stack([I.haar_orthogonal(k, rng) for _ in range(B)]).astype(np.float32).astype(np.float64)
    opt = _dobb([(4, B * k)], B, refresh_period=0, refresh="orth", orth_steps=1)
    _load(opt, A, Q0, k, B)
    opt.refresh()
    torch.cuda.synchronize()
    assert np.all(opt.block_flags() == 0)
    st = opt.block_stats()
    Q = to_np(opt.tensor("bases", 0))
    for b in range(B):
        T = A[b] @ Q0[b]
        assert np.linalg.norm(Q[b].T @ Q[b] - np.eye(k)) <= 1e-5 * np.sqrt(k)
        assert np.linalg.norm(np.tril(Q[b].T @ T, -1)) <= 1e-4 * np.linalg.norm(T)
        assert (st[b, 3] >= 1.0) == (conds[b] > 1e3)


@pytest.mark.parametrize("pdt", ["f32", "bf16"])
def test_run_with_orth_refresh_matches_oracle_updates(pdt):
    """A short run refreshing by one orthogonal-iteration step every 2 steps:
    moments against the oracle, every update against the oracle with the
    GPU's basis."""
    shapes, B = [(96, 200), (64, 128)], 2
    rng = np.random.default_rng(21)
    opt = _dobb(shapes, B, beta1=0.9, beta2=0.9, refresh_period=2, scale_s=1.0, param_dtype=pdt,
                refresh="orth", orth_steps=1)
    orc = O.DobbOracle(shapes, B, beta1=0.9, beta2=0.9, refresh_period=0, param_dtype=pdt)
    Wd = [to_dev(I.weights(m, n, rng, dtype=pdt), pdt) for m, n in shapes]
    for t in range(5):
        Xs = [I.activations(512, n, 0.3, rng) for _, n in shapes]
        Gs = [I.gradients(m, X, rng, dtype=pdt) for (m, _), X in zip(shapes, Xs)]
        Gd = [to_dev(g, pdt) for g in Gs]
        Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Wd]
        W_prev = [to_np(w) for w in Wd]
        M_prev = [m.copy() for m in orc.M]
        opt.accumulate([to_dev(x, "f32") for x in Xs])
        orc.accumulate(Xs)
        opt.step(Wd, Gd, 0.02, signs=Sd)
        torch.cuda.synchronize()
        check_moments(opt, orc)
        for i, (m, n) in enumerate(shapes):
            Q = to_np(opt.tensor("bases", i))
            r = check_update(W_prev[i], M_prev[i], to_np(Gd[i]), Q, to_np(Sd[i]), to_np(Wd[i]),
                             to_np(opt.tensor("momentum", i)), 0.9, 0.02, 1.0, pdt, n // B)
            orc.M[i] = O.momentum(M_prev[i], to_np(Gd[i]), 0.9)
            assert np.linalg.norm(Q[0].T @ Q[0] - np.eye(n // B)) <= 1e-5 * np.sqrt(n // B)


# --------------------------------------------------------------------------
# (f2) Dobb-l2: column l2 normalisation ([Dobb, Tables 9 and 11])
# --------------------------------------------------------------------------

@pytest.mark.parametrize("pdt", ["f32", "bf16"])
@pytest.mark.parametrize("shapes,B", [
    ([(37, 96)], 2),            # k = 48, ragged rows
    ([(1, 24), (17, 24)], 3),   # m = 1 (l2 = sign there), k = 8
    ([(130, 200)], 2),          # k = 100
    ([(200, 400)], 1),          # k = 400
    ([(9, 15)], 5),             # k = 3 (odd)
])
def test_update_with_l2_normalisation_matches_oracle(pdt, shapes, B):
    N = max(256, 4 * max(n // B for _, n in shapes))
    Xs, Gs, Ws = make_problem(shapes, N, 0.2, seed=24, param_dtype=pdt)
    opt = _dobb(shapes, B, beta1=0.9, beta2=0.95, refresh_period=1, scale_s=1.5, param_dtype=pdt,
                norm="l2")
    Wd = [to_dev(w, pdt) for w in Ws]
    Gd = [to_dev(g, pdt) for g in Gs]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Ws]
    W_prev = [to_np(w) for w in Wd]
    opt.accumulate([to_dev(x, "f32") for x in Xs])
    opt.step(Wd, Gd, 0.02, signs=Sd)
    torch.cuda.synchronize()
    st = opt.block_stats()
    for i, (m, n) in enumerate(shapes):
        k = n // B
        Q = to_np(opt.tensor("bases", i))
        check_update_l2(W_prev[i], np.zeros((m, n)), to_np(Gd[i]), Q, to_np(Wd[i]),
                        to_np(opt.tensor("momentum", i)), 0.9, 0.02, 1.5, pdt)
        # the returned signs are those of C
        ref = O.update_from_bases(W_prev[i], np.zeros((m, n)), to_np(Gd[i]), Q, 0.9, 0.02, 1.5, "f32")
        sa = MX.sign_agreement(ref["C"], to_np(Sd[i]), k)
        assert sa["outside_band"] == 0
        # ||U_b||_F^2 = m k: every column of S has norm sqrt(m), Q_b orthonormal
        for b in range(B):
            assert abs(st[opt.block_offset(i) + b, 0] - m * k) <= 1e-4 * m * k


def test_run_with_l2_normalisation_and_refresh():
    """Several steps with refreshes: moments, bases and every Dobb-l2 update
    against the oracle with the GPU's basis."""
    shapes, B = [(64, 192), (96, 128)], 2
    rng = np.random.default_rng(25)
    opt = _dobb(shapes, B, beta1=0.95, beta2=0.9, refresh_period=2, scale_s=1.0, norm="l2")
    orc = O.DobbOracle(shapes, B, beta1=0.95, beta2=0.9, refresh_period=0, norm="l2")
    Wd = [to_dev(I.weights(m, n, rng), "f32") for m, n in shapes]
    for t in range(5):
        Xs = [I.activations(512, n, 0.3, rng) for _, n in shapes]
        Gd = [to_dev(I.gradients(m, X, rng), "f32") for (m, _), X in zip(shapes, Xs)]
        W_prev = [to_np(w) for w in Wd]
        M_prev = [m.copy() for m in orc.M]
        opt.accumulate([to_dev(x, "f32") for x in Xs])
        orc.accumulate(Xs)
        opt.step(Wd, Gd, 0.02)
        torch.cuda.synchronize()
        check_moments(opt, orc)
        if t % 2 == 0:
            check_bases(opt, [to_np(opt.tensor("moments", i)) for i in range(len(shapes))])
        for i, (m, n) in enumerate(shapes):
            Q = to_np(opt.tensor("bases", i))
            check_update_l2(W_prev[i], M_prev[i], to_np(Gd[i]), Q, to_np(Wd[i]),
                            to_np(opt.tensor("momentum", i)), 0.95, 0.02, 1.0, "f32")
            orc.M[i] = O.momentum(M_prev[i], to_np(Gd[i]), 0.95)


# --------------------------------------------------------------------------
# (f4) Dobb-G: bases of the output-gradient second moment, row blocks
# ([Dobb, Tables 12-13]); W, G and signs in the caller's (m, n) layout
# --------------------------------------------------------------------------

@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_output_side_moments_match_oracle(act):
    shapes, B = [(96, 24), (64, 33)], 2
    Ds, _, _ = make_output_side_problem(shapes, 77, 0.3, seed=30, act_dtype=act)
    opt = _dobb(shapes, B, beta2=0.9, refresh_period=0, act_dtype=act, side="output")
    orc = O.DobbOracle(shapes, B, beta2=0.9, refresh_period=0, side="output")
    for _ in range(2):
        opt.accumulate([to_dev(d, act) for d in Ds])
        orc.accumulate(Ds)
    torch.cuda.synchronize()
    for i, (m, n) in enumerate(shapes):
        assert tuple(opt.tensor("moments", i).shape) == (B, m // B, m // B)
    check_moments(opt, orc)


@pytest.mark.parametrize("pdt", ["f32", "bf16"])
@pytest.mark.parametrize("norm", ["sign", "l2"])
@pytest.mark.parametrize("shapes,B", [
    ([(96, 37)], 2),            # k = 48, ragged columns
    ([(24, 1), (24, 17)], 3),   # n = 1, k = 8
    ([(200, 130)], 2),          # k = 100
    ([(400, 200)], 1),          # k = 400
    ([(15, 9)], 5),             # k = 3 (odd)
])
def test_output_side_update_matches_oracle(pdt, norm, shapes, B):
    N = max(256, 4 * max(m // B for m, _ in shapes))
    Ds, Gs, Ws = make_output_side_problem(shapes, N, 0.2, seed=31, param_dtype=pdt)
    opt = _dobb(shapes, B, beta1=0.9, beta2=0.95, refresh_period=1, scale_s=1.5, param_dtype=pdt,
                norm=norm, side="output")
    Wd = [to_dev(w, pdt) for w in Ws]
    Gd = [to_dev(g, pdt) for g in Gs]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Ws]
    W_prev = [to_np(w) for w in Wd]
    opt.accumulate([to_dev(d, "f32") for d in Ds])
    opt.step(Wd, Gd, 0.02, signs=Sd)
    torch.cuda.synchronize()
    st = opt.block_stats()
    for i, (m, n) in enumerate(shapes):
        k = m // B
        Q = to_np(opt.tensor("bases", i))
        M_gpu = to_np(opt.tensor("momentum", i)).T    # registered as W^T
        if norm == "sign":
            check_update(W_prev[i], np.zeros((m, n)), to_np(Gd[i]), Q, to_np(Sd[i]), to_np(Wd[i]),
                         M_gpu, 0.9, 0.02, 1.5, pdt, k, side="output")
        else:
            check_update_l2(W_prev[i], np.zeros((m, n)), to_np(Gd[i]), Q, to_np(Wd[i]), M_gpu,
                            0.9, 0.02, 1.5, pdt, side="output")
            # sign output: the signs of C = Q_b^T M_b
            ref = O.update_from_bases(W_prev[i], np.zeros((m, n)), to_np(Gd[i]), Q, 0.9, 0.02,
                                      1.5, "f32", side="output")
            sa = MX.sign_agreement(ref["C"].T, to_np(Sd[i]).T, k)
            assert sa["outside_band"] == 0
        # ||U_b||_F^2: number of nonzero signs, or k n for the row-l2 update
        S = to_np(Sd[i])
        for b in range(B):
            want = np.count_nonzero(S[b * k:(b + 1) * k, :]) if norm == "sign" else n * k
            assert abs(st[opt.block_offset(i) + b, 0] - want) <= 1e-4 * max(want, 1)


@pytest.mark.parametrize("path,pdt", [("ffma", "f32"), ("auto", "f32"), ("auto", "bf16")])
def test_output_side_is_input_side_on_the_transpose(path, pdt):
    """Dobb-G on W with output gradients D is Dobb on W^T with D as the
    activations: both runs of the same registered problem agree bit for bit,
    on the FP32 update kernel and on the tensor-core one (k = 64: the
    transposed parameter addressing is the only difference)."""
    m, n, B = 192, 80, 3
    rng = np.random.default_rng(32)
    W = I.weights(m, n, rng, dtype=pdt)
    kw = dict(beta1=0.9, beta2=0.95, refresh_period=2, scale_s=1.0, param_dtype=pdt)
    opt_g = _dobb([(m, n)], B, side="output", **kw)
    opt_t = _dobb([(n, m)], B, **kw)
    opt_g.set_step_path(path)
    opt_t.set_step_path(path)
    Wg, Wt = to_dev(W, pdt), to_dev(np.ascontiguousarray(W.T), pdt)
    Sg = torch.zeros((m, n), dtype=torch.int8, device="cuda")
    St = torch.zeros((n, m), dtype=torch.int8, device="cuda")
    for _ in range(4):
        D = I.activations(300, m, 0.25, rng)
        X = I.activations(300, n, 0.5, rng)
        G = (D.astype(np.float64).T @ X / 300).astype(np.float32)
        if pdt == "bf16":
            G = I.round_bf16_np(G)
        opt_g.accumulate([to_dev(D, "f32")])
        opt_t.accumulate([to_dev(D, "f32")])
        opt_g.step([Wg], [to_dev(G, pdt)], 0.01, signs=[Sg])
        opt_t.step([Wt], [to_dev(np.ascontiguousarray(G.T), pdt)], 0.01, signs=[St])
    torch.cuda.synchronize()
    assert torch.equal(opt_g.tensor("bases", 0), opt_t.tensor("bases", 0))
    assert torch.equal(opt_g.tensor("momentum", 0), opt_t.tensor("momentum", 0))
    assert torch.equal(Wg, Wt.T)
    assert torch.equal(Sg, St.T)


def test_mixed_sides_run_matches_oracle():
    """One input-side and one output-side matrix in one handle, several steps
    with refreshes; each scored against the oracle of its side."""
    shapes, B = [(64, 96), (96, 64)], 2
    sides = ["input", "output"]
    rng = np.random.default_rng(33)
    opt = _dobb(shapes, B, beta1=0.95, beta2=0.9, refresh_period=2, side=sides)
    orcs = [O.DobbOracle([s], B, beta1=0.95, beta2=0.9, refresh_period=0, side=sd)
            for s, sd in zip(shapes, sides)]
    Wd = [to_dev(I.weights(m, n, rng), "f32") for m, n in shapes]
    for t in range(5):
        Xs = [I.activations(400, n if sd == "input" else m, 0.3, rng)
              for (m, n), sd in zip(shapes, sides)]
        Gs = [I.gradients(shapes[0][0], Xs[0], rng),
              (Xs[1].astype(np.float64).T @ I.activations(400, shapes[1][1], 0.5, rng) / 400
               ).astype(np.float32)]
        Gd = [to_dev(g, "f32") for g in Gs]
        Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Wd]
        W_prev = [to_np(w) for w in Wd]
        M_prev = [o.M[0].copy() for o in orcs]
        opt.accumulate([to_dev(x, "f32") for x in Xs])
        for o, X in zip(orcs, Xs):
            o.accumulate([X])
        opt.step(Wd, Gd, 0.02, signs=Sd)
        torch.cuda.synchronize()
        for i, ((m, n), sd) in enumerate(zip(shapes, sides)):
            Ag = to_np(opt.tensor("moments", i))
            rel = np.linalg.norm(Ag - orcs[i].A[0]) / np.linalg.norm(orcs[i].A[0])
            assert rel <= TOL_A
            if t % 2 == 0:
                check_bases(opt, {i: Ag}, matrices=[i])
            Q = to_np(opt.tensor("bases", i))
            M_gpu = to_np(opt.tensor("momentum", i))
            check_update(W_prev[i], M_prev[i], to_np(Gd[i]), Q, to_np(Sd[i]), to_np(Wd[i]),
                         M_gpu.T if sd == "output" else M_gpu, 0.95, 0.02, 1.0, "f32",
                         (m if sd == "output" else n) // B, side=sd)
            orcs[i].M[0] = O.momentum(M_prev[i], to_np(Gd[i]), 0.95)


# --------------------------------------------------------------------------
# (a8) the invariant check and the per-block sums, scored against fp64
# --------------------------------------------------------------------------

def test_check_bases_matches_oracle_residuals():
    """dobb_check_bases gives, per block, the three residuals of
    `oracle.metrics.eig_residuals` evaluated on the same fp32 A, Q, Lambda:
    on converged bases, and on bases with a planted error (a column mixed
    with its neighbour, a column scaled), where the residuals are large."""
    shapes, B = [(16, 96), (16, 400), (8, 1600)], 2     # k = 48, 200, 800
    Xs, _, _ = make_problem(shapes, 2048, 0.3, seed=40)
    opt = _dobb(shapes, B, beta2=0.0, refresh_period=0)
    opt.accumulate([to_dev(x, "f32") for x in Xs])
    opt.refresh()
    torch.cuda.synchronize()

    def compare():
        chk = opt.check_bases()
        for i in range(len(shapes)):
            A = to_np(opt.tensor("moments", i))
            Q = to_np(opt.tensor("bases", i))
            lam = to_np(opt.tensor("eigvals", i))
            for b in range(B):
                r = MX.eig_residuals(A[b], Q[b], lam[b])
                got = chk[opt.block_offset(i) + b]
                for j, key in enumerate(("residual", "orth", "recon")):
                    assert abs(got[j] - r[key]) <= 1e-5 * r[key] + 1e-12, (i, b, key, got[j], r[key])
        return chk

    chk = compare()
    assert chk[:, 0].max() <= 1e-5
    # planted errors in the stored bases (written through the state view)
    Qv = opt.tensor("bases", 1)
    Qv[0, :, 0] += 1e-2 * Qv[0, :, 50]
    Qv[1, :, 7] *= 1.01
    torch.cuda.synchronize()
    chk = compare()
    assert chk[opt.block_offset(1), 0] > 1e-5 and chk[opt.block_offset(1) + 1, 1] > 1e-2


@pytest.mark.parametrize("path", ["auto", "ffma"])
def test_block_stats_match_fp64_coefficient_norms(path):
    """Per-block sums of a step: ||C_b||_F^2 against the fp64 ||M_b Q_b||_F^2
    of the GPU's momentum and basis, within the fp32 bound of its evaluation:
    (k + ceil(m / 32) + 8) u for the sums of squares, and 2 sqrt(k) (k u +
    2^-21) for C itself (|sum 2 C e| <= 2 ||C|| ||e||, ||e|| <= (k u +
    2^-21) || |M_b| |Q_b| ||_F <= (k u + 2^-21) sqrt(k) ||C||, the 2^-21 from
    the split-precision products); ||U_b||_F^2 against the number of nonzero
    signs."""
    shapes, B = [(300, 1600), (130, 800), (64, 96)], 16     # k = 100, 50, 6
    Xs, Gs, Ws = make_problem(shapes, 1024, 0.2, seed=41, param_dtype="bf16")
    opt = _dobb(shapes, B, beta1=0.9, refresh_period=1, param_dtype="bf16")
    opt.set_step_path(path)
    Wd = [to_dev(w, "bf16") for w in Ws]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Ws]
    opt.accumulate([to_dev(x, "f32") for x in Xs])
    opt.step(Wd, [to_dev(g, "bf16") for g in Gs], 0.02, signs=Sd)
    torch.cuda.synchronize()
    st = opt.block_stats()
    u = 2.0 ** -24
    for i, (m, n) in enumerate(shapes):
        k = n // B
        M = to_np(opt.tensor("momentum", i))
        Q = to_np(opt.tensor("bases", i))
        S = to_np(Sd[i])
        for b in range(B):
            C = M[:, b * k:(b + 1) * k] @ Q[b]
            want = float((C ** 2).sum())
            tol = (k + math.ceil(m / 32) + 8) * u + 2 * math.sqrt(k) * (k * u + 2.0 ** -21)
            got = float(st[opt.block_offset(i) + b, 1])
            assert abs(got - want) <= tol * want, (i, b, got, want)
            nnz = np.count_nonzero(S[:, b * k:(b + 1) * k])
            assert abs(st[opt.block_offset(i) + b, 0] - nnz) <= 1e-4 * max(nnz, 1)


# --------------------------------------------------------------------------
# failure detection without a GPU fault: the eigensolver's sweep cap
# --------------------------------------------------------------------------

def test_sweep_cap_sets_not_converged_and_writes_a_basis():
    """With the sweep cap at 1, a cold refresh of an ill-conditioned block
    cannot converge: the block gets DOBB_FLAG_NOT_CONVERGED, the basis is
    still written (orthonormal to fp32 level, no longer the identity) and
    the step that follows runs.  Raising the cap again clears the
    condition on the next refresh."""
    k, B = 100, 2
    rng = np.random.default_rng(42)
    A = np.stack([I.spd_with_gap(k, rng, cond=1e6)[0] for _ in range(B)])
    opt = _dobb([(64, B * k)], B, refresh_period=0)
    opt.tensor("moments", 0).copy_(torch.from_numpy(A.astype(np.float32)).view(B, k, k))
    opt.set_jacobi(max_sweeps=1)
    opt.refresh()
    torch.cuda.synchronize()
    flags = opt.block_flags()
    assert np.all(flags & 8), flags
    st = opt.block_stats()
    assert np.all(st[:, 2] == 1.0)
    Q = to_np(opt.tensor("bases", 0))
    for b in range(B):
        assert np.all(np.isfinite(Q[b]))
        assert np.linalg.norm(Q[b].T @ Q[b] - np.eye(k)) <= 1e-4 * np.sqrt(k)
        assert np.abs(Q[b] - np.eye(k)).max() > 0.1
    W = to_dev(I.weights(64, B * k, rng), "f32")
    opt.step([W], [to_dev(rng.standard_normal((64, B * k)).astype(np.float32), "f32")], 0.01)
    torch.cuda.synchronize()
    assert opt.device_error() == 0 and torch.isfinite(W).all()
    opt.clear_flags()
    opt.set_jacobi(max_sweeps=40)
    opt.refresh()
    torch.cuda.synchronize()
    assert np.all(opt.block_flags() == 0)
    check_bases(opt, [A.astype(np.float32).astype(np.float64)])


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """The bounded mbarrier wait of the tensor-core kernels, on a barrier
    nothing arrives on (a flag nothing sets): it gives up after its limit,
    the error word carries 0x100, and the next optimizer step runs."""
    import ctypes
    import time
    from block_eigenbasis_preconditioning_gb300 import binding
    lib = binding.load_library()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = lib.dobb_selftest_wait_timeout(ctypes.cast(ctypes.c_void_p(err.data_ptr()),
                                                    ctypes.POINTER(ctypes.c_uint32)),
                                        ctypes.c_uint64(50_000_000), None)
    assert st == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) == 0x100
    assert 0.04 <= dt < 2.0
    shapes = [(64, 256)]
    Xs, Gs, Ws = make_problem(shapes, 512, 0.3, seed=43, param_dtype="bf16", act_dtype="bf16")
    opt = _dobb(shapes, 2, refresh_period=1, param_dtype="bf16", act_dtype="bf16")
    Wd = [to_dev(Ws[0], "bf16")]
    opt.accumulate([to_dev(Xs[0], "bf16")])
    opt.step(Wd, [to_dev(Gs[0], "bf16")], 0.02)
    torch.cuda.synchronize()
    assert opt.device_error() == 0 and np.all(opt.block_flags() == 0)
