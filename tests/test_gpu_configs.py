"""The workload configurations of the method, run on the GPU and scored
against the fp64 oracle on the same seeded inputs:

* a single fp32 768 x 768 matrix, B = 4 (k = 192), 10 steps, refresh every
  5 (tests/test_gpu_parity.py::test_single_matrix_ten_steps);
* the GPT-2 Small parameter set: 72 fp32 matrices, B = 16 (k = 48 / 192),
  4096 tokens per matrix at effective rank 20 %, refresh every 10, 50 steps;
* the refresh stress set: SPD blocks with relative eigenvalue gaps >= 1e-3
  and condition number 1e6 on GPT-2 XL shapes, refreshed at every step, at
  B = 16, 4 and 1 (k from 100 to 6400);
* the Llama-3-8B parameter set, B = 32 (k = 128 / 448), bf16: one layer and
  the two 128256-row matrices, with the update of those checked on sampled
  rows (each row's update depends on that row and the block bases only).

Every step is scored like the small cases: moments (relative Frobenius
1e-5 per block), bases at refresh steps (eigen residuals 1e-5), and the
update against the oracle run with the GPU's basis (sign band rule, W rule).
"""
import numpy as np
import pytest
import torch

from block_eigenbasis_preconditioning_gb300 import inputs as I
from oracle import dobb as O

from parity_util import check_bases, check_moments, check_update, to_dev, to_np

pytestmark = pytest.mark.gpu


def _dobb(*a, **k):
    from block_eigenbasis_preconditioning_gb300 import Dobb
    return Dobb(*a, **k)


def _streams(shapes, eff, rng):
    """One activation stream per matrix; matrices of one width share a Haar
    basis up to a row permutation and sign flips."""
    bases = {}
    out = []
    for (_, n), e in zip(shapes, eff):
        if n not in bases:
            bases[n] = I.haar_orthogonal(n, rng)
        out.append(I.ActivationStream(n, e, rng, shared_basis=bases[n]))
    return out


def test_gpt2_small_fifty_steps():
    """GPT-2 Small: 12 layers x {q, k, v, o 768 x 768; fc 3072 x 768; proj
    768 x 3072}, fp32 parameters, gradients and activations, B = 16, beta1
    0.95, beta2 0.99, lr 0.02, s 1, refresh every 10 steps, 50 steps.  The
    moments of every block are checked at every step, the bases at every
    refresh, the update of all 72 matrices at every fifth step and at the
    step after each refresh, and of one layer's matrices at the others."""
    ms = I.gpt2_small_shapes()
    shapes, B, N, T, steps = ms.shapes, 16, 4096, 10, 50
    rng = np.random.default_rng(60)
    streams = _streams(shapes, [0.20] * len(shapes), rng)
    opt = _dobb(shapes, B, beta1=0.95, beta2=0.99, refresh_period=T, scale_s=1.0)
    orc = O.DobbOracle(shapes, B, beta1=0.95, beta2=0.99, refresh_period=0)
    Wd = [to_dev(I.weights(m, n, rng), "f32") for m, n in shapes]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Wd]
    for t in range(steps):
        Xs = [s.draw(N, rng) for s in streams]
        Gs = [I.gradients_fp32(m, X, rng) for (m, _), X in zip(shapes, Xs)]
        Gd = [to_dev(g, "f32") for g in Gs]
        W_prev = [to_np(w) for w in Wd]
        M_prev = [m.copy() for m in orc.M]
        opt.accumulate([to_dev(x, "f32") for x in Xs])
        orc.accumulate(Xs)
        opt.step(Wd, Gd, 0.02, signs=Sd)
        torch.cuda.synchronize()
        assert opt.device_error() == 0
        check_moments(opt, orc, N=N)
        if t % T == 0:
            check_bases(opt, [to_np(opt.tensor("moments", i)) for i in range(len(shapes))])
            assert np.all(opt.block_flags() == 0)
        # every matrix's update at every fifth step (the refresh steps and the
        # steps right after them among them), one layer's six matrices otherwise
        full = t % 5 == 0 or t % T == 1
        for i, (m, n) in enumerate(shapes):
            if full or i // 6 == t % 12:
                check_update(W_prev[i], M_prev[i], Gs[i], to_np(opt.tensor("bases", i)),
                             to_np(Sd[i]), to_np(Wd[i]), to_np(opt.tensor("momentum", i)), 0.95,
                             0.02, 1.0, "f32", n // B)
            orc.M[i] = O.momentum(M_prev[i], Gs[i], 0.95)


def _stress_blocks(k, count, rng):
    return np.stack([I.spd_with_gap(k, rng, cond=1e6, min_rel_gap=1e-3)[0] for _ in range(count)])


@pytest.mark.parametrize("B", [16, 4])
def test_refresh_stress_every_step(B):
    """Refresh stress on GPT-2 XL layer shapes (q 1600 x 1600, fc 6400 x
    1600, proj 1600 x 6400): every block of every matrix re-eigensolved at
    every step (refresh period 1) from moments set to fresh SPD blocks with
    relative gaps >= 1e-3 and condition number 1e6 (k = 100 / 400 at B = 16,
    400 / 1600 at B = 4); two steps, the second warm-started from the first
    step's bases on new blocks."""
    shapes = [(1600, 1600), (6400, 1600), (1600, 6400)]
    rng = np.random.default_rng(61 + B)
    opt = _dobb(shapes, B, beta1=0.95, beta2=0.99, refresh_period=1, param_dtype="bf16",
                act_dtype="bf16")
    Wd = [to_dev(I.weights(m, n, rng, dtype="bf16"), "bf16") for m, n in shapes]
    for t in range(2):
        A = [_stress_blocks(n // B, B, rng) for _, n in shapes]
        for i, a in enumerate(A):
            opt.tensor("moments", i).copy_(torch.from_numpy(a.astype(np.float32)))
        Gd = [to_dev(rng.standard_normal((m, n)).astype(np.float32) * 1e-3, "bf16")
              for m, n in shapes]
        opt.step(Wd, Gd, 0.02)
        torch.cuda.synchronize()
        assert opt.device_error() == 0
        assert np.all(opt.block_flags() == 0)
        check_bases(opt, [a.astype(np.float32).astype(np.float64) for a in A])


def test_llama3_8b_layer_and_vocabulary_matrices():
    """Llama-3-8B shapes at B = 32 (k = 128 for n = 4096, 448 for n = 14336):
    one layer {q, o 4096 x 4096; k, v 1024 x 4096; gate, up 14336 x 4096;
    down 4096 x 14336} and the 128256 x 4096 embedding and head, bf16
    parameters, gradients and activations (4096 tokens, effective rank
    15 %), refresh every 20 steps; two steps.  Moments and bases of every
    block are checked; the update of the layer matrices in full and of the
    two vocabulary matrices on 4096 sampled rows plus the last row tile."""
    ms = I.llama3_8b_shapes()
    keep = [i for i, li in enumerate(ms.layer) if li in (0, 32)]
    shapes = [ms.shapes[i] for i in keep]
    B, N, T = 32, 4096, 20
    rng = np.random.default_rng(62)
    streams = _streams(shapes, [0.15] * len(shapes), rng)
    opt = _dobb(shapes, B, beta1=0.95, beta2=0.99, refresh_period=T, param_dtype="bf16",
                act_dtype="bf16")
    orc = O.DobbOracle(shapes, B, beta1=0.95, beta2=0.99, refresh_period=0)
    Wd = [to_dev(I.weights(m, n, rng, dtype="bf16"), "bf16") for m, n in shapes]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Wd]
    M_prev = [np.zeros((m, n), dtype=np.float32) for m, n in shapes]
    for t in range(2):
        Xs = [s.draw(N, rng, dtype="bf16") for s in streams]
        Gs = [I.gradients_fp32(m, X, rng, dtype="bf16") for (m, _), X in zip(shapes, Xs)]
        Gd = [to_dev(g, "bf16") for g in Gs]
        W_prev = [w.clone() for w in Wd]
        opt.accumulate([to_dev(x, "bf16") for x in Xs])
        orc.accumulate(Xs)
        opt.step(Wd, Gd, 0.02, signs=Sd)
        torch.cuda.synchronize()
        assert opt.device_error() == 0
        check_moments(opt, orc, N=N)
        if t % T == 0:
            # the eigensolver is scored on the moments it was given; the
            # moments were scored against the oracle just above
            check_bases(opt, [to_np(opt.tensor("moments", i)) for i in range(len(shapes))])
            assert np.all(opt.block_flags() == 0)
        for i, (m, n) in enumerate(shapes):
            rows = np.arange(m)
            if m > 20000:
                rows = np.unique(np.concatenate([rng.choice(m - 128, 4096, replace=False),
                                                 np.arange(m - 128, m)]))
            ridx = torch.from_numpy(rows).cuda()
            Q = to_np(opt.tensor("bases", i))
            check_update(to_np(W_prev[i][ridx]), M_prev[i][rows].astype(np.float64), Gs[i][rows], Q,
                         to_np(Sd[i][ridx]), to_np(Wd[i][ridx]),
                         to_np(opt.tensor("momentum", i)[ridx]), 0.95, 0.02, 1.0, "bf16", n // B)
            M_prev[i] = (0.95 * M_prev[i].astype(np.float64) + Gs[i]).astype(np.float32) \
                if m <= 20000 else to_np(opt.tensor("momentum", i)).astype(np.float32)


def test_refresh_stress_one_block_per_matrix_k6400():
    """The widest refresh-stress block: GPT-2 XL proj at B = 1 (k = 6400),
    an SPD block with relative gaps >= 1e-3 and condition number 1e6,
    eigensolved from the identity by the grid solver, scored with the eigen
    tolerances (residual, reconstruction, orthogonality, eigenvalues)."""
    k = 6400
    rng = np.random.default_rng(63)
    A = I.spd_with_gap(k, rng, cond=1e6, min_rel_gap=1e-3)[0]
    opt = _dobb([(4, k)], 1, refresh_period=0)
    opt.tensor("moments", 0).copy_(torch.from_numpy(A.astype(np.float32)).view(1, k, k))
    opt.refresh()
    torch.cuda.synchronize()
    assert np.all(opt.block_flags() == 0)
    check_bases(opt, [A.astype(np.float32).astype(np.float64)[None]])
