"""Parity of the grouped scheduler at model scale: handles whose launches
split into several chunks, and parameter matrices of embedding size, each
scored against the fp64 oracle like the small cases."""
import numpy as np
import pytest
import torch

from block_eigenbasis_preconditioning_gb300 import binding
from block_eigenbasis_preconditioning_gb300 import inputs as I
from oracle import dobb as O

from parity_util import check_bases, check_moments, check_update, to_dev, to_np

pytestmark = pytest.mark.gpu


def _dobb(*a, **k):
    from block_eigenbasis_preconditioning_gb300 import Dobb
    return Dobb(*a, **k)


def test_grouped_launches_over_270_matrices():
    """270 tensor-core-eligible matrices of mixed block widths (k = 16 ...
    200), bf16 activations and parameters: the moments run as two
    tensor-core launch chunks (at most 200 matrices each, the second with
    its own pointer-table base), the refresh and the update as grouped
    launches.  Every matrix's moments, bases and update against the oracle."""
    rng = np.random.default_rng(50)
    ks = [16, 48, 100, 128, 200]
    shapes = [(int(rng.integers(8, 140)), 2 * ks[i % len(ks)]) for i in range(270)]
    B = 2
    work = binding.describe_work(shapes, B, 1)
    assert len({e[2] for e in work if e[1] == 0}) == 2      # two chunk bases
    N = 1024
    Xs = [I.activations(N, n, 0.3, rng, dtype="bf16") for _, n in shapes]
    Gs = [I.gradients(m, X, rng, dtype="bf16") for (m, _), X in zip(shapes, Xs)]
    Ws = [I.weights(m, n, rng, dtype="bf16") for m, n in shapes]
    opt = _dobb(shapes, B, beta1=0.9, beta2=0.95, refresh_period=1, param_dtype="bf16",
                act_dtype="bf16")
    orc = O.DobbOracle(shapes, B, beta1=0.9, beta2=0.95, refresh_period=0)
    Wd = [to_dev(w, "bf16") for w in Ws]
    Gd = [to_dev(g, "bf16") for g in Gs]
    Sd = [torch.zeros(w.shape, dtype=torch.int8, device="cuda") for w in Ws]
    opt.accumulate([to_dev(x, "bf16") for x in Xs])
    orc.accumulate(Xs)
    opt.step(Wd, Gd, 0.02, signs=Sd)
    torch.cuda.synchronize()
    assert opt.device_error() == 0
    assert np.all(opt.block_flags() == 0)
    check_moments(opt, orc)
    check_bases(opt, orc.A)
    for i, (m, n) in enumerate(shapes):
        check_update(Ws[i], np.zeros((m, n)), to_np(Gd[i]), to_np(opt.tensor("bases", i)),
                     to_np(Sd[i]), to_np(Wd[i]), to_np(opt.tensor("momentum", i)), 0.9, 0.02, 1.0,
                     "bf16", n // B)


def test_embedding_sized_matrix_two_steps():
    """The GPT-2 XL token embedding as one Dobb matrix: 50257 x 1600, B = 16
    (k = 100), bf16 parameters, gradients and activations, two steps with a
    refresh before the first: moments, all 16 bases, and each update over
    all 80 M entries against the oracle with the GPU's basis."""
    m, n, B = 50257, 1600, 16
    rng = np.random.default_rng(51)
    opt = _dobb([(m, n)], B, beta1=0.95, beta2=0.99, refresh_period=2, param_dtype="bf16",
                act_dtype="bf16")
    orc = O.DobbOracle([(m, n)], B, beta1=0.95, beta2=0.99, refresh_period=0)
    W = I.weights(m, n, rng, dtype="bf16")
    Wd = to_dev(W, "bf16")
    Sd = torch.zeros((m, n), dtype=torch.int8, device="cuda")
    M_prev = np.zeros((m, n))
    for t in range(2):
        X = I.activations(2048, n, 0.10, rng, dtype="bf16")
        G = I.gradients(m, X, rng, dtype="bf16")
        Gd = to_dev(G, "bf16")
        W_prev = to_np(Wd)
        opt.accumulate([to_dev(X, "bf16")])
        orc.accumulate([X])
        opt.step([Wd], [Gd], 0.02, signs=[Sd])
        torch.cuda.synchronize()
        assert opt.device_error() == 0
        check_moments(opt, orc)
        if t == 0:
            check_bases(opt, orc.A)
        check_update(W_prev, M_prev, G, to_np(opt.tensor("bases", 0)), to_np(Sd), to_np(Wd),
                     to_np(opt.tensor("momentum", 0)), 0.95, 0.02, 1.0, "bf16", n // B)
        M_prev = O.momentum(M_prev, G, 0.95)
