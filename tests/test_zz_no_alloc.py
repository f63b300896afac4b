"""The allocation-free eigendecomposition entry point.

Some callers of this library cannot call cudaMalloc: runtimes whose device
memory is reserved up front by an arena they do not control, and plugins of
frameworks that forbid allocations outside their own allocator.
dobb_eigh_noalloc serves them from a fixed file-scope device array.  This
test calls it through the C ABI twice in a row, on different blocks, and
checks each result against the optimizer's own refresh (dobb_refresh_bases
on the same moments) within the eigen tolerance the other GPU tests use.
The file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

from block_eigenbasis_preconditioning_gb300 import binding
from block_eigenbasis_preconditioning_gb300 import inputs as I
from oracle import metrics as MX

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _blocks(k, count, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        if i % 2:
            X = I.activations(4 * k, k, 0.2, rng).astype(np.float64)
            A = X.T @ X / (4 * k)
        else:
            A = I.spd_with_gap(k, rng, cond=1e5)[0]
        out.append(A.astype(np.float32))
    return np.stack(out)


def _noalloc(A):
    lib = binding.load_library()
    count, k, _ = A.shape
    Ad = torch.from_numpy(A).cuda().contiguous()
    Qd = torch.empty_like(Ad)
    Ld = torch.empty(count, k, dtype=torch.float32, device="cuda")
    flags = (ctypes.c_uint32 * count)()
    st = lib.dobb_eigh_noalloc(ctypes.c_void_p(Ad.data_ptr()), ctypes.c_void_p(Qd.data_ptr()),
                               ctypes.c_void_p(Ld.data_ptr()), k, count, 40, flags,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.dobb_eigh_noalloc_last_error()
    torch.cuda.synchronize()
    return Qd.double().cpu().numpy(), Ld.double().cpu().numpy(), np.frombuffer(flags, np.uint32)


def _refresh(A):
    from block_eigenbasis_preconditioning_gb300 import Dobb
    count, k, _ = A.shape
    opt = Dobb([(8, count * k)], count, refresh_period=0)
    opt.tensor("moments", 0).copy_(torch.from_numpy(A).view(count, k, k))
    opt.refresh()
    torch.cuda.synchronize()
    return (opt.tensor("bases", 0).double().cpu().numpy(),
            opt.tensor("eigvals", 0).double().cpu().numpy())


@pytest.mark.parametrize("k,count", [(100, 6), (200, 3)])
def test_noalloc_matches_refresh_two_calls(k, count):
    for call, seed in enumerate((31, 32)):
        A = _blocks(k, count, seed)
        Qn, Ln, flags = _noalloc(A)
        Qr, Lr = _refresh(A)
        assert np.all(flags == 0)
        for b in range(count):
            A64 = A[b].astype(np.float64)
            fro = np.linalg.norm(A64)
            rn = MX.eig_residuals(A64, Qn[b], Ln[b])
            assert rn["recon"] <= TOL and rn["residual"] <= TOL, (call, b, rn)
            # same eigen-blocks and eigenvalues as the optimizer's refresh
            Bn = (Qn[b] * Ln[b][None, :]) @ Qn[b].T
            Br = (Qr[b] * Lr[b][None, :]) @ Qr[b].T
            assert np.linalg.norm(Bn - Br) / fro <= 2 * TOL
            assert np.abs(Ln[b] - Lr[b]).max() <= TOL * fro


def test_noalloc_rejects_oversized_requests():
    lib = binding.load_library()
    # 3 * 1024^2 * 2 floats > 4 Mi floats
    st = lib.dobb_eigh_noalloc(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                               1024, 2, 40, None, None)
    assert st == 1 and b"16 MiB" in lib.dobb_eigh_noalloc_last_error()
    st = lib.dobb_eigh_noalloc(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                               2048, 1, 40, None, None)
    assert st == 1
