"""`Dobb`: the optimizer over a list of weight matrices, on one GPU.

A thin object around one library handle.  It owns the state buffer (a
PyTorch uint8 tensor on the device) and passes raw device pointers and the
current CUDA stream to the C ABI; all arithmetic runs in the CUDA kernels.
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import torch

from .binding import (DTYPES, NORMS, REFRESH_METHODS, SIDES, TENSORS, _i64, _ptrs, check,
                      load_library)

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(int(s.cuda_stream))


class Dobb:
    """Dobb optimizer state and steps for matrices W_i of shape (m_i, n_i).

    Arguments follow the C ABI's dobb_create: B blocks per matrix, beta1,
    beta2, refresh_period (T, 0 = never automatic), scale_s (s in
    W <- W - lr s U), param_dtype of W / G and act_dtype of X ("f32" or
    "bf16"), basis_dtype of the basis the update multiplies with ("f32", or
    "bf16" as in the pages' principal setting), and the refresh method:
    "eigh" (complete eigendecomposition) or "orth" (orth_steps steps of
    orthogonal iteration with Cholesky QR, the pages' principal refresh), and
    the coefficient normalisation norm: "sign" (Dobb) or "l2" (Dobb-l2).

    side ("input", "output", or one of them per matrix) picks the axis the
    blocks cover: "input" is Dobb (blocks of W's n columns, accumulate takes
    input activations N x n), "output" is Dobb-G (blocks of W's m rows,
    accumulate takes output gradients N x m).  W, G and signs always keep
    the caller's (m, n) layout; the library registers an output-side matrix
    as its transpose, so its moments, bases and momentum views are those of
    W^T (blocks of width m / B, momentum n x m)."""

    def __init__(self, shapes: Sequence[Tuple[int, int]], B: int, beta1: float = 0.95,
                 beta2: float = 0.99, refresh_period: int = 10, scale_s: float = 1.0,
                 param_dtype: str = "f32", act_dtype: str = "f32",
                 device: Optional[torch.device] = None, stream: Optional[torch.cuda.Stream] = None,
                 basis_dtype: str = "f32", refresh: str = "eigh", orth_steps: int = 1,
                 norm: str = "sign", side="input"):
        self.lib = load_library()
        self.shapes = [(int(m), int(n)) for m, n in shapes]
        self.sides = [side] * len(self.shapes) if isinstance(side, str) else list(side)
        if len(self.sides) != len(self.shapes) or any(sd not in SIDES for sd in self.sides):
            raise ValueError(f"side must be 'input', 'output' or one per matrix, got {side!r}")
        # the problem the library sees: an output-side matrix is registered transposed
        self.reg_shapes = [(n, m) if sd == "output" else (m, n)
                           for (m, n), sd in zip(self.shapes, self.sides)]
        self.B = int(B)
        self.param_dtype = param_dtype
        self.act_dtype = act_dtype
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        ms = _i64([s[0] for s in self.reg_shapes])
        ns = _i64([s[1] for s in self.reg_shapes])
        nbytes = self.lib.dobb_state_bytes(len(self.shapes), ms, ns, self.B)
        if nbytes == 0:
            check(1)
        with torch.cuda.device(self.device):
            self.state = torch.empty(int(nbytes), dtype=torch.uint8, device=self.device)
            h = ctypes.c_void_p()
            check(self.lib.dobb_create(ctypes.byref(h), len(self.shapes), ms, ns, self.B,
                                       float(beta1), float(beta2), int(refresh_period),
                                       float(scale_s), DTYPES[param_dtype], DTYPES[act_dtype],
                                       ctypes.c_void_p(self.state.data_ptr()),
                                       ctypes.c_size_t(nbytes), _stream_ptr(stream)))
        self.handle = h
        self.num_blocks = int(self.lib.dobb_num_blocks(h))
        self.basis_dtype = basis_dtype
        if basis_dtype != "f32":
            check(self.lib.dobb_set_basis_dtype(h, DTYPES[basis_dtype], _stream_ptr(stream)))
        self.refresh_method = refresh
        if refresh != "eigh" or orth_steps != 1:
            check(self.lib.dobb_set_refresh(h, REFRESH_METHODS[refresh], int(orth_steps)))
        self.norm = norm
        if norm != "sign":
            check(self.lib.dobb_set_normalization(h, NORMS[norm]))
        for i, sd in enumerate(self.sides):
            if sd != "input":
                check(self.lib.dobb_set_side(h, i, SIDES[sd], _stream_ptr(stream)))

    # -- phases --------------------------------------------------------------
    def accumulate(self, X: Sequence[Optional[torch.Tensor]], stream=None) -> None:
        ptrs = _ptrs([None if x is None else x.data_ptr() for x in X])
        Ns = _i64([0 if x is None else x.shape[0] for x in X])
        check(self.lib.dobb_accumulate_moments(self.handle, ptrs, Ns, _stream_ptr(stream)))

    def refresh(self, stream=None) -> None:
        check(self.lib.dobb_refresh_bases(self.handle, _stream_ptr(stream)))

    def step(self, W: Sequence[torch.Tensor], G: Sequence[torch.Tensor], lr: float,
             signs: Optional[Sequence[Optional[torch.Tensor]]] = None, stream=None) -> None:
        wp = _ptrs([w.data_ptr() for w in W])
        gp = _ptrs([g.data_ptr() for g in G])
        if signs is None:
            check(self.lib.dobb_step(self.handle, wp, gp, ctypes.c_float(lr), _stream_ptr(stream)))
        else:
            sp = _ptrs([None if s is None else s.data_ptr() for s in signs])
            check(self.lib.dobb_step_with_signs(self.handle, wp, gp, ctypes.c_float(lr), sp,
                                                _stream_ptr(stream)))

    # -- state access ----------------------------------------------------------
    def tensor(self, which: str, matrix: int = -1) -> torch.Tensor:
        """A view into the state buffer: moments / bases (B, k, k), eigvals
        (B, k), momentum (m, n), flags (int32 per block), stats (blocks, 4).
        Shapes are those of the registered problem (W^T for an output-side
        matrix)."""
        ptr = ctypes.c_void_p()
        nbytes = ctypes.c_size_t()
        check(self.lib.dobb_state_tensor(self.handle, TENSORS[which], int(matrix),
                                         ctypes.byref(ptr), ctypes.byref(nbytes)))
        off = int(ptr.value) - self.state.data_ptr()
        raw = self.state[off:off + int(nbytes.value)]
        if which in ("flags", "error"):
            return raw.view(torch.int32)
        t = raw.view(torch.float32)
        if matrix < 0:
            return t
        m, n = self.reg_shapes[matrix]
        k = n // self.B
        if which in ("moments", "bases"):
            return t.view(self.B, k, k)
        if which == "eigvals":
            return t.view(self.B, k)
        if which == "momentum":
            return t.view(m, n)
        if which == "stats":
            return t.view(self.B, 4)
        return t

    @property
    def t(self) -> int:
        v = ctypes.c_int64()
        check(self.lib.dobb_get_step(self.handle, ctypes.byref(v)))
        return int(v.value)

    @t.setter
    def t(self, value: int) -> None:
        check(self.lib.dobb_set_step(self.handle, int(value)))

    def set_step_path(self, path: str = "auto") -> None:
        """"auto": tensor-core kernel where eligible; "ffma": FP32 FFMA kernel only."""
        check(self.lib.dobb_set_step_path(self.handle, {"auto": 0, "ffma": 1}[path]))

    def sync_bases(self, stream=None) -> None:
        check(self.lib.dobb_sync_bases(self.handle, _stream_ptr(stream)))

    def device_error(self) -> int:
        return int(self.tensor("error").item())

    def set_refresh_period(self, refresh_period: int) -> None:
        """Refresh every `refresh_period` steps from now on (0 = never)."""
        check(self.lib.dobb_set_refresh_period(self.handle, int(refresh_period)))

    def set_eig_grid(self, min_k: int, batch_bytes: int = 0) -> None:
        """Blocks at least `min_k` wide refresh with the grid eigensolver (0 =
        never), in batches of blocks of one width whose scratch fits
        `batch_bytes` (0 = all blocks of a width at once)."""
        check(self.lib.dobb_set_eig_grid(self.handle, int(min_k), int(batch_bytes)))

    def set_jacobi(self, max_sweeps: int = 40, tol: float = 0.0) -> None:
        check(self.lib.dobb_set_jacobi(self.handle, int(max_sweeps), float(tol)))

    def block_flags(self, stream=None):
        import numpy as np
        out = (ctypes.c_uint32 * self.num_blocks)()
        check(self.lib.dobb_get_block_flags(self.handle, out, _stream_ptr(stream)))
        return np.frombuffer(out, dtype=np.uint32).copy()

    def clear_flags(self, stream=None) -> None:
        check(self.lib.dobb_clear_block_flags(self.handle, _stream_ptr(stream)))

    def block_stats(self, stream=None):
        import numpy as np
        out = (ctypes.c_float * (4 * self.num_blocks))()
        check(self.lib.dobb_get_block_stats(self.handle, out, _stream_ptr(stream)))
        return np.frombuffer(out, dtype=np.float32).reshape(self.num_blocks, 4).copy()

    def check_bases(self, stream=None):
        import numpy as np
        out = (ctypes.c_float * (3 * self.num_blocks))()
        check(self.lib.dobb_check_bases(self.handle, out, _stream_ptr(stream)))
        return np.frombuffer(out, dtype=np.float32).reshape(self.num_blocks, 3).copy()

    def block_offset(self, matrix: int) -> int:
        return int(self.lib.dobb_block_offset(self.handle, int(matrix)))

    def checkpoint_bytes(self) -> int:
        return int(self.lib.dobb_checkpoint_bytes(self.handle))

    def get_state(self, stream=None):
        buf = torch.empty(self.checkpoint_bytes(), dtype=torch.uint8, device=self.device)
        t = ctypes.c_int64()
        check(self.lib.dobb_get_state(self.handle, ctypes.c_void_p(buf.data_ptr()),
                                      ctypes.c_size_t(buf.numel()), ctypes.byref(t),
                                      _stream_ptr(stream)))
        return buf, int(t.value)

    def set_state(self, buf: torch.Tensor, t: int, stream=None) -> None:
        check(self.lib.dobb_set_state(self.handle, ctypes.c_void_p(buf.data_ptr()),
                                      ctypes.c_size_t(buf.numel()), int(t), _stream_ptr(stream)))

    @property
    def launch_count(self) -> int:
        return int(self.lib.dobb_launch_count(self.handle))

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            check(self.lib.dobb_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
