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


def _check_work_lists(shapes, B):
    """Every unit of every phase appears exactly once in the scheduler's
    lists, and every launch addresses its matrices within the slots of its
    pointer table (512 matrices; 200 for the tensor-core moments launch,
    whose activation tensor maps travel in the parameter block)."""
    from collections import defaultdict
    # update: the row tiles of every (matrix, block) partition [0, m)
    upd = binding.describe_work(shapes, B, 0)
    rows = defaultdict(list)
    kinds = defaultdict(set)
    for launch, kind, base, mat, blk, a, b in upd:
        assert 0 <= mat - base < 512
        assert b >= 1 and (kind == 1 or b <= 128)
        rows[(mat, blk)].append((a, a + b))
        kinds[mat].add(kind)
    assert len(rows) == len(shapes) * B
    for (mat, blk), iv in rows.items():
        iv.sort()
        assert iv[0][0] == 0 and iv[-1][1] == shapes[mat][0]
        assert all(x[1] == y[0] for x, y in zip(iv, iv[1:])), (mat, blk, iv[:4])
        assert len(kinds[mat]) == 1
    # moments: tensor-core units partition each block's 128-row slices; FFMA
    # tiles cover the upper triangle of 64 x 64 tiles once
    acc = binding.describe_work(shapes, B, 1)
    units = defaultdict(list)
    per_launch = defaultdict(set)
    for launch, kind, base, mat, blk, a, b in acc:
        units[(mat, blk, kind)].append((a, b))
        per_launch[launch].add((kind, base))
        assert 0 <= mat - base < (200 if kind == 0 else 512)
    assert all(len(v) == 1 for v in per_launch.values())
    seen = set()
    for (mat, blk, kind), v in units.items():
        k = shapes[mat][1] // B
        seen.add((mat, blk))
        if kind == 0:
            d = (blk * k) & 7
            ns = (k + d + 127) // 128
            v.sort()
            assert v[0][0] == 0 and v[-1][1] == ns and all(x[1] == y[0] for x, y in zip(v, v[1:]))
            assert all(b > a for a, b in v)
        else:
            nt = (k + 63) // 64
            assert sorted(v) == [(i, j) for i in range(nt) for j in range(i, nt)]
    assert len(seen) == len(shapes) * B
    # refresh: every block once
    eig = binding.describe_work(shapes, B, 2)
    assert sorted((e[3], e[4]) for e in eig) == [(i, b) for i in range(len(shapes)) for b in range(B)]
    assert all(0 <= e[3] - e[2] < 512 for e in eig)
    return upd, acc, eig


def test_work_lists_cover_every_unit():
    """The grouped scheduler over 600 mixed matrices (two 512-matrix launch
    chunks, four tensor-core moment chunks of <= 200 matrices, blocks of
    width 5 ... 400 and ragged row counts): every unit of every phase once."""
    widths = [64, 400, 1600, 36, 20, 1792]          # B = 4: k = 16, 100, 400, 9, 5, 448
    shapes = [(1 + (37 * i) % 300, widths[i % len(widths)]) for i in range(600)]
    upd, acc, eig = _check_work_lists(shapes, 4)
    assert len({e[0] for e in eig}) == 2                       # 512 + 88 matrices
    assert len({e[2] for e in acc if e[1] == 0}) >= 3          # several moment chunks
    assert {e[1] for e in upd} == {0, 1} and {e[1] for e in acc} == {0, 1}


def test_work_lists_of_the_gpt2_xl_set():
    """The 289-matrix GPT-2 XL set at B = 16, with the 50257-row embedding:
    two tensor-core moment chunks, one update chunk."""
    from block_eigenbasis_preconditioning_gb300 import inputs as I
    ms_ = I.gpt2_xl_shapes()
    upd, acc, eig = _check_work_lists(ms_.shapes, 16)
    assert len({e[2] for e in acc}) == 2
    emb = [i for i, (m, n) in enumerate(ms_.shapes) if m == 50257]
    assert len(emb) == 1
    assert sum(1 for e in upd if e[3] == emb[0]) == 16 * ((50257 + 127) // 128)


def test_describe_work_rejects_bad_arguments():
    lib = binding.load_library()
    ms, ns = _shape_args([(8, 30)])
    assert lib.dobb_describe_work(1, ms, ns, 4, 0, None, 0) == -1
    assert b"divisible" in lib.dobb_last_error()
    ms, ns = _shape_args([(8, 32)])
    assert lib.dobb_describe_work(1, ms, ns, 4, 3, None, 0) == -1


def test_noalloc_eigh_rejects_overlapping_outputs_without_device():
    """The allocation-free eigensolver writes the identity into Q before it
    reads A, so an output that overlaps the input is refused before any
    device work (fake addresses: the checks run first)."""
    lib = binding.load_library()
    k, count = 8, 2
    nbytes = 4 * count * k * k
    base = 1 << 20
    # Q_dev == A_dev (in place)
    st = lib.dobb_eigh_noalloc(ctypes.c_void_p(base), ctypes.c_void_p(base),
                               ctypes.c_void_p(base + 4 * nbytes), k, count, 40, None, None)
    assert st == 1 and b"overlap" in lib.dobb_eigh_noalloc_last_error()
    # lam_dev inside A's last block
    st = lib.dobb_eigh_noalloc(ctypes.c_void_p(base), ctypes.c_void_p(base + 2 * nbytes),
                               ctypes.c_void_p(base + nbytes - 16), k, count, 40, None, None)
    assert st == 1 and b"overlap" in lib.dobb_eigh_noalloc_last_error()
    # Q_dev ending exactly where A_dev starts is fine up to the device checks,
    # which a count of 0 skips entirely
    st = lib.dobb_eigh_noalloc(ctypes.c_void_p(base), ctypes.c_void_p(base - nbytes),
                               ctypes.c_void_p(base + nbytes), k, 0, 40, None, None)
    assert st == 0
