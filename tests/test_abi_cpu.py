"""C-ABI checks that need no GPU.

libtb.so must load, export every function include/tb.h declares, and reject
bad arguments synchronously -- these checks all return before any CUDA call, so
they run on a machine without a GPU (the pointers below are never dereferenced).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TB_OK, INVALID, DTYPE, MISALIGNED, ALIAS, WORKSPACE = 0, 1, 2, 3, 4, 5
F32, F16, BF16 = 0, 1, 2


@pytest.fixture(scope="module")
def tb():
    import __graft_entry__
    __graft_entry__.build()
    import ln_backward_gb300
    return ln_backward_gb300


def declared_functions():
    text = open(os.path.join(ROOT, "include", "tb.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tb_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for want in ("tb_adamw_plan_create", "tb_adamw_step", "tb_adamw_plan_destroy",
                 "tb_softmax_bwd", "tb_layernorm_bwd_workspace_size", "tb_layernorm_bwd"):
        assert want in names


def test_library_exports_every_declared_symbol(tb):
    lib = ctypes.CDLL(tb.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), f"libtb.so does not export {name}"
    assert set(declared_functions()) == set(tb.EXPORTS)


def test_status_strings(tb):
    for code, name in tb.STATUS.items():
        assert tb.tb_status_string(code) == name
    assert tb.tb_version() >= 100


# ----------------------------------------------------------------------------- softmax
def _sm(tb, dY, P, dX, rows, cols, dt):
    return tb._binding.lib.tb_softmax_bwd(dY, P, dX, rows, cols, dt, None)


def test_softmax_validation(tb):
    A, B, C = 0x10000, 0x20000, 0x30000          # disjoint fake device addresses
    assert _sm(tb, A, B, C, -1, 4, F32) == INVALID
    assert _sm(tb, A, B, C, 4, -1, F32) == INVALID
    assert _sm(tb, A, B, C, 4, 4, 7) == DTYPE
    assert _sm(tb, A, B, C, 0, 4, F32) == TB_OK          # empty: nothing enqueued
    assert _sm(tb, A, B, C, 4, 0, F32) == TB_OK
    assert _sm(tb, None, B, C, 4, 4, F32) == INVALID
    assert _sm(tb, A + 2, B, C, 4, 4, F32) == MISALIGNED
    assert _sm(tb, A + 1, B, C, 4, 4, BF16) == MISALIGNED
    assert _sm(tb, A, B, A, 4, 4, F32) == ALIAS          # dX == dY
    assert _sm(tb, A, B, B + 8, 4, 4, F32) == ALIAS      # dX overlaps P


# ----------------------------------------------------------------------------- AdamW
def _desc(tb, p, m, v, g, c, n):
    return tb._binding.tb_tensor_desc(p, m, v, g, c, n)


def _create(tb, descs, gdt=BF16, cdt=BF16):
    arr = (tb._binding.tb_tensor_desc * len(descs))(*descs)
    h = ctypes.c_void_p(None)
    return tb._binding.lib.tb_adamw_plan_create(arr, len(descs), gdt, cdt, ctypes.byref(h))


def test_adamw_plan_validation(tb):
    lib = tb._binding.lib
    base = 1 << 20
    ok = _desc(tb, base, base + 4096, base + 8192, base + 12288, base + 14336, 1024)
    h = ctypes.c_void_p(None)
    assert lib.tb_adamw_plan_create(None, 1, BF16, BF16, ctypes.byref(h)) == INVALID
    arr = (tb._binding.tb_tensor_desc * 1)(ok)
    assert lib.tb_adamw_plan_create(arr, 0, BF16, BF16, ctypes.byref(h)) == INVALID
    assert lib.tb_adamw_plan_create(arr, 1, BF16, BF16, None) == INVALID
    assert _create(tb, [ok], gdt=7) == DTYPE
    assert _create(tb, [ok], cdt=F32) == DTYPE
    assert _create(tb, [_desc(tb, base, base + 4096, base + 8192, base + 12288, base + 14336, -1)]) == INVALID
    assert _create(tb, [_desc(tb, None, base + 4096, base + 8192, base + 12288, base + 14336, 8)]) == INVALID
    assert _create(tb, [_desc(tb, base + 2, base + 4096, base + 8192, base + 12288, base + 14336, 8)]) == MISALIGNED
    assert _create(tb, [_desc(tb, base, base + 4096, base + 8192, base + 12289, base + 14336, 8)]) == MISALIGNED
    # m overlaps param
    assert _create(tb, [_desc(tb, base, base + 2048, base + 8192, base + 12288, base + 14336, 1024)]) == ALIAS
    # fp32 gradients must be 4-byte aligned
    assert _create(tb, [_desc(tb, base, base + 4096, base + 8192, base + 12290, None, 8)],
                   gdt=F32) == MISALIGNED
    # working copies for some tensors only
    other_nc = _desc(tb, base + 65536, base + 69632, base + 73728, base + 77824, None, 64)
    assert _create(tb, [ok, other_nc]) == INVALID
    # two tensors sharing a grad buffer
    other = _desc(tb, base + 65536, base + 69632, base + 73728, base + 12288, base + 81920, 64)
    assert _create(tb, [ok, other]) == ALIAS


def test_adamw_step_rejects_null_plan(tb):
    lib = tb._binding.lib
    hp = tb._binding.tb_adamw_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert lib.tb_adamw_step(None, 1, ctypes.byref(hp), 1.0, None) == INVALID
    assert lib.tb_adamw_plan_destroy(None) == TB_OK


def test_pointers_that_are_not_live_plans_are_never_dereferenced(tb):
    """Handles are looked up among the live plans first: a pointer that was never a
    plan (here an address with nothing mapped behind it) is rejected, not read."""
    lib = tb._binding.lib
    hp = tb._binding.tb_adamw_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    bogus = ctypes.c_void_p(0x1000)
    size = ctypes.c_size_t(0)
    assert lib.tb_adamw_step(bogus, 1, ctypes.byref(hp), 1.0, None) == INVALID
    assert lib.tb_adamw_step_clipped(bogus, 1, ctypes.byref(hp), 1.0, 0x2000, None) == INVALID
    assert lib.tb_adamw_grad_norm_workspace_size(bogus, ctypes.byref(size)) == INVALID
    assert lib.tb_adamw_grad_norm(bogus, 1.0, 1.0, 0x2000, 0x3000, 64, None) == INVALID
    assert lib.tb_adamw_step_device(bogus, 0x2000, ctypes.byref(hp), 1.0, None, None) == INVALID
    assert lib.tb_adamw_step_device(None, None, ctypes.byref(hp), 1.0, None, None) == INVALID
    assert lib.tb_adamw_selftest_stale_counter(bogus, 5, None) == INVALID
    assert lib.tb_adamw_selftest_stale_counter(None, 5, None) == INVALID
    assert lib.tb_adamw_plan_destroy(bogus) == INVALID


# ----------------------------------------------------------------------------- LayerNorm
def _ln(tb, dY, x, mean, rstd, gamma, dX, dg, db, rows, D, dt, ws, wsb):
    return tb._binding.lib.tb_layernorm_bwd(dY, x, mean, rstd, gamma, dX, dg, db, rows, D, dt,
                                             ws, wsb, None)


def test_layernorm_validation(tb):
    b = 1 << 24
    dY, x, mean, rstd, gamma = b, b + 0x100000, b + 0x200000, b + 0x210000, b + 0x220000
    dX, dg, db, ws = b + 0x300000, b + 0x400000, b + 0x410000, b + 0x500000
    args = [dY, x, mean, rstd, gamma, dX, dg, db]
    assert _ln(tb, *args, -1, 16, F32, ws, 1 << 20) == INVALID
    assert _ln(tb, *args, 4, -1, F32, ws, 1 << 20) == INVALID
    assert _ln(tb, *args, 4, 16, 9, ws, 1 << 20) == DTYPE
    assert _ln(tb, *args, 4, 0, F32, ws, 1 << 20) == TB_OK         # D == 0: nothing to do
    bad = list(args)
    bad[6] = None
    assert _ln(tb, *bad, 4, 16, F32, ws, 1 << 20) == INVALID       # dgamma NULL
    bad = list(args)
    bad[5] = dY                                                     # dX == dY
    assert _ln(tb, *bad, 4, 16, F32, ws, 1 << 20) == ALIAS
    bad = list(args)
    bad[7] = dg + 32                                                # dbeta overlaps dgamma
    assert _ln(tb, *bad, 4, 16, F32, ws, 1 << 20) == ALIAS
    assert _ln(tb, *args, 4, 16, F32, dX + 64, 1 << 20) == ALIAS    # workspace overlaps dX
    bad = list(args)
    bad[1] = x + 2
    assert _ln(tb, *bad, 4, 16, F32, ws, 1 << 20) == MISALIGNED


def test_layernorm_workspace_query_validation(tb):
    lib = tb._binding.lib
    out = ctypes.c_size_t(123)
    assert lib.tb_layernorm_bwd_workspace_size(4, 16, F32, None) == INVALID
    assert lib.tb_layernorm_bwd_workspace_size(-1, 16, F32, ctypes.byref(out)) == INVALID
    assert lib.tb_layernorm_bwd_workspace_size(4, 16, 5, ctypes.byref(out)) == DTYPE
    assert lib.tb_layernorm_bwd_workspace_size(0, 16, F32, ctypes.byref(out)) == TB_OK
    assert out.value == 0


def test_product_path_does_not_touch_the_oracle():
    """The library and its binding must never load, import or link the oracle."""
    pkg = os.path.join(ROOT, "ln_backward_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text and "oracle.c" not in text, f


def test_cast_validation(tb):
    lib = tb._binding.lib
    A, B = 0x10000, 0x40000
    assert lib.tb_cast_to_f32(A, F16, 1.0, B, -1, None) == INVALID
    assert lib.tb_cast_to_f32(A, 9, 1.0, B, 4, None) == DTYPE
    assert lib.tb_cast_to_f32(A, F16, 1.0, B, 0, None) == TB_OK
    assert lib.tb_cast_to_f32(A + 1, F16, 1.0, B, 4, None) == MISALIGNED
    assert lib.tb_cast_to_f32(A, F16, 1.0, A + 4, 4, None) == ALIAS
    assert lib.tb_cast_from_f32(A, B, F32, 4, None) == DTYPE
    assert lib.tb_cast_from_f32(A, A + 2, BF16, 4, None) == ALIAS
    assert lib.tb_cast_from_f32(None, B, BF16, 4, None) == INVALID
    # element counts whose byte ranges would overflow are rejected before any CUDA call
    assert lib.tb_cast_to_f32(A, F16, 1.0, B, 2**62, None) == INVALID
    assert lib.tb_cast_from_f32(A, B, BF16, 2**62, None) == INVALID


def test_selftest_limit_validation(tb):
    lib = tb._binding.lib
    for bad in (-1, 0, 999, 1_000_000_001):
        assert lib.tb_layernorm_bwd_selftest_timeout(bad, None) == INVALID
