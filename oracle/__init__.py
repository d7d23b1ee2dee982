"""CPU oracle -- test infrastructure only.

Thin ctypes/numpy marshalling around ``oracle.c`` (the plain, single-threaded
definitions of the fused AdamW step, the softmax backward and the LayerNorm
backward).  Only the test-suite, the smoke check and the benchmark's CPU
baseline leg may import this package; the product path never does.

No arithmetic of the methods lives here: every number is computed by the C
file, which is compiled with ``-O2 -ffp-contract=off`` so that the fp32 variant
rounds once per operation.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16 = 0, 1, 2
KIND = {"f32": F32, "f16": F16, "bf16": BF16}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (plain gcc, libm only)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _configure(lib):
    i64, i32 = ctypes.c_int64, ctypes.c_int
    f32, f64 = ctypes.c_float, ctypes.c_double
    vp = ctypes.c_void_p
    lib.orc_decode16.argtypes = [ctypes.c_uint16, i32]
    lib.orc_decode16.restype = f64
    lib.orc_encode16_rne.argtypes = [f64, i32]
    lib.orc_encode16_rne.restype = ctypes.c_uint16
    lib.orc_decode16_array.argtypes = [i64, vp, i32, vp]
    lib.orc_encode16_array.argtypes = [i64, vp, i32, vp]
    lib.orc_bias_correction.argtypes = [f32, i64]
    lib.orc_bias_correction.restype = f64
    lib.orc_adamw_step_f64.argtypes = [i64, vp, vp, vp, vp, i32, f64, i64,
                                       f32, f32, f32, f32, f32, vp, i32, vp]
    lib.orc_adamw_step_f32.argtypes = [i64, vp, vp, vp, vp, i32, f32, i64,
                                       f32, f32, f32, f32, f32, vp, i32, vp]
    for name in ("orc_softmax_bwd_f64", "orc_softmax_bwd_f32"):
        getattr(lib, name).argtypes = [i64, i64, vp, vp, vp]
    for name in ("orc_layernorm_bwd_f64", "orc_layernorm_bwd_f32"):
        getattr(lib, name).argtypes = [i64, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.orc_rmsnorm_bwd_f64.argtypes = [i64, i64, vp, vp, vp, vp, vp, vp]
    lib.orc_grad_sumsq_f64.argtypes = [i64, vp, i32, f64, ctypes.POINTER(i32)]
    lib.orc_grad_sumsq_f64.restype = f64
    lib.orc_clip_factor.argtypes = [f64, f64]
    lib.orc_clip_factor.restype = f64
    lib.orc_adamw_step_clipped_f64.argtypes = [i64, vp, vp, vp, vp, i32, f64, f64, i32, i64,
                                               f32, f32, f32, f32, f32, vp, i32, vp]
    lib.orc_cast_to_f32.argtypes = [i64, vp, i32, f32, vp]
    lib.orc_cast_from_f32.argtypes = [i64, vp, i32, vp]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _configure(ctypes.CDLL(_LIB_PATH))
    return _lib


@contextlib.contextmanager
def swapped_library(path: str):
    """Temporarily route every wrapper through another build of ``oracle.c``
    (the tests use this to plant a mistake in a copy and check a pin fails)."""
    global _lib
    saved = _load()
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def source_path() -> str:
    return _SRC


def compile_variant(src_text: str, out_dir: str, name: str) -> str:
    """Compile a (modified) copy of the oracle source with the same flags."""
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", c, "-o", so, "-lm"], check=True)
    return so


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- codecs
def decode16(bits, kind: str) -> np.ndarray:
    """Exact float64 values of 16-bit patterns (``kind`` is "f16" or "bf16")."""
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().orc_decode16_array(b.size, _ptr(b), KIND[kind], _ptr(out))
    return out


def encode16(x, kind: str) -> np.ndarray:
    """Round float64 values to 16-bit patterns, nearest-even."""
    a = _c(x, np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().orc_encode16_array(a.size, _ptr(a), KIND[kind], _ptr(out))
    return out


def bias_correction(beta: float, t: int) -> float:
    return _load().orc_bias_correction(beta, t)


# --------------------------------------------------------------------------- AdamW
def adamw_step_f64(theta, m, v, grad_bits, grad_kind, inv_loss_scale, t,
                   lr, beta1, beta2, eps, weight_decay, copy_kind="bf16"):
    """One AdamW step in double.  ``theta, m, v`` are float64 arrays updated in
    place; returns ``(copy_bits, zeroed_grad_bits)``."""
    for a in (theta, m, v):
        assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    g = _c(grad_bits, np.uint16)
    n = theta.size
    assert m.size == n and v.size == n and g.size == n
    copy = np.empty(n, np.uint16)
    gout = np.empty(n, np.uint16)
    _load().orc_adamw_step_f64(n, _ptr(theta), _ptr(m), _ptr(v), _ptr(g),
                               KIND[grad_kind], float(inv_loss_scale), int(t),
                               lr, beta1, beta2, eps, weight_decay,
                               _ptr(copy), KIND[copy_kind], _ptr(gout))
    return copy, gout


def adamw_step_f32(theta, m, v, grad_bits, grad_kind, inv_loss_scale, t,
                   lr, beta1, beta2, eps, weight_decay, copy_kind="bf16"):
    """One AdamW step in IEEE fp32, one rounding per operation (float32 arrays
    updated in place); returns ``(copy_bits, zeroed_grad_bits)``."""
    for a in (theta, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    g = _c(grad_bits, np.uint16)
    n = theta.size
    copy = np.empty(n, np.uint16)
    gout = np.empty(n, np.uint16)
    _load().orc_adamw_step_f32(n, _ptr(theta), _ptr(m), _ptr(v), _ptr(g),
                               KIND[grad_kind], float(inv_loss_scale), int(t),
                               lr, beta1, beta2, eps, weight_decay,
                               _ptr(copy), KIND[copy_kind], _ptr(gout))
    return copy, gout


# --------------------------------------------------------------------------- grad-norm clipping
def grad_norm_f64(grad_bits_list, kind, inv_loss_scale):
    """Global L2 norm of the unscaled gradients of several tensors, and whether any
    element is non-finite.  Returns ``(norm, nonfinite)``."""
    flag = ctypes.c_int(0)
    total = 0.0
    for gb in grad_bits_list:
        g = _c(gb, np.uint16)
        total += _load().orc_grad_sumsq_f64(g.size, _ptr(g), KIND[kind], float(inv_loss_scale),
                                            ctypes.byref(flag))
    return float(np.sqrt(total)), bool(flag.value)


def clip_factor(norm, max_norm) -> float:
    return _load().orc_clip_factor(float(norm), float(max_norm))


def adamw_step_clipped_f64(theta, m, v, grad_bits, grad_kind, inv_loss_scale, clip, skip, t,
                           lr, beta1, beta2, eps, weight_decay, copy_kind="bf16", copy_in=None):
    """AdamW step on the clipped gradient (see oracle.c); same conventions as
    ``adamw_step_f64``.  ``copy_in`` is the working copy before the step (returned
    unchanged when the step is skipped); zeros if omitted."""
    for a in (theta, m, v):
        assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    g = _c(grad_bits, np.uint16)
    n = theta.size
    copy = np.zeros(n, np.uint16) if copy_in is None else _c(copy_in, np.uint16).copy()
    gout = np.empty(n, np.uint16)
    _load().orc_adamw_step_clipped_f64(n, _ptr(theta), _ptr(m), _ptr(v), _ptr(g),
                                       KIND[grad_kind], float(inv_loss_scale), float(clip),
                                       int(bool(skip)), int(t), lr, beta1, beta2, eps,
                                       weight_decay, _ptr(copy), KIND[copy_kind], _ptr(gout))
    return copy, gout


# --------------------------------------------------------------------------- casts
def cast_to_f32(src, kind: str, scale: float) -> np.ndarray:
    """float32(src * scale); ``src`` holds 16-bit patterns (kind f16/bf16) or float32."""
    a = _c(src, np.float32 if kind == "f32" else np.uint16)
    out = np.empty(a.shape, np.float32)
    _load().orc_cast_to_f32(a.size, _ptr(a), KIND[kind], float(scale), _ptr(out))
    return out


def cast_from_f32(src, kind: str) -> np.ndarray:
    a = _c(src, np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().orc_cast_from_f32(a.size, _ptr(a), KIND[kind], _ptr(out))
    return out


# --------------------------------------------------------------------------- softmax bwd
def softmax_bwd_f64(dY, P) -> np.ndarray:
    dY = _c(dY, np.float64)
    P = _c(P, np.float64)
    assert dY.shape == P.shape and dY.ndim == 2
    out = np.empty_like(dY)
    _load().orc_softmax_bwd_f64(dY.shape[0], dY.shape[1], _ptr(dY), _ptr(P), _ptr(out))
    return out


def softmax_bwd_f32(dY, P) -> np.ndarray:
    dY = _c(dY, np.float32)
    P = _c(P, np.float32)
    assert dY.shape == P.shape and dY.ndim == 2
    out = np.empty_like(dY)
    _load().orc_softmax_bwd_f32(dY.shape[0], dY.shape[1], _ptr(dY), _ptr(P), _ptr(out))
    return out


# --------------------------------------------------------------------------- LayerNorm bwd
def layernorm_bwd_f64(dY, x, mean, inv_std, gamma):
    """Returns ``(dX, dgamma, dbeta)`` in float64."""
    dY = _c(dY, np.float64)
    x = _c(x, np.float64)
    mean = _c(mean, np.float64)
    inv_std = _c(inv_std, np.float64)
    gamma = _c(gamma, np.float64)
    rows, D = x.shape
    assert dY.shape == x.shape and mean.shape == (rows,) and inv_std.shape == (rows,)
    assert gamma.shape == (D,)
    dX = np.empty_like(x)
    dg = np.empty(D, np.float64)
    db = np.empty(D, np.float64)
    _load().orc_layernorm_bwd_f64(rows, D, _ptr(dY), _ptr(x), _ptr(mean), _ptr(inv_std),
                                  _ptr(gamma), _ptr(dX), _ptr(dg), _ptr(db))
    return dX, dg, db


def layernorm_bwd_f32(dY, x, mean, inv_std, gamma):
    """Returns ``(dX, dgamma, dbeta)`` in float32."""
    dY = _c(dY, np.float32)
    x = _c(x, np.float32)
    mean = _c(mean, np.float32)
    inv_std = _c(inv_std, np.float32)
    gamma = _c(gamma, np.float32)
    rows, D = x.shape
    dX = np.empty_like(x)
    dg = np.empty(D, np.float32)
    db = np.empty(D, np.float32)
    _load().orc_layernorm_bwd_f32(rows, D, _ptr(dY), _ptr(x), _ptr(mean), _ptr(inv_std),
                                  _ptr(gamma), _ptr(dX), _ptr(dg), _ptr(db))
    return dX, dg, db


# --------------------------------------------------------------------------- RMSNorm bwd
def rmsnorm_bwd_f64(dY, x, inv_rms, gamma):
    """Returns ``(dX, dgamma)`` in float64."""
    dY = _c(dY, np.float64)
    x = _c(x, np.float64)
    inv_rms = _c(inv_rms, np.float64)
    gamma = _c(gamma, np.float64)
    rows, D = x.shape
    assert dY.shape == x.shape and inv_rms.shape == (rows,) and gamma.shape == (D,)
    dX = np.empty_like(x)
    dg = np.empty(D, np.float64)
    _load().orc_rmsnorm_bwd_f64(rows, D, _ptr(dY), _ptr(x), _ptr(inv_rms), _ptr(gamma),
                                _ptr(dX), _ptr(dg))
    return dX, dg


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
