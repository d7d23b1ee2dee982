"""ctypes binding over libtb.so -- argument marshalling only.

Every function here carries the name of the C entry point it calls, turns
torch tensors into (pointer, size, dtype) arguments, passes torch's current
CUDA stream unless one is given, and raises ``TbError`` on a non-OK status.
No arithmetic of the kernels happens in Python, and there is no fallback:
if libtb.so is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtb.so")

TB_F32, TB_F16, TB_BF16 = 0, 1, 2
_DTYPE = {torch.float32: TB_F32, torch.float16: TB_F16, torch.bfloat16: TB_BF16}

STATUS = {0: "TB_OK", 1: "TB_ERR_INVALID_VALUE", 2: "TB_ERR_UNSUPPORTED_DTYPE",
          3: "TB_ERR_MISALIGNED", 4: "TB_ERR_ALIAS", 5: "TB_ERR_WORKSPACE", 6: "TB_ERR_OOM",
          7: "TB_ERR_CUDA", 8: "TB_ERR_DEVICE", 9: "TB_ERR_TIMEOUT"}

# Every symbol include/tb.h declares.
EXPORTS = ("tb_status_string", "tb_version", "tb_device_error", "tb_adamw_plan_create",
           "tb_adamw_step", "tb_adamw_plan_destroy", "tb_softmax_bwd",
           "tb_layernorm_bwd_workspace_size", "tb_layernorm_bwd", "tb_layernorm_bwd_noalloc",
           "tb_softmax_bwd_causal", "tb_rmsnorm_bwd_workspace_size", "tb_rmsnorm_bwd",
           "tb_adamw_grad_norm_workspace_size", "tb_adamw_grad_norm", "tb_adamw_step_clipped",
           "tb_cast_to_f32", "tb_cast_from_f32", "tb_layernorm_bwd_selftest_timeout",
           "tb_adamw_step_device", "tb_adamw_selftest_stale_counter")


class TbError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


class tb_tensor_desc(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("grad", ctypes.c_void_p), ("copy", ctypes.c_void_p), ("n", ctypes.c_int64)]


class tb_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


def _load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -c 'import __graft_entry__ as g; "
                          "g.build()'` (needs nvcc) -- there is no CPU fallback")
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.tb_status_string.argtypes = [i32]
    lib.tb_status_string.restype = ctypes.c_char_p
    lib.tb_version.argtypes = []
    lib.tb_version.restype = i32
    lib.tb_device_error.argtypes = [ctypes.POINTER(i32), i32]
    lib.tb_device_error.restype = i32
    lib.tb_adamw_plan_create.argtypes = [ctypes.POINTER(tb_tensor_desc), i32, i32, i32,
                                         ctypes.POINTER(vp)]
    lib.tb_adamw_plan_create.restype = i32
    lib.tb_adamw_step.argtypes = [vp, i64, ctypes.POINTER(tb_adamw_hparams), f32, vp]
    lib.tb_adamw_step.restype = i32
    lib.tb_adamw_plan_destroy.argtypes = [vp]
    lib.tb_adamw_plan_destroy.restype = i32
    lib.tb_softmax_bwd.argtypes = [vp, vp, vp, i64, i64, i32, vp]
    lib.tb_softmax_bwd.restype = i32
    lib.tb_layernorm_bwd_workspace_size.argtypes = [i64, i64, i32, ctypes.POINTER(ctypes.c_size_t)]
    lib.tb_layernorm_bwd_workspace_size.restype = i32
    lib.tb_layernorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, vp,
                                     ctypes.c_size_t, vp]
    lib.tb_layernorm_bwd.restype = i32
    lib.tb_layernorm_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, vp]
    lib.tb_layernorm_bwd_noalloc.restype = i32
    lib.tb_softmax_bwd_causal.argtypes = [vp, vp, vp, i64, i64, i64, i64, i32, vp]
    lib.tb_softmax_bwd_causal.restype = i32
    lib.tb_rmsnorm_bwd_workspace_size.argtypes = [i64, i64, i32, ctypes.POINTER(ctypes.c_size_t)]
    lib.tb_rmsnorm_bwd_workspace_size.restype = i32
    lib.tb_rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i32, vp, ctypes.c_size_t, vp]
    lib.tb_rmsnorm_bwd.restype = i32
    lib.tb_adamw_grad_norm_workspace_size.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
    lib.tb_adamw_grad_norm_workspace_size.restype = i32
    lib.tb_adamw_grad_norm.argtypes = [vp, f32, f32, vp, vp, ctypes.c_size_t, vp]
    lib.tb_adamw_grad_norm.restype = i32
    lib.tb_adamw_step_clipped.argtypes = [vp, i64, ctypes.POINTER(tb_adamw_hparams), f32, vp, vp]
    lib.tb_adamw_step_clipped.restype = i32
    lib.tb_cast_to_f32.argtypes = [vp, i32, f32, vp, i64, vp]
    lib.tb_cast_to_f32.restype = i32
    lib.tb_cast_from_f32.argtypes = [vp, vp, i32, i64, vp]
    lib.tb_cast_from_f32.restype = i32
    lib.tb_adamw_step_device.argtypes = [vp, vp, ctypes.POINTER(tb_adamw_hparams), f32, vp, vp]
    lib.tb_adamw_step_device.restype = i32
    lib.tb_layernorm_bwd_selftest_timeout.argtypes = [i64, vp]
    lib.tb_layernorm_bwd_selftest_timeout.restype = i32
    lib.tb_adamw_selftest_stale_counter.argtypes = [vp, ctypes.c_uint64, vp]
    lib.tb_adamw_selftest_stale_counter.restype = i32
    return lib


lib = _load_library()


def library_path() -> str:
    return _LIB_PATH


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise TbError(fn, code)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    """Device pointer of a contiguous CUDA tensor on the current device (the C entry
    points take device pointers and launch on the current device)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libtb must be CUDA tensors")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libtb must be contiguous")
    return t.data_ptr() if t.numel() > 0 else (t.data_ptr() or None)


def _want(t: torch.Tensor, n: int, dtype: torch.dtype, name: str) -> None:
    """The kernels index `t` by the sizes of the other arguments: check it holds them."""
    if t.numel() != n or t.dtype != dtype:
        raise ValueError(f"{name} must hold {n} {dtype} values, got {t.numel()} {t.dtype}")


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPE[t.dtype]
    except KeyError:
        raise TbError("dtype", 2) from None


# ----------------------------------------------------------------------------- misc
def tb_status_string(code: int) -> str:
    return lib.tb_status_string(int(code)).decode()


def tb_version() -> int:
    return lib.tb_version()


def tb_device_error(reset: bool = True) -> int:
    """Device-side error word of the current device (0: no kernel gave up)."""
    code = ctypes.c_int(0)
    _check("tb_device_error", lib.tb_device_error(ctypes.byref(code), int(reset)))
    return code.value


def tb_layernorm_bwd_selftest_timeout(wait_limit_ns: int = 2_000_000, stream=None) -> None:
    """Runs the LayerNorm ring kernel with its copies withheld so that its bounded
    waits run out; synchronises. tb_device_error() then reports TB_ERR_TIMEOUT."""
    _check("tb_layernorm_bwd_selftest_timeout",
           lib.tb_layernorm_bwd_selftest_timeout(int(wait_limit_ns), _stream(stream)))


# ----------------------------------------------------------------------------- AdamW
class AdamWPlan:
    """Owns a ``tb_adamw_plan*``; keeps the tensors it points at alive."""

    def __init__(self, handle: int, tensors):
        self.handle = handle
        self._keep = tensors

    def close(self) -> None:
        if self.handle:
            _check("tb_adamw_plan_destroy", lib.tb_adamw_plan_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tb_adamw_plan_create(params: Sequence[torch.Tensor], ms: Sequence[torch.Tensor],
                         vs: Sequence[torch.Tensor], grads: Sequence[torch.Tensor],
                         copies: Sequence[torch.Tensor]) -> AdamWPlan:
    n = len(params)
    if not (len(ms) == len(vs) == len(grads) == len(copies) == n):
        raise ValueError("params, m, v, grads and copies must have one entry per tensor")
    gdtype = grads[0].dtype if n else None
    cdtypes = {c.dtype for c in copies if c is not None}
    if len(cdtypes) > 1:
        raise ValueError("every working copy must have the same dtype")
    for i in range(n):
        k = params[i].numel()
        _want(params[i], k, torch.float32, f"params[{i}]")
        _want(ms[i], k, torch.float32, f"m[{i}]")
        _want(vs[i], k, torch.float32, f"v[{i}]")
        _want(grads[i], k, gdtype, f"grads[{i}]")
        if copies[i] is not None:
            _want(copies[i], k, copies[i].dtype, f"copies[{i}]")
    descs = (tb_tensor_desc * max(n, 1))()
    for i in range(n):
        descs[i] = tb_tensor_desc(_ptr(params[i]), _ptr(ms[i]), _ptr(vs[i]), _ptr(grads[i]),
                                  _ptr(copies[i]), params[i].numel())
    gdt = _dtype(grads[0]) if n else TB_BF16
    with_copy = [c for c in copies if c is not None]
    cdt = _dtype(with_copy[0]) if with_copy else TB_BF16
    handle = ctypes.c_void_p(None)
    _check("tb_adamw_plan_create",
           lib.tb_adamw_plan_create(descs, n, gdt, cdt, ctypes.byref(handle)))
    return AdamWPlan(handle.value, (list(params), list(ms), list(vs), list(grads), list(copies)))


def tb_adamw_step(plan: AdamWPlan, step: int, lr: float, beta1: float, beta2: float, eps: float,
                  weight_decay: float, inv_loss_scale: float, stream=None) -> None:
    hp = tb_adamw_hparams(lr, beta1, beta2, eps, weight_decay)
    _check("tb_adamw_step", lib.tb_adamw_step(plan.handle, int(step), ctypes.byref(hp),
                                              float(inv_loss_scale), _stream(stream)))


def tb_adamw_step_device(plan: AdamWPlan, step: torch.Tensor, lr: float, beta1: float, beta2: float,
                         eps: float, weight_decay: float, inv_loss_scale: float,
                         clip: Optional[torch.Tensor] = None, stream=None) -> None:
    """The step counter is a 1-element int64 CUDA tensor, read when the kernel runs."""
    if step.dtype != torch.int64 or step.numel() != 1 or not step.is_cuda:
        raise ValueError("step must be a 1-element int64 CUDA tensor")
    if clip is not None and (clip.dtype != torch.float32 or clip.numel() < 3):
        raise ValueError("clip must hold 3 fp32 values")
    hp = tb_adamw_hparams(lr, beta1, beta2, eps, weight_decay)
    _check("tb_adamw_step_device",
           lib.tb_adamw_step_device(plan.handle, _ptr(step), ctypes.byref(hp), float(inv_loss_scale),
                                    _ptr(clip), _stream(stream)))


def tb_adamw_plan_destroy(plan: AdamWPlan) -> None:
    plan.close()


def tb_adamw_selftest_stale_counter(plan: AdamWPlan, next_tile: int, stream=None) -> None:
    """Test hook: leaves a stale value in the plan's tile counter (synchronises)."""
    _check("tb_adamw_selftest_stale_counter",
           lib.tb_adamw_selftest_stale_counter(plan.handle, int(next_tile), _stream(stream)))


def tb_adamw_grad_norm_workspace_size(plan: AdamWPlan) -> int:
    out = ctypes.c_size_t(0)
    _check("tb_adamw_grad_norm_workspace_size",
           lib.tb_adamw_grad_norm_workspace_size(plan.handle, ctypes.byref(out)))
    return out.value


def tb_adamw_grad_norm(plan: AdamWPlan, inv_loss_scale: float, max_norm: float,
                       out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Writes {norm, clip factor, nonfinite} (3 fp32 values) into ``out`` on the device."""
    if out.dtype != torch.float32 or out.numel() < 3:
        raise ValueError("out must hold 3 fp32 values")
    _check("tb_adamw_grad_norm",
           lib.tb_adamw_grad_norm(plan.handle, float(inv_loss_scale), float(max_norm), _ptr(out),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def tb_adamw_step_clipped(plan: AdamWPlan, step: int, lr: float, beta1: float, beta2: float,
                          eps: float, weight_decay: float, inv_loss_scale: float,
                          clip: torch.Tensor, stream=None) -> None:
    """tb_adamw_step with the gradient scaled by clip[1]; skipped when clip[2] != 0."""
    if clip.dtype != torch.float32 or clip.numel() < 3:
        raise ValueError("clip must hold 3 fp32 values")
    hp = tb_adamw_hparams(lr, beta1, beta2, eps, weight_decay)
    _check("tb_adamw_step_clipped",
           lib.tb_adamw_step_clipped(plan.handle, int(step), ctypes.byref(hp), float(inv_loss_scale),
                                     _ptr(clip), _stream(stream)))


# ----------------------------------------------------------------------------- casts
def tb_cast_to_f32(src: torch.Tensor, dst: torch.Tensor, scale: float = 1.0, stream=None) -> None:
    """dst = float(src) * scale (dst fp32, same number of elements)."""
    if dst.dtype != torch.float32 or dst.numel() != src.numel():
        raise ValueError("dst must be fp32 with as many elements as src")
    _check("tb_cast_to_f32", lib.tb_cast_to_f32(_ptr(src), _dtype(src), float(scale), _ptr(dst),
                                                src.numel(), _stream(stream)))


def tb_cast_from_f32(src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """dst = round-to-nearest-even(src) in dst's 16-bit dtype."""
    if src.dtype != torch.float32 or dst.numel() != src.numel():
        raise ValueError("src must be fp32 with as many elements as dst")
    _check("tb_cast_from_f32", lib.tb_cast_from_f32(_ptr(src), _ptr(dst), _dtype(dst), src.numel(),
                                                    _stream(stream)))


# ----------------------------------------------------------------------------- softmax bwd
def tb_softmax_bwd(dY: torch.Tensor, P: torch.Tensor, dX: torch.Tensor, stream=None) -> None:
    """dX = P * (dY - rowsum(P*dY)) over the last dimension of [rows, cols] tensors."""
    if not (dY.shape == P.shape == dX.shape) or dY.dim() != 2:
        raise ValueError("dY, P and dX must be [rows, cols] tensors of one shape")
    if not (dY.dtype == P.dtype == dX.dtype):
        raise ValueError("dY, P and dX must share a dtype")
    rows, cols = dY.shape
    _check("tb_softmax_bwd", lib.tb_softmax_bwd(_ptr(dY), _ptr(P), _ptr(dX), rows, cols,
                                                _dtype(dY), _stream(stream)))


def tb_softmax_bwd_causal(dY: torch.Tensor, P: torch.Tensor, dX: torch.Tensor, period: int,
                          offset: int = 0, stream=None) -> None:
    """Softmax backward reading only the causally open columns of each row:
    row r is nonzero only on its first min(cols, r % period + 1 + offset) columns."""
    if not (dY.shape == P.shape == dX.shape) or dY.dim() != 2:
        raise ValueError("dY, P and dX must be [rows, cols] tensors of one shape")
    if not (dY.dtype == P.dtype == dX.dtype):
        raise ValueError("dY, P and dX must share a dtype")
    rows, cols = dY.shape
    _check("tb_softmax_bwd_causal",
           lib.tb_softmax_bwd_causal(_ptr(dY), _ptr(P), _ptr(dX), rows, cols, int(period),
                                     int(offset), _dtype(dY), _stream(stream)))


# ----------------------------------------------------------------------------- RMSNorm bwd
def tb_rmsnorm_bwd_workspace_size(rows: int, D: int, dtype: torch.dtype) -> int:
    out = ctypes.c_size_t(0)
    _check("tb_rmsnorm_bwd_workspace_size",
           lib.tb_rmsnorm_bwd_workspace_size(int(rows), int(D), _DTYPE[dtype], ctypes.byref(out)))
    return out.value


def tb_rmsnorm_bwd(dY: torch.Tensor, x: torch.Tensor, inv_rms: torch.Tensor, gamma: torch.Tensor,
                   dX: torch.Tensor, dgamma: torch.Tensor, workspace: Optional[torch.Tensor],
                   stream=None) -> None:
    if x.dim() != 2 or dY.shape != x.shape or dX.shape != x.shape:
        raise ValueError("x, dY and dX must be [rows, D] tensors of one shape")
    if not (dY.dtype == x.dtype == dX.dtype):
        raise ValueError("x, dY and dX must share a dtype")
    rows, D = x.shape
    _want(inv_rms, rows, torch.float32, "inv_rms")
    _want(gamma, D, torch.float32, "gamma")
    _want(dgamma, D, torch.float32, "dgamma")
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("tb_rmsnorm_bwd",
           lib.tb_rmsnorm_bwd(_ptr(dY), _ptr(x), _ptr(inv_rms), _ptr(gamma), _ptr(dX),
                              _ptr(dgamma), rows, D, _dtype(x), ws_ptr, ws_bytes, _stream(stream)))


# ----------------------------------------------------------------------------- LayerNorm bwd
def tb_layernorm_bwd_workspace_size(rows: int, D: int, dtype: torch.dtype) -> int:
    out = ctypes.c_size_t(0)
    _check("tb_layernorm_bwd_workspace_size",
           lib.tb_layernorm_bwd_workspace_size(int(rows), int(D), _DTYPE[dtype], ctypes.byref(out)))
    return out.value


def tb_layernorm_bwd(dY: torch.Tensor, x: torch.Tensor, mean: torch.Tensor, inv_std: torch.Tensor,
                     gamma: torch.Tensor, dX: torch.Tensor, dgamma: torch.Tensor,
                     dbeta: torch.Tensor, workspace: Optional[torch.Tensor], stream=None) -> None:
    if x.dim() != 2 or dY.shape != x.shape or dX.shape != x.shape:
        raise ValueError("x, dY and dX must be [rows, D] tensors of one shape")
    if not (dY.dtype == x.dtype == dX.dtype):
        raise ValueError("x, dY and dX must share a dtype")
    rows, D = x.shape
    _want(mean, rows, torch.float32, "mean")
    _want(inv_std, rows, torch.float32, "inv_std")
    _want(gamma, D, torch.float32, "gamma")
    _want(dgamma, D, torch.float32, "dgamma")
    _want(dbeta, D, torch.float32, "dbeta")
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("tb_layernorm_bwd",
           lib.tb_layernorm_bwd(_ptr(dY), _ptr(x), _ptr(mean), _ptr(inv_std), _ptr(gamma),
                                _ptr(dX), _ptr(dgamma), _ptr(dbeta), rows, D, _dtype(x), ws_ptr,
                                ws_bytes, _stream(stream)))


def tb_layernorm_bwd_noalloc(dY: torch.Tensor, x: torch.Tensor, mean: torch.Tensor,
                             inv_std: torch.Tensor, gamma: torch.Tensor, dX: torch.Tensor,
                             dgamma: torch.Tensor, dbeta: torch.Tensor, stream=None) -> None:
    """tb_layernorm_bwd without a workspace: the library's own fixed scratch array is
    used, nothing is allocated (see include/tb.h for the limits)."""
    if x.dim() != 2 or dY.shape != x.shape or dX.shape != x.shape:
        raise ValueError("x, dY and dX must be [rows, D] tensors of one shape")
    if not (dY.dtype == x.dtype == dX.dtype):
        raise ValueError("x, dY and dX must share a dtype")
    rows, D = x.shape
    _want(mean, rows, torch.float32, "mean")
    _want(inv_std, rows, torch.float32, "inv_std")
    _want(gamma, D, torch.float32, "gamma")
    _want(dgamma, D, torch.float32, "dgamma")
    _want(dbeta, D, torch.float32, "dbeta")
    _check("tb_layernorm_bwd_noalloc",
           lib.tb_layernorm_bwd_noalloc(_ptr(dY), _ptr(x), _ptr(mean), _ptr(inv_std), _ptr(gamma),
                                        _ptr(dX), _ptr(dgamma), _ptr(dbeta), rows, D, _dtype(x),
                                        _stream(stream)))
