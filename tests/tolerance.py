"""Comparison helpers for the GPU-vs-oracle parity tests.

fp32 outputs use the error measures the targets are stated in:
* floored relative error  max |got - ref| / max(|ref|, rms(ref)) -- the rms
  floor keeps elements that cancel to ~0 from dominating;
* plain max absolute error.

16-bit outputs (bf16 / fp16) are compared with the rule "within one unit in
the last place of the oracle's exact result rounded to nearest even", i.e. the
integer distance between ordered bit patterns is <= 1.  Where the kernel's own
fp32 arithmetic may legitimately be off by more than half a 16-bit ulp before
the final rounding (a result that cancels to far below its terms), the caller
passes an absolute bound ``err`` on that fp32 error, derived from the inputs;
an element then also passes when |got - ref| <= err + ulp(|ref| + err) / 2,
which is exactly "got is the rounding of a value within err of ref".
"""
from __future__ import annotations

import numpy as np

import oracle


def floored_rel(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    floor = np.sqrt(np.mean(ref * ref))
    floor = floor if floor > 0 else 1e-300
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


def _ordered(bits: np.ndarray) -> np.ndarray:
    """Map 16-bit float patterns to integers that increase with the value."""
    b = bits.astype(np.int64)
    neg = (b & 0x8000) != 0
    mag = b & 0x7FFF
    return np.where(neg, -mag, mag)


def ulp16(x: np.ndarray, kind: str) -> np.ndarray:
    """Spacing of the 16-bit format at |x| (normal and subnormal ranges)."""
    frac_bits, emin = (7, -126) if kind == "bf16" else (10, -14)
    a = np.abs(np.asarray(x, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - frac_bits).astype(np.int64))


def lowp_check(got_bits, ref, kind: str, err=None):
    """Returns (ok_mask, n_needing_err_bound, max_ulp_distance)."""
    ref = np.asarray(ref, np.float64)
    if err is not None:
        err = np.broadcast_to(np.asarray(err, np.float64), ref.shape).ravel()
    got_bits = np.asarray(got_bits).view(np.uint16).ravel()
    ref = ref.ravel()
    ref_bits = oracle.encode16(ref, kind)
    dist = np.abs(_ordered(got_bits) - _ordered(ref_bits))
    ok = dist <= 1
    n_err = 0
    if err is not None:
        got = oracle.decode16(got_bits, kind)
        ok2 = np.abs(got - ref) <= err + 0.5 * ulp16(np.abs(ref) + err, kind)
        n_err = int(np.sum(ok2 & ~ok))
        ok = ok | ok2
    return ok, n_err, int(dist.max()) if dist.size else 0


def to_bits(t) -> np.ndarray:
    """uint16 view of a 16-bit torch tensor, on the host."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def within_bound(got, ref, err) -> np.ndarray:
    """|got - ref| <= err elementwise (fp32 outputs with a derived error bound)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref) <= np.broadcast_to(np.asarray(err, np.float64), ref.shape)


def layernorm_dx_err_bound(x, dY, mean, rstd, gamma):
    """Bound on |dX_fp32 - dX_exact| of the LayerNorm backward (numpy float64 inputs):
    xhat and dxhat carry a few fp32 roundings, the two row sums at most D/32 + 64
    rounded additions each."""
    D = x.shape[1]
    xh = (x - mean[:, None]) * rstd[:, None]
    dxh = dY * gamma[None, :]
    sa = np.sum(np.abs(dxh), axis=1, keepdims=True) / D
    sb = np.sum(np.abs(dxh * xh), axis=1, keepdims=True) / D
    mb = np.abs(np.sum(dxh * xh, axis=1, keepdims=True)) / D
    ma = np.abs(np.sum(dxh, axis=1, keepdims=True)) / D
    k = D / 32 + 64
    u = 2.0 ** -24
    return rstd[:, None] * (4 * u * (np.abs(dxh) + ma + np.abs(xh) * mb) +
                            k * u * (sa + np.abs(xh) * sb))
