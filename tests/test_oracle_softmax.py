"""Pins for the oracle's softmax backward.

Source: "GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环",
section 2.1 "Softmax 反向内核": dX_i = P_i (dY_i - sum_j P_j dY_j) per row.

Independent checks: special cases with closed forms (one-hot and uniform P),
the row-sum invariant, central finite differences of L = sum dY*softmax(z), and
torch autograd of softmax in float64.
"""
import numpy as np
import torch


def _softmax(z):
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def test_one_hot_rows_give_exact_zero(orc):
    rows, cols = 7, 33
    rng = np.random.default_rng(0)
    P = np.zeros((rows, cols))
    P[np.arange(rows), rng.integers(0, cols, rows)] = 1.0
    dY = rng.standard_normal((rows, cols))
    assert np.all(orc.softmax_bwd_f64(dY, P) == 0.0)
    assert np.all(orc.softmax_bwd_f32(dY, P) == 0.0)


def test_uniform_rows_give_centered_dy(orc):
    rows, cols = 5, 64                      # 1/64 is exact in binary
    rng = np.random.default_rng(1)
    P = np.full((rows, cols), 1.0 / cols)
    dY = rng.standard_normal((rows, cols))
    expect = (dY - dY.mean(axis=1, keepdims=True)) / cols
    np.testing.assert_allclose(orc.softmax_bwd_f64(dY, P), expect, rtol=1e-12, atol=1e-16)


def test_rows_sum_to_zero(orc):
    """sum_j dX_j = dot * (1 - sum_j P_j): zero up to rounding for a normalised row."""
    rows, cols = 64, 1000
    rng = np.random.default_rng(2)
    P = _softmax(rng.standard_normal((rows, cols)))
    dY = rng.standard_normal((rows, cols))
    dX = orc.softmax_bwd_f64(dY, P)
    scale = np.sum(np.abs(P * dY), axis=1) + np.abs(np.sum(P * dY, axis=1))
    assert np.all(np.abs(dX.sum(axis=1)) <= 8 * cols * 2.0 ** -53 * scale)
    dX32 = orc.softmax_bwd_f32(dY.astype(np.float32), P.astype(np.float32)).astype(np.float64)
    P32 = P.astype(np.float32).astype(np.float64)
    dY32 = dY.astype(np.float32).astype(np.float64)
    scale32 = np.sum(np.abs(P32 * dY32), axis=1) + np.abs(np.sum(P32 * dY32, axis=1))
    # the fp32 row's probabilities sum to 1 only within fp32 rounding
    resid = np.abs(np.sum(P32 * dY32, axis=1) * (1 - P32.sum(axis=1)))
    assert np.all(np.abs(dX32.sum(axis=1)) <= 8 * cols * 2.0 ** -24 * scale32 + resid)


def test_central_finite_differences(orc):
    rows, cols, h = 3, 5, 1e-6
    rng = np.random.default_rng(3)
    z = rng.standard_normal((rows, cols))
    dY = rng.standard_normal((rows, cols))

    def loss(zz):
        return float(np.sum(dY * _softmax(zz)))

    fd = np.zeros_like(z)
    for r in range(rows):
        for c in range(cols):
            zp, zm = z.copy(), z.copy()
            zp[r, c] += h
            zm[r, c] -= h
            fd[r, c] = (loss(zp) - loss(zm)) / (2 * h)
    got = orc.softmax_bwd_f64(dY, _softmax(z))
    np.testing.assert_allclose(got, fd, rtol=1e-7, atol=1e-9)


def test_matches_torch_autograd_float64(orc):
    rows, cols = 17, 129
    rng = np.random.default_rng(4)
    z = torch.from_numpy(rng.standard_normal((rows, cols))).requires_grad_(True)
    dY = torch.from_numpy(rng.standard_normal((rows, cols)))
    P = torch.softmax(z, dim=1)
    P.backward(dY)
    got = orc.softmax_bwd_f64(dY.numpy(), P.detach().numpy())
    np.testing.assert_allclose(got, z.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_fp32_variant_within_rounding_of_fp64(orc):
    rows, cols = 128, 1024
    rng = np.random.default_rng(5)
    P = _softmax(rng.standard_normal((rows, cols))).astype(np.float32)
    dY = rng.standard_normal((rows, cols)).astype(np.float32)
    d64 = orc.softmax_bwd_f64(dY, P)
    d32 = orc.softmax_bwd_f32(dY, P)
    # sequential fp32 dot: |err| <= cols * 2^-24 * sum|P dY|; then two roundings
    bound = cols * 2.0 ** -24 * np.sum(np.abs(P * dY), axis=1, keepdims=True) * P + \
        2 * 2.0 ** -24 * np.abs(d64)
    assert np.all(np.abs(d32 - d64) <= bound + 1e-30)
