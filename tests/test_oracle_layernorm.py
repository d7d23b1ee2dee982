"""Pins for the oracle's LayerNorm backward.

Sources: "GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环",
section 2.2 "LayerNorm 反向" (saved mean / inv_std, gamma and beta gradients by
reduction, dX from the normalised values), and "Mastering LLM Training with
CUDA and ROCm", section "Layer Normalization Backpropagation".

Independent checks: dbeta is the column sum of dY; rows of dX sum to zero and
(with eps = 0) are orthogonal to xhat; D = 1 degenerates to zero gradients;
central finite differences of L = sum dY * LN(x) with the statistics recomputed
from x; torch autograd of layer_norm in float64.
"""
import numpy as np
import torch


def _stats(x, eps):
    mu = x.mean(axis=1)
    var = ((x - mu[:, None]) ** 2).mean(axis=1)
    return mu, 1.0 / np.sqrt(var + eps)


def _inputs(rows, D, seed, eps=1e-5):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, D))
    dY = rng.standard_normal((rows, D))
    gamma = 1.0 + 0.1 * rng.standard_normal(D)
    mu, rs = _stats(x, eps)
    return x, dY, mu, rs, gamma


def test_dbeta_is_column_sum(orc):
    x, dY, mu, rs, g = _inputs(300, 40, 0)
    _, _, db = orc.layernorm_bwd_f64(dY, x, mu, rs, g)
    np.testing.assert_allclose(db, dY.sum(axis=0), rtol=1e-13, atol=1e-13)


def test_dgamma_is_column_sum_of_dy_xhat(orc):
    x, dY, mu, rs, g = _inputs(300, 40, 1)
    _, dg, _ = orc.layernorm_bwd_f64(dY, x, mu, rs, g)
    xhat = (x - mu[:, None]) * rs[:, None]
    np.testing.assert_allclose(dg, np.einsum("rd,rd->d", dY, xhat), rtol=1e-12, atol=1e-12)


def test_rows_of_dx_sum_to_zero(orc):
    x, dY, mu, rs, g = _inputs(64, 256, 2)
    dX, _, _ = orc.layernorm_bwd_f64(dY, x, mu, rs, g)
    scale = rs * np.sum(np.abs(dY * g), axis=1)
    assert np.all(np.abs(dX.sum(axis=1)) <= 1e-12 * scale)


def test_dx_orthogonal_to_xhat_when_eps_zero(orc):
    x, dY, mu, rs, g = _inputs(64, 256, 3, eps=0.0)
    dX, _, _ = orc.layernorm_bwd_f64(dY, x, mu, rs, g)
    xhat = (x - mu[:, None]) * rs[:, None]
    scale = rs * np.sum(np.abs(dY * g * xhat), axis=1)
    assert np.all(np.abs(np.sum(dX * xhat, axis=1)) <= 1e-12 * scale)


def test_dx_orthogonality_defect_with_eps_matches_closed_form(orc):
    """With eps > 0, sum_j xhat_j^2 = D*var/(var+eps) and the defect is
    rs * sum(dxhat*xhat) * (1 - sum(xhat^2)/D) exactly."""
    x, dY, mu, rs, g = _inputs(16, 128, 4, eps=1e-1)
    dX, _, _ = orc.layernorm_bwd_f64(dY, x, mu, rs, g)
    xhat = (x - mu[:, None]) * rs[:, None]
    dxhat = dY * g
    D = x.shape[1]
    expect = rs * np.sum(dxhat * xhat, axis=1) * (1 - np.sum(xhat * xhat, axis=1) / D)
    np.testing.assert_allclose(np.sum(dX * xhat, axis=1), expect, rtol=1e-9, atol=1e-14)


def test_d_equals_one_is_degenerate(orc):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 1))
    dY = rng.standard_normal((9, 1))
    mu, rs = _stats(x, 1e-5)
    dX, dg, db = orc.layernorm_bwd_f64(dY, x, mu, rs, np.array([1.3]))
    assert np.all(dX == 0.0) and np.all(dg == 0.0)
    np.testing.assert_allclose(db, dY.sum(axis=0), rtol=1e-14)


def test_central_finite_differences(orc):
    rows, D, eps, h = 3, 5, 1e-5, 1e-6
    rng = np.random.default_rng(6)
    x = rng.standard_normal((rows, D))
    dY = rng.standard_normal((rows, D))
    gamma = 1.0 + 0.1 * rng.standard_normal(D)
    beta = 0.1 * rng.standard_normal(D)

    def loss(xx, gg, bb):
        mu, rs = _stats(xx, eps)
        y = gg * (xx - mu[:, None]) * rs[:, None] + bb
        return float(np.sum(dY * y))

    fdx = np.zeros_like(x)
    for r in range(rows):
        for c in range(D):
            xp, xm = x.copy(), x.copy()
            xp[r, c] += h
            xm[r, c] -= h
            fdx[r, c] = (loss(xp, gamma, beta) - loss(xm, gamma, beta)) / (2 * h)
    fdg = np.zeros(D)
    fdb = np.zeros(D)
    for c in range(D):
        e = np.zeros(D)
        e[c] = h
        fdg[c] = (loss(x, gamma + e, beta) - loss(x, gamma - e, beta)) / (2 * h)
        fdb[c] = (loss(x, gamma, beta + e) - loss(x, gamma, beta - e)) / (2 * h)
    mu, rs = _stats(x, eps)
    dX, dg, db = orc.layernorm_bwd_f64(dY, x, mu, rs, gamma)
    np.testing.assert_allclose(dX, fdx, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dg, fdg, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(db, fdb, rtol=1e-6, atol=1e-8)


def test_matches_torch_autograd_float64(orc):
    rows, D, eps = 37, 96, 1e-5
    rng = np.random.default_rng(7)
    x = torch.from_numpy(rng.standard_normal((rows, D))).requires_grad_(True)
    w = torch.from_numpy(1.0 + 0.1 * rng.standard_normal(D)).requires_grad_(True)
    b = torch.from_numpy(0.1 * rng.standard_normal(D)).requires_grad_(True)
    dY = torch.from_numpy(rng.standard_normal((rows, D)))
    torch.nn.functional.layer_norm(x, (D,), w, b, eps).backward(dY)
    xn = x.detach().numpy()
    mu, rs = _stats(xn, eps)
    dX, dg, db = orc.layernorm_bwd_f64(dY.numpy(), xn, mu, rs, w.detach().numpy())
    np.testing.assert_allclose(dX, x.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, w.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db, b.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_fp32_variant_close_to_fp64(orc):
    x, dY, mu, rs, g = _inputs(256, 512, 8)
    x32, dY32 = x.astype(np.float32), dY.astype(np.float32)
    mu32, rs32, g32 = mu.astype(np.float32), rs.astype(np.float32), g.astype(np.float32)
    d64 = orc.layernorm_bwd_f64(dY32, x32, mu32, rs32, g32)
    d32 = orc.layernorm_bwd_f32(dY32, x32, mu32, rs32, g32)
    for a, b in zip(d32, d64):
        floor = np.sqrt(np.mean(b * b))
        # sequential fp32 sums over <= 512 terms: error ~ n * 2^-24 of the term scale
        assert np.max(np.abs(a - b) / np.maximum(np.abs(b), floor)) <= 512 * 2.0 ** -24 * 4
