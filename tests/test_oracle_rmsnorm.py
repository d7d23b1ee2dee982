"""Pins for the oracle's RMSNorm backward.

RMSNorm is the LayerNorm of "GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环"
section 2.2 "LayerNorm 反向" without the mean subtraction and without beta
(the norm layers of the Llama-7B table): y = gamma * x * inv_rms with
inv_rms = 1/sqrt(mean(x^2) + eps).

Independent checks: dgamma is the column sum of dY*xhat; with eps = 0 every
row of dX is orthogonal to xhat (y is invariant to scaling x); the defect
with eps > 0 has a closed form; central finite differences with inv_rms
recomputed from x; torch's rms_norm autograd in float64.
"""
import numpy as np
import torch


def _inv_rms(x, eps):
    return 1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)


def _inputs(rows, D, seed, eps=1e-5):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, D))
    dY = rng.standard_normal((rows, D))
    gamma = 1.0 + 0.1 * rng.standard_normal(D)
    return x, dY, _inv_rms(x, eps), gamma


def test_dgamma_is_column_sum_of_dy_xhat(orc):
    x, dY, rs, g = _inputs(200, 48, 0)
    _, dg = orc.rmsnorm_bwd_f64(dY, x, rs, g)
    np.testing.assert_allclose(dg, np.einsum("rd,rd->d", dY, x * rs[:, None]), rtol=1e-12, atol=1e-12)


def test_dx_orthogonal_to_xhat_when_eps_zero(orc):
    x, dY, rs, g = _inputs(64, 256, 1, eps=0.0)
    dX, _ = orc.rmsnorm_bwd_f64(dY, x, rs, g)
    xhat = x * rs[:, None]
    scale = rs * np.sum(np.abs(dY * g * xhat), axis=1)
    assert np.all(np.abs(np.sum(dX * xhat, axis=1)) <= 1e-12 * scale)


def test_orthogonality_defect_with_eps_matches_closed_form(orc):
    x, dY, rs, g = _inputs(16, 128, 2, eps=0.3)
    dX, _ = orc.rmsnorm_bwd_f64(dY, x, rs, g)
    xhat = x * rs[:, None]
    D = x.shape[1]
    expect = rs * np.sum(dY * g * xhat, axis=1) * (1 - np.sum(xhat * xhat, axis=1) / D)
    np.testing.assert_allclose(np.sum(dX * xhat, axis=1), expect, rtol=1e-9, atol=1e-14)


def test_central_finite_differences(orc):
    rows, D, eps, h = 3, 5, 1e-5, 1e-6
    rng = np.random.default_rng(3)
    x = rng.standard_normal((rows, D))
    dY = rng.standard_normal((rows, D))
    gamma = 1.0 + 0.1 * rng.standard_normal(D)

    def loss(xx, gg):
        return float(np.sum(dY * gg * xx * _inv_rms(xx, eps)[:, None]))

    fdx = np.zeros_like(x)
    for r in range(rows):
        for c in range(D):
            xp, xm = x.copy(), x.copy()
            xp[r, c] += h
            xm[r, c] -= h
            fdx[r, c] = (loss(xp, gamma) - loss(xm, gamma)) / (2 * h)
    fdg = np.zeros(D)
    for c in range(D):
        e = np.zeros(D)
        e[c] = h
        fdg[c] = (loss(x, gamma + e) - loss(x, gamma - e)) / (2 * h)
    dX, dg = orc.rmsnorm_bwd_f64(dY, x, _inv_rms(x, eps), gamma)
    np.testing.assert_allclose(dX, fdx, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dg, fdg, rtol=1e-6, atol=1e-8)


def test_matches_torch_rms_norm_autograd_float64(orc):
    rows, D, eps = 29, 80, 1e-5
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.standard_normal((rows, D))).requires_grad_(True)
    w = torch.from_numpy(1.0 + 0.1 * rng.standard_normal(D)).requires_grad_(True)
    dY = torch.from_numpy(rng.standard_normal((rows, D)))
    torch.nn.functional.rms_norm(x, (D,), w, eps).backward(dY)
    xn = x.detach().numpy()
    dX, dg = orc.rmsnorm_bwd_f64(dY.numpy(), xn, _inv_rms(xn, eps), w.detach().numpy())
    np.testing.assert_allclose(dX, x.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, w.grad.numpy(), rtol=1e-10, atol=1e-12)
