"""Pins for the oracle's AdamW step.

Sources: "Mastering LLM Training with CUDA and ROCm: The Backpropagation and
Optimization Workflow", section "AdamW Algorithm" (the update rule), and
"GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环", sections
"AdamW 优化器——融合内核" and "混合精度训练（FP16 / BF16）".

What fixes the oracle here, independently of its own code:
* closed forms: step 1 from m=v=0; a constant gradient with no decay; a zero
  gradient (pure decay);
* a library routine on a special case: torch.optim.AdamW in float64 with the
  loss scale folded into the gradient (decoupled decay, bias corrections and
  eps placement all have to agree);
* the fp32 variant against the fp64 one after 100 steps.
"""
import numpy as np
import pytest
import torch

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def f32(x):
    return float(np.float32(x))


def _grads(rng, n, std, scale, kind):
    import oracle
    return oracle.encode16(rng.standard_normal(n) * std * scale, kind)


def test_bias_correction_is_one_minus_beta_pow_t(orc):
    for beta in (0.9, 0.999):
        for t in (1, 2, 10, 1000):
            assert orc.bias_correction(beta, t) == 1.0 - float(np.float32(beta)) ** t


@pytest.mark.parametrize("kind, scale", [("f16", 1024.0), ("bf16", 65536.0)])
def test_step1_closed_form(orc, kind, scale):
    """From m=v=0, m_hat=g and v_hat=g^2, so theta_1 = theta_0 - lr*g/(|g|+eps) - lr*wd*theta_0."""
    rng = np.random.default_rng(0)
    n = 4096
    th0 = rng.standard_normal(n) * 0.02
    gb = _grads(rng, n, 1e-3, scale, kind)
    g = orc.decode16(gb, kind) / scale
    lr, eps, wd = f32(HP["lr"]), f32(HP["eps"]), f32(HP["weight_decay"])
    expect = th0 - lr * g / (np.abs(g) + eps) - lr * wd * th0

    th, m, v = th0.copy(), np.zeros(n), np.zeros(n)
    copy, gz = orc.adamw_step_f64(th, m, v, gb, kind, 1.0 / scale, 1, **HP)
    np.testing.assert_allclose(th, expect, rtol=1e-15, atol=1e-18)
    np.testing.assert_allclose(m, (1 - f32(0.9)) * g, rtol=1e-15)
    np.testing.assert_allclose(v, (1 - f32(0.999)) * g * g, rtol=1e-15)
    assert np.all(gz == 0)
    assert np.array_equal(copy, orc.encode16(th, "bf16"))

    # fp32 variant: same closed form from the fp32-rounded start; each operand
    # rounds once, so the error is a few fp32 ulps of the operand scale |theta_0|
    th32 = th0.astype(np.float32)
    m32, v32 = np.zeros(n, np.float32), np.zeros(n, np.float32)
    t0 = th32.astype(np.float64)
    expect32 = t0 - lr * g / (np.abs(g) + eps) - lr * wd * t0
    orc.adamw_step_f32(th32, m32, v32, gb, kind, 1.0 / scale, 1, **HP)
    ulp = np.spacing(np.maximum(np.abs(t0), np.abs(expect32)).astype(np.float32))
    assert np.max(np.abs(th32 - expect32) / ulp.astype(np.float64)) <= 4.0


def test_constant_gradient_no_decay(orc):
    """g_t = c for all t and wd = 0: m_t = c(1-b1^t), v_t = c^2(1-b2^t), so
    m_hat = c, v_hat = c^2 and theta_t = theta_0 - t*lr*c/(|c|+eps)."""
    n, scale = 64, 1024.0
    rng = np.random.default_rng(1)
    gb = orc.encode16(rng.standard_normal(n) * 1e-3 * scale, "f16")
    c = orc.decode16(gb, "f16") / scale
    th0 = rng.standard_normal(n) * 0.02
    th, m, v = th0.copy(), np.zeros(n), np.zeros(n)
    hp = dict(HP, weight_decay=0.0)
    lr, eps = f32(hp["lr"]), f32(hp["eps"])
    b1, b2 = f32(0.9), f32(0.999)
    for t in range(1, 31):
        orc.adamw_step_f64(th, m, v, gb, "f16", 1.0 / scale, t, **hp)
        np.testing.assert_allclose(m, c * (1 - b1 ** t), rtol=1e-13)
        np.testing.assert_allclose(v, c * c * (1 - b2 ** t), rtol=1e-12)
        np.testing.assert_allclose(th, th0 - t * lr * c / (np.abs(c) + eps), rtol=1e-12)


def test_zero_gradient_is_pure_decay(orc):
    n = 128
    rng = np.random.default_rng(2)
    th0 = rng.standard_normal(n) * 0.02
    th, m, v = th0.copy(), np.zeros(n), np.zeros(n)
    gb = np.zeros(n, np.uint16)
    lr, wd = f32(HP["lr"]), f32(HP["weight_decay"])
    for t in range(1, 21):
        orc.adamw_step_f64(th, m, v, gb, "bf16", 1.0 / 65536, t, **HP)
        assert np.all(m == 0) and np.all(v == 0)
        np.testing.assert_allclose(th, th0 * (1 - lr * wd) ** t, rtol=1e-14)


def test_matches_torch_adamw_float64(orc):
    """torch.optim.AdamW (decoupled decay, bias-corrected moments, eps outside
    the root) fed the unscaled gradients must follow the same trajectory."""
    n, scale, steps = 2048, 1024.0, 10
    rng = np.random.default_rng(3)
    th0 = rng.standard_normal(n) * 0.02
    p = torch.nn.Parameter(torch.from_numpy(th0.copy()))
    opt = torch.optim.AdamW([p], lr=f32(HP["lr"]), betas=(f32(0.9), f32(0.999)),
                            eps=f32(HP["eps"]), weight_decay=f32(HP["weight_decay"]),
                            foreach=False, fused=False)
    th, m, v = th0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, steps + 1):
        gb = _grads(rng, n, 1e-3, scale, "f16")
        g = orc.decode16(gb, "f16") / scale
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        orc.adamw_step_f64(th, m, v, gb, "f16", 1.0 / scale, t, **HP)
        np.testing.assert_allclose(th, p.detach().numpy(), rtol=1e-12, atol=1e-16)
        st = opt.state[p]
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-12, atol=1e-20)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-12, atol=1e-24)


def floored_rel(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    floor = np.sqrt(np.mean(y * y))
    return float(np.max(np.abs(x - y) / np.maximum(np.abs(y), floor)))


def test_fp32_variant_tracks_fp64_over_100_steps(orc):
    n, scale = 1 << 14, 65536.0
    rng = np.random.default_rng(4)
    th0 = rng.standard_normal(n) * 0.02
    th64, m64, v64 = th0.copy(), np.zeros(n), np.zeros(n)
    th32 = th0.astype(np.float32)
    m32, v32 = np.zeros(n, np.float32), np.zeros(n, np.float32)
    th64 = th32.astype(np.float64)  # same start
    for t in range(1, 101):
        gb = _grads(rng, n, 1e-3, scale, "bf16")
        c64, _ = orc.adamw_step_f64(th64, m64, v64, gb, "bf16", 1.0 / scale, t, **HP)
        c32, _ = orc.adamw_step_f32(th32, m32, v32, gb, "bf16", 1.0 / scale, t, **HP)
    # each step adds at most ~4 fp32 roundings (2^-24 relative to the operands);
    # bound their accumulation linearly over the 100 steps
    bound = 4 * 100 * 2.0 ** -24
    assert floored_rel(th32, th64) <= bound
    assert floored_rel(m32, m64) <= bound
    assert floored_rel(v32, v64) <= bound
    # the working copies are roundings of nearly equal masters: at most 1 ulp apart
    d = np.abs(c64.astype(np.int32) - c32.astype(np.int32))
    assert d.max() <= 1


def test_copy_can_be_fp16(orc):
    n = 256
    rng = np.random.default_rng(5)
    th = rng.standard_normal(n) * 0.02
    m, v = np.zeros(n), np.zeros(n)
    gb = _grads(rng, n, 1e-3, 1024.0, "f16")
    copy, _ = orc.adamw_step_f64(th, m, v, gb, "f16", 1 / 1024.0, 1, copy_kind="f16", **HP)
    assert np.array_equal(copy, th.astype(np.float16).view(np.uint16))
