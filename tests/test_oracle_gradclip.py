"""Pins for the oracle's global gradient-norm clipping.

Source: "GPU 优化实战 Part 2：用 CUDA/ROCm 实现 LLM 反向传播与训练循环", section
"完整训练循环（整合一切）", gradient clipping: the L2 norm of the unscaled gradient over all
parameters; when it exceeds max_norm the gradients are multiplied by
max_norm / norm before the optimizer step.

Independent checks: numpy's norm of the decoded gradients; special cases (zero
gradient, one nonzero element, NaN and infinity flagged); the clip factor's
closed forms; and torch.nn.utils.clip_grad_norm_ followed by torch.optim.AdamW
in float64 on the same gradients.
"""
import numpy as np
import torch

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def f32(x):
    return float(np.float32(x))


def test_norm_matches_numpy_over_several_tensors(orc):
    rng = np.random.default_rng(0)
    parts = [orc.encode16(rng.standard_normal(n) * 65.5, "bf16") for n in (1, 7, 1000, 4096)]
    norm, bad = orc.grad_norm_f64(parts, "bf16", 1 / 65536.0)
    dec = np.concatenate([orc.decode16(p, "bf16") for p in parts]) / 65536.0
    assert not bad
    assert abs(norm - np.linalg.norm(dec)) <= 1e-14 * norm


def test_norm_special_cases(orc):
    z = np.zeros(100, np.uint16)
    assert orc.grad_norm_f64([z], "f16", 1.0) == (0.0, False)
    one = z.copy()
    one[37] = orc.encode16(np.array([-3.0]), "f16")[0]
    assert orc.grad_norm_f64([one], "f16", 0.5) == (1.5, False)
    for special in (np.inf, -np.inf, np.nan):
        g = z.copy()
        g[5] = orc.encode16(np.array([special]), "bf16")[0]
        assert orc.grad_norm_f64([z, g], "bf16", 1.0)[1] is True


def test_clip_factor_closed_forms(orc):
    assert orc.clip_factor(2.0, 1.0) == 0.5
    assert orc.clip_factor(1.0, 1.0) == 1.0           # not above max_norm: unchanged
    assert orc.clip_factor(0.5, 1.0) == 1.0
    assert orc.clip_factor(5.0, 0.0) == 1.0           # clipping disabled


def test_clipped_step_matches_torch_clip_then_adamw(orc):
    n, steps, scale, max_norm = 3000, 6, 1024.0, 0.02
    rng = np.random.default_rng(1)
    th0 = rng.standard_normal(n) * 0.02
    p = torch.nn.Parameter(torch.from_numpy(th0.copy()))
    opt = torch.optim.AdamW([p], lr=f32(HP["lr"]), betas=(f32(0.9), f32(0.999)),
                            eps=f32(HP["eps"]), weight_decay=f32(HP["weight_decay"]),
                            foreach=False, fused=False)
    th, m, v = th0.copy(), np.zeros(n), np.zeros(n)
    clipped_any = False
    for t in range(1, steps + 1):
        gb = orc.encode16(rng.standard_normal(n) * 1e-3 * scale * (1 + t), "f16")
        g = orc.decode16(gb, "f16") / scale
        p.grad = torch.from_numpy(g.copy())
        torch.nn.utils.clip_grad_norm_([p], max_norm, foreach=False)
        opt.step()
        norm, bad = orc.grad_norm_f64([gb], "f16", 1 / scale)
        clip = orc.clip_factor(norm, max_norm)
        clipped_any |= clip < 1.0
        orc.adamw_step_clipped_f64(th, m, v, gb, "f16", 1 / scale, clip, bad, t, **HP)
        # torch adds 1e-6 to the norm inside its clip coefficient: the clipped gradients
        # differ by ~1e-6/norm relative, which Adam's near scale-invariance turns into
        # at most ~lr * 1e-5 absolute in theta
        np.testing.assert_allclose(th, p.detach().numpy(), rtol=1e-6, atol=1e-8)
    assert clipped_any


def test_skip_leaves_state_and_zeroes_gradient(orc):
    n = 64
    rng = np.random.default_rng(2)
    th = rng.standard_normal(n)
    m = rng.standard_normal(n) * 1e-3
    v = np.abs(rng.standard_normal(n)) * 1e-6
    before = (th.copy(), m.copy(), v.copy())
    gb = orc.encode16(rng.standard_normal(n), "bf16")
    copy_in = rng.integers(0, 65535, n).astype(np.uint16)
    copy, gz = orc.adamw_step_clipped_f64(th, m, v, gb, "bf16", 1.0, 1.0, True, 3,
                                          copy_in=copy_in, **HP)
    for a, b in zip((th, m, v), before):
        assert np.array_equal(a, b)
    assert np.all(gz == 0)
    assert np.array_equal(copy, copy_in)


def test_clip_one_equals_plain_step(orc):
    n = 500
    rng = np.random.default_rng(3)
    th0 = rng.standard_normal(n) * 0.02
    gb = orc.encode16(rng.standard_normal(n) * 65.0, "bf16")
    a = [th0.copy(), np.zeros(n), np.zeros(n)]
    b = [th0.copy(), np.zeros(n), np.zeros(n)]
    ca, _ = orc.adamw_step_f64(*a, gb, "bf16", 1 / 65536.0, 1, **HP)
    cb, _ = orc.adamw_step_clipped_f64(*b, gb, "bf16", 1 / 65536.0, 1.0, False, 1, **HP)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert np.array_equal(ca, cb)
