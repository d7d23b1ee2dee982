"""GPU parity of the gradient-norm clipping path against the CPU oracle.

tb_adamw_grad_norm (global L2 norm of the unscaled gradient, clip factor,
non-finite flag, all left on the device) and tb_adamw_step_clipped (the fused
AdamW step reading that factor on the device, skipping the update on a
non-finite gradient).  Tolerances: the norm and factor within 1e-5 relative
(fp32 rounds of at most 32 squares, fp32 over a tile's rounds, fp64 beyond: a
worst-case relative error of about 40 fp32 ulps); the clipped step within
the AdamW targets (theta/m/v 1e-5 floored relative, copy exact RNE of the master).
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import floored_rel, to_bits

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


def _plan(tb, st):
    k = len(st.sizes)
    return tb.tb_adamw_plan_create(*[[st.tensor(a, i) for i in range(k)]
                                     for a in ("theta", "m", "v", "grad", "copy")])


def _norm(tb, plan, inv, max_norm):
    out = torch.full((3,), float("nan"), device="cuda")
    ws = torch.empty(tb.tb_adamw_grad_norm_workspace_size(plan), dtype=torch.uint8, device="cuda")
    tb.tb_adamw_grad_norm(plan, inv, max_norm, out, ws)
    torch.cuda.synchronize()
    return out


def _grad_bits(st):
    return [to_bits(st.tensor("grad", i)) for i in range(len(st.sizes))]


def test_norm_and_factor_match_oracle_gpt2_table(tb, synth):
    st = synth.make_adamw_state(synth.gpt2_small_shapes(), seed=0, device="cuda")
    plan = _plan(tb, st)
    norm, bad = oracle.grad_norm_f64(_grad_bits(st), "bf16", 1 / 65536.0)
    for max_norm in (0.0, norm / 3, norm * 2):
        out = _norm(tb, plan, 1 / 65536.0, max_norm).double().cpu().numpy()
        assert abs(out[0] - norm) <= 1e-5 * norm
        assert abs(out[1] - oracle.clip_factor(norm, max_norm)) <= 1e-5
        assert out[2] == 0.0 and not bad


@pytest.mark.parametrize("align", [1, 128])
def test_nonfinite_flag_ragged_tables(tb, synth, align):
    sizes = [1, 7, 9, 0, 17, 1000, 8193, 65541]
    st = synth.make_adamw_state([(f"t{i}", (n,)) for i, n in enumerate(sizes)], seed=1,
                                device="cuda", align=align)
    plan = _plan(tb, st)
    norm, _ = oracle.grad_norm_f64(_grad_bits(st), "bf16", 1 / 65536.0)
    out = _norm(tb, plan, 1 / 65536.0, 0.0).cpu().numpy()
    assert abs(out[0] - norm) <= 1e-5 * norm and out[2] == 0.0
    for i, special in ((2, float("inf")), (6, float("nan")), (0, float("-inf"))):
        saved = st.tensor("grad", i).clone()
        st.tensor("grad", i)[-1] = special
        assert _norm(tb, plan, 1 / 65536.0, 0.0)[2].item() == 1.0
        st.tensor("grad", i).copy_(saved)


def test_clipped_steps_match_oracle(tb, synth):
    """Five steps on a ragged table with max_norm set so that some steps clip."""
    sizes = [3001, 4096, 17, 65536 + 5]
    st = synth.make_adamw_state([(f"t{i}", (n,)) for i, n in enumerate(sizes)], seed=2,
                                device="cuda", grad_dtype=torch.float16, loss_scale=1024.0)
    plan = _plan(tb, st)
    idx = np.concatenate([np.arange(o, o + n) for o, n in zip(st.offsets, st.sizes)])
    it = torch.from_numpy(idx).cuda()
    th = st.theta.index_select(0, it).double().cpu().numpy()
    m = np.zeros_like(th)
    v = np.zeros_like(th)
    cb = np.zeros(th.size, np.uint16)
    clipped = 0
    for t in range(1, 6):
        synth.fill_grads(st, t)
        gb = to_bits(st.grad.index_select(0, it))
        onorm, bad = oracle.grad_norm_f64([gb], "f16", 1 / 1024.0)
        max_norm = onorm * (0.5 if t % 2 else 2.0)
        out = torch.empty(3, device="cuda")
        ws = torch.empty(tb.tb_adamw_grad_norm_workspace_size(plan), dtype=torch.uint8, device="cuda")
        tb.tb_adamw_grad_norm(plan, 1 / 1024.0, max_norm, out, ws)
        tb.tb_adamw_step_clipped(plan, t, inv_loss_scale=1 / 1024.0, clip=out, **HP)
        clip = oracle.clip_factor(onorm, max_norm)
        clipped += clip < 1
        cb, _ = oracle.adamw_step_clipped_f64(th, m, v, gb, "f16", 1 / 1024.0, clip, bad, t,
                                              copy_in=cb, **HP)
        torch.cuda.synchronize()
        assert np.all(to_bits(st.grad.index_select(0, it)) == 0)
    assert clipped >= 2
    got = st.theta.index_select(0, it).double().cpu().numpy()
    assert floored_rel(got, th) <= 1e-5
    assert floored_rel(st.m.index_select(0, it).double().cpu().numpy(), m) <= 1e-5
    assert floored_rel(st.v.index_select(0, it).double().cpu().numpy(), v) <= 1e-5
    assert np.array_equal(to_bits(st.copy.index_select(0, it)), oracle.encode16(got, "bf16"))


def test_nonfinite_gradient_skips_the_step(tb, synth):
    st = synth.make_adamw_state([("a", (5000,)), ("b", (777,))], seed=3, device="cuda")
    plan = _plan(tb, st)
    tb.tb_adamw_step(plan, 1, inv_loss_scale=1 / 65536.0, **HP)     # some state to keep
    synth.fill_grads(st, 2)
    st.tensor("grad", 1)[100] = float("nan")
    before = [getattr(st, k).clone() for k in ("theta", "m", "v", "copy")]
    out = _norm(tb, plan, 1 / 65536.0, 1.0)
    assert out[2].item() == 1.0
    tb.tb_adamw_step_clipped(plan, 2, inv_loss_scale=1 / 65536.0, clip=out, **HP)
    torch.cuda.synchronize()
    for k, b in zip(("theta", "m", "v", "copy"), before):
        assert torch.equal(getattr(st, k), b), k
    assert torch.all(st.grad.view(torch.int16) == 0)


def test_factor_one_is_bitwise_the_plain_step(tb, synth):
    shapes = synth.gpt2_small_shapes()[:30]
    a = synth.make_adamw_state(shapes, seed=4, device="cuda")
    b = synth.make_adamw_state(shapes, seed=4, device="cuda")
    pa, pb = _plan(tb, a), _plan(tb, b)
    one = torch.tensor([1.0, 1.0, 0.0], device="cuda")
    for t in (1, 2):
        synth.fill_grads(a, t)
        synth.fill_grads(b, t)
        tb.tb_adamw_step(pa, t, inv_loss_scale=1 / 65536.0, **HP)
        tb.tb_adamw_step_clipped(pb, t, inv_loss_scale=1 / 65536.0, clip=one, **HP)
    torch.cuda.synchronize()
    for k in ("theta", "m", "v", "copy", "grad"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k


def test_norm_llama7b_table_against_float64_reduction(tb, synth):
    """Full 6.74 B-parameter table: the norm agrees with a float64 reduction of the
    same gradients (computed with torch on the device, chunk by chunk)."""
    st = synth.make_adamw_state(synth.llama7b_shapes(), seed=5, device="cuda", grad_std=1e-4)
    plan = _plan(tb, st)
    out_t = _norm(tb, plan, 1 / 65536.0, 1.0)
    out = out_t.double().cpu().numpy()
    assert torch.equal(_norm(tb, plan, 1 / 65536.0, 1.0), out_t)   # reproducible bit for bit
    total = 0.0
    for i in range(len(st.sizes)):
        g = st.tensor("grad", i)
        for s0 in range(0, g.numel(), 1 << 28):
            c = g[s0:s0 + (1 << 28)].double() / 65536.0
            total += float(torch.dot(c, c))
    ref = np.sqrt(total)
    # a non-finite element in one chunk of this table raises the flag (this table is large
    # enough for the one-CTA-per-chunk grid); an Inf in another chunk as well
    last = st.tensor("grad", len(st.sizes) - 1)
    emb = st.tensor("grad", 0)
    last[-3] = float("nan")
    flagged_nan = _norm(tb, plan, 1 / 65536.0, 1.0).cpu().numpy()[2]
    last[-3] = 0.0
    emb[123457] = float("inf")
    flagged_inf = _norm(tb, plan, 1 / 65536.0, 1.0).cpu().numpy()[2]
    plan.close()
    del st, last, emb
    torch.cuda.empty_cache()
    assert abs(out[0] - ref) <= 1e-5 * ref
    assert abs(out[1] - min(1.0, 1.0 / ref)) <= 1e-5 and out[2] == 0.0
    assert flagged_nan == 1.0 and flagged_inf == 1.0


def test_norm_special_cases(tb, synth):
    """All-zero gradients: norm 0, factor 1, no flag.  A max_norm that is negative or
    equal to the norm leaves the factor at exactly 1."""
    st = synth.make_adamw_state([("a", (4096,)), ("b", (77,))], seed=9, device="cuda")
    plan = _plan(tb, st)
    st.grad.zero_()
    out = _norm(tb, plan, 1 / 65536.0, 1.0).cpu().numpy()
    assert out[0] == 0.0 and out[1] == 1.0 and out[2] == 0.0
    # gradients whose unscaled norm is exactly 2: four elements of 1 (bf16 65536 * 1/65536)
    st.tensor("grad", 0)[:4] = 65536.0
    for max_norm in (-1.0, 2.0, 3.0):
        out = _norm(tb, plan, 1 / 65536.0, max_norm).cpu().numpy()
        assert out[0] == 2.0 and out[1] == 1.0 and out[2] == 0.0, max_norm
    out = _norm(tb, plan, 1 / 65536.0, 0.5).cpu().numpy()
    assert out[0] == 2.0 and out[1] == 0.25
    plan.close()
