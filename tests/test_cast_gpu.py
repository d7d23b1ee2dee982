"""GPU parity of the stand-alone casts and of the unfused optimizer pipeline.

The casts are bit-exact against the oracle (one rounding each).  The pages'
unfused tail -- cast the 16-bit gradient to fp32 times 1/loss_scale, AdamW on
fp32 gradients without a working copy, cast the master to bf16 -- must give
bit for bit the state the fused step gives, since every rounding is the same.
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import floored_rel, to_bits

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
KIND = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


def _src(n, dtype, offset=0, seed=0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(n + offset, generator=g, device="cuda") * torch.exp(
        torch.empty(n + offset, device="cuda").uniform_(-12, 12, generator=g))
    return x.to(dtype)[offset:]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32],
                         ids=["f16", "bf16", "f32"])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, (1 << 20) + 3])
# (source offset, destination offset) in elements: both aligned for the 32-byte store
# path; a 16- but not 32-byte aligned destination for the 4-element chunk path (a source
# offset of 8 keeps it 16-byte aligned, one of 4 leaves a 16-bit source only 8-byte
# aligned, which that path still takes); both misaligned for the scalar path
@pytest.mark.parametrize("offsets", [(0, 0), (8, 4), (4, 8), (1, 1)],
                         ids=["v32", "v16", "chunk-src8", "scalar"])
def test_cast_to_f32_bit_exact(tb, dtype, n, offsets):
    so, do = offsets
    src = _src(n, dtype, so, seed=n)
    dst = torch.full((n + do,), float("nan"), device="cuda")[do:]
    tb.tb_cast_to_f32(src, dst, scale=1 / 1024.0)
    raw = src.view(torch.int32 if dtype == torch.float32 else torch.int16).cpu().numpy()
    ref = oracle.cast_to_f32(raw.view(np.float32 if dtype == torch.float32 else np.uint16),
                             KIND[dtype], 1 / 1024.0)
    assert np.array_equal(dst.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, (1 << 20) + 3])
# (source offset, destination offset) in elements: the chunk path needs a 16-byte aligned
# source and an 8-byte aligned destination; the others take the scalar loop
@pytest.mark.parametrize("offsets", [(0, 0), (0, 4), (4, 0), (1, 1), (0, 1)],
                         ids=["chunk", "chunk-dst8", "chunk-src16", "scalar", "scalar-dst"])
def test_cast_from_f32_bit_exact(tb, dtype, n, offsets):
    so, do = offsets
    src = _src(n, torch.float32, so, seed=n + 1)
    dst = torch.empty(n + do, dtype=dtype, device="cuda")[do:]
    tb.tb_cast_from_f32(src, dst)
    ref = oracle.cast_from_f32(src.cpu().numpy(), KIND[dtype])
    assert np.array_equal(to_bits(dst), ref)


def _plan(tb, st, with_copy=True, grads=None):
    k = len(st.sizes)
    g = grads if grads is not None else st.grad
    return tb.tb_adamw_plan_create(
        [st.tensor("theta", i) for i in range(k)], [st.tensor("m", i) for i in range(k)],
        [st.tensor("v", i) for i in range(k)],
        [g.narrow(0, st.offsets[i], st.sizes[i]) for i in range(k)],
        [st.tensor("copy", i) if with_copy else None for i in range(k)])


@pytest.mark.parametrize("align", [1, 128])
def test_fp32_gradients_match_oracle(tb, synth, align):
    sizes = [1, 9, 4096, 30001]
    st = synth.make_adamw_state([(f"t{i}", (n,)) for i, n in enumerate(sizes)], seed=3,
                                device="cuda", grad_dtype=torch.bfloat16, align=align)
    g32 = st.grad.float()                     # bf16 values, held as fp32 gradients
    plan = _plan(tb, st, grads=g32)
    live = np.concatenate([np.arange(o, o + n) for o, n in zip(st.offsets, st.sizes)])
    it = torch.from_numpy(live).cuda()
    th = st.theta.index_select(0, it).double().cpu().numpy()
    m = np.zeros_like(th)
    v = np.zeros_like(th)
    gb = to_bits(st.grad.index_select(0, it))
    tb.tb_adamw_step(plan, 1, inv_loss_scale=1 / 65536.0, **HP)
    cb, _ = oracle.adamw_step_f64(th, m, v, gb, "bf16", 1 / 65536.0, 1, **HP)
    torch.cuda.synchronize()
    got = st.theta.index_select(0, it).double().cpu().numpy()
    assert floored_rel(got, th) <= 1e-5
    assert torch.all(g32.index_select(0, it) == 0)
    assert np.array_equal(to_bits(st.copy.index_select(0, it)), oracle.encode16(got, "bf16"))


def test_unfused_pipeline_equals_fused_step_bitwise(tb, synth):
    shapes = synth.gpt2_small_shapes()[:20]
    a = synth.make_adamw_state(shapes, seed=4, device="cuda")
    b = synth.make_adamw_state(shapes, seed=4, device="cuda")
    pa = _plan(tb, a)
    g32 = torch.zeros(b.grad.numel(), device="cuda")
    pb = _plan(tb, b, with_copy=False, grads=g32)
    for t in (1, 2, 3):
        synth.fill_grads(a, t)
        synth.fill_grads(b, t)
        tb.tb_adamw_step(pa, t, inv_loss_scale=1 / 65536.0, **HP)
        sentinel = b.copy.clone()
        tb.tb_cast_to_f32(b.grad, g32, scale=1 / 65536.0)          # the loop's unscale cast
        tb.tb_adamw_step(pb, t, inv_loss_scale=1.0, **HP)         # step 8: fp32 AdamW, no copy
        torch.cuda.synchronize()
        assert torch.equal(b.copy, sentinel)                      # the step wrote no copy
        tb.tb_cast_from_f32(b.theta, b.copy)                      # the loop's copy-back cast
    torch.cuda.synchronize()
    for k in ("theta", "m", "v"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    live = torch.zeros(a.copy.numel(), dtype=torch.bool, device="cuda")
    for o, n in zip(a.offsets, a.sizes):
        live[o:o + n] = True
    assert torch.equal(a.copy[live], b.copy[live])
