"""GPU parity of the fused multi-tensor AdamW step against the CPU oracle.

Targets: fp32 theta/m/v within 1e-5 floored relative error of the float64
oracle after the stated number of steps, the 16-bit working copy within one
16-bit ulp of the oracle's theta rounded to nearest even, and the gradient
zeroed bit-exactly after every step.  Sizes: the tiny flat tensor (every
element compared), ragged / misaligned tables, the GPT-2-small table for 100
steps and the Llama-7B table for 20 steps (sampled windows replayed by the
oracle), plus determinism, resume and NaN-confinement checks.
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import floored_rel, lowp_check, to_bits

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
KIND = {torch.bfloat16: "bf16", torch.float16: "f16"}


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
    return tb.tb_adamw_plan_create([st.tensor("theta", i) for i in range(k)],
                                   [st.tensor("m", i) for i in range(k)],
                                   [st.tensor("v", i) for i in range(k)],
                                   [st.tensor("grad", i) for i in range(k)],
                                   [st.tensor("copy", i) for i in range(k)])


def _windows(st, edge=2048, n_random=0, rlen=32768, seed=0):
    """Arena indices to compare: each tensor's first and last `edge` elements,
    plus random windows inside the larger tensors."""
    rng = np.random.default_rng(seed)
    parts = []
    for off, n in zip(st.offsets, st.sizes):
        if n == 0:
            continue
        parts.append(np.arange(off, off + min(n, edge)))
        if n > edge:
            parts.append(np.arange(off + max(edge, n - edge), off + n))
    big = [(o, n) for o, n in zip(st.offsets, st.sizes) if n > 4 * rlen]
    for _ in range(n_random if big else 0):
        o, n = big[rng.integers(len(big))]
        s = int(rng.integers(0, n - rlen))
        parts.append(np.arange(o + s, o + s + rlen))
    return np.unique(np.concatenate(parts))


def _all_live(st):
    return np.concatenate([np.arange(o, o + n) for o, n in zip(st.offsets, st.sizes) if n > 0])


def _run(tb, synth, st, steps, idx, first_step=1, hp=None):
    """Runs `steps` GPU steps and the oracle on arena indices `idx`; returns errors."""
    hp = HP if hp is None else hp
    dev = st.theta.device
    gkind, ckind = KIND[st.grad.dtype], KIND[st.copy.dtype]
    inv = 1.0 / st.loss_scale
    plan = _plan(tb, st)
    it = torch.from_numpy(idx).to(dev)
    th = st.theta.index_select(0, it).double().cpu().numpy()
    m = st.m.index_select(0, it).double().cpu().numpy()
    v = st.v.index_select(0, it).double().cpu().numpy()
    for t in range(first_step, first_step + steps):
        if t != 1:
            synth.fill_grads(st, t)
        gb = to_bits(st.grad.index_select(0, it))
        tb.tb_adamw_step(plan, t, inv_loss_scale=inv, **hp)
        cb, _ = oracle.adamw_step_f64(th, m, v, gb, gkind, inv, t, copy_kind=ckind, **hp)
        torch.cuda.synchronize()
        gz = to_bits(st.grad.index_select(0, it))
        assert np.all(gz == 0), f"gradient not zeroed at step {t}"
        # every element of every tensor, not only the sampled ones: each tile was visited
        ity = torch.int16 if st.grad.element_size() == 2 else torch.int32
        assert all(bool((st.tensor("grad", i).view(ity) == 0).all())
                   for i in range(len(st.sizes)) if st.sizes[i] > 0), \
            f"gradient not zeroed everywhere at step {t}"
    plan.close()
    got_th = st.theta.index_select(0, it).double().cpu().numpy()
    got_m = st.m.index_select(0, it).double().cpu().numpy()
    got_v = st.v.index_select(0, it).double().cpu().numpy()
    got_c = to_bits(st.copy.index_select(0, it))
    # (a) the copy is exactly the round-to-nearest-even of the kernel's own fp32 master
    copy_exact = bool(np.array_equal(got_c, oracle.encode16(got_th, ckind)))
    # (b) within one 16-bit ulp of the oracle's master rounded to nearest even, or --
    #     where theta has decayed far below its starting scale -- the rounding of a
    #     value within the theta tolerance (1e-5, floored at rms) of the oracle
    rms = np.sqrt(np.mean(th * th))
    tol = 1e-5 * np.maximum(np.abs(th), rms)
    ok, n_tol, dmax = lowp_check(got_c, th, ckind, err=tol)
    ok_1ulp, _, _ = lowp_check(got_c, th, ckind)
    widened = ok & ~ok_1ulp          # pass only under the widened rule
    return dict(theta=floored_rel(got_th, th), m=floored_rel(got_m, m), v=floored_rel(got_v, v),
                copy_exact=copy_exact, copy_ok=bool(ok.all()), copy_max_ulps=dmax,
                copy_beyond_1ulp=n_tol,
                copy_widened_max_theta_over_rms=float(np.max(np.abs(th[widened])) / rms)
                if widened.any() else 0.0)


def _assert_within_targets(err):
    assert err["theta"] <= 1e-5, err
    assert err["m"] <= 1e-5, err
    assert err["v"] <= 1e-5, err
    assert err["copy_exact"], err
    assert err["copy_ok"], err
    # The widened copy rule covers only parameters that have decayed below the rms
    # of their tensor set: a copy more than 1 ulp off anywhere else fails.
    assert err["copy_widened_max_theta_over_rms"] < 1.0, err
    print(f"copies beyond 1 ulp (widened rule): {err['copy_beyond_1ulp']}, "
          f"largest |theta|/rms among them: {err['copy_widened_max_theta_over_rms']:.3g}")


# ----------------------------------------------------------------------------- tiny config
def test_tiny_flat_tensor_10_steps(tb, synth):
    """1,048,576 params, fp16 grads = N(0,1e-3)*1024, bf16 copy, 10 steps, every element."""
    st = synth.make_adamw_state([("w", (1 << 20,))], seed=0, device="cuda",
                                grad_dtype=torch.float16, copy_dtype=torch.bfloat16,
                                grad_std=1e-3, loss_scale=1024.0)
    err = _run(tb, synth, st, 10, _all_live(st))
    _assert_within_targets(err)


def test_tiny_flat_tensor_fp16_copy(tb, synth):
    st = synth.make_adamw_state([("w", (1 << 20,))], seed=1, device="cuda",
                                grad_dtype=torch.float16, copy_dtype=torch.float16,
                                grad_std=1e-3, loss_scale=1024.0)
    _assert_within_targets(_run(tb, synth, st, 3, _all_live(st)))


@pytest.mark.parametrize("align", [1, 3, 128])
def test_ragged_and_misaligned_tables(tb, synth, align):
    """Tensor sizes around the 8-element unit, empty tensors, and arenas packed
    with no alignment (most tensors then take the scalar path)."""
    sizes = [1, 7, 8, 9, 0, 15, 16, 17, 1000, 8191, 8193, 0, 65541, 3, 300_007]
    shapes = [(f"t{i}", (n,)) for i, n in enumerate(sizes)]
    st = synth.make_adamw_state(shapes, seed=2, device="cuda", grad_std=1e-3,
                                loss_scale=65536.0, align=align)
    _assert_within_targets(_run(tb, synth, st, 4, _all_live(st)))


def test_bf16_grads_bf16_copy_many_small_tensors(tb, synth):
    shapes = [(f"t{i}", (int(n),)) for i, n in enumerate(np.random.default_rng(3).integers(1, 5000, 700))]
    st = synth.make_adamw_state(shapes, seed=3, device="cuda", grad_std=1e-3, loss_scale=65536.0)
    _assert_within_targets(_run(tb, synth, st, 3, _all_live(st)))


# ----------------------------------------------------------------------------- full-size configs
def test_gpt2_small_table_100_steps(tb, synth):
    """148 tensors, 124,439,808 params, bf16 grads * 65536, steps 1..100."""
    shapes = synth.gpt2_small_shapes()
    st = synth.make_adamw_state(shapes, seed=0, device="cuda", grad_std=1e-3, loss_scale=65536.0)
    assert len(st.sizes) == 148 and st.n_params == 124_439_808
    idx = _windows(st, edge=2048, n_random=24)
    _assert_within_targets(_run(tb, synth, st, 100, idx))


def test_llama7b_table_20_steps(tb, synth):
    """291 tensors, 6,738,415,616 params (~108 GB of state), bf16 grads * 65536 with
    sigma 1e-4, steps 1..20, in the launch configuration the benchmark times."""
    shapes = synth.llama7b_shapes()
    st = synth.make_adamw_state(shapes, seed=0, device="cuda", grad_std=1e-4, loss_scale=65536.0)
    assert len(st.sizes) == 291 and st.n_params == 6_738_415_616
    idx = _windows(st, edge=1024, n_random=32, rlen=65536)
    err = _run(tb, synth, st, 20, idx)
    del st
    torch.cuda.empty_cache()
    _assert_within_targets(err)


# ----------------------------------------------------------------------------- properties
def _clone_state(st):
    import copy
    c = copy.copy(st)
    for k in ("theta", "m", "v", "grad", "copy"):
        setattr(c, k, getattr(st, k).clone())
    return c


def test_deterministic_bitwise(tb, synth):
    st = synth.make_adamw_state(synth.gpt2_small_shapes()[:20], seed=4, device="cuda")
    st2 = _clone_state(st)
    for s in (st, st2):
        p = _plan(tb, s)
        for t in (1, 2, 3):
            synth.fill_grads(s, t)
            tb.tb_adamw_step(p, t, inv_loss_scale=1 / 65536.0, **HP)
        p.close()
    torch.cuda.synchronize()
    for k in ("theta", "m", "v", "copy", "grad"):
        assert torch.equal(getattr(st, k), getattr(st2, k)), k


def test_resume_is_bitwise(tb, synth):
    """10 steps straight == 5 steps, state copied to fresh buffers, 5 more steps."""
    shapes = [("a", (3001,)), ("b", (64, 64))]
    a = synth.make_adamw_state(shapes, seed=5, device="cuda")
    b = _clone_state(a)
    pa = _plan(tb, a)
    for t in range(1, 11):
        synth.fill_grads(a, t)
        tb.tb_adamw_step(pa, t, inv_loss_scale=1 / 65536.0, **HP)
    pb = _plan(tb, b)
    for t in range(1, 6):
        synth.fill_grads(b, t)
        tb.tb_adamw_step(pb, t, inv_loss_scale=1 / 65536.0, **HP)
    pb.close()
    c = _clone_state(b)          # "checkpoint": copy theta/m/v out, resume from the copy
    del b
    pc = _plan(tb, c)
    for t in range(6, 11):
        synth.fill_grads(c, t)
        tb.tb_adamw_step(pc, t, inv_loss_scale=1 / 65536.0, **HP)
    torch.cuda.synchronize()
    for k in ("theta", "m", "v", "copy"):
        assert torch.equal(getattr(a, k), getattr(c, k)), k


def test_nan_gradient_stays_confined(tb, synth):
    shapes = [("a", (4096,))]
    a = synth.make_adamw_state(shapes, seed=6, device="cuda")
    b = _clone_state(a)
    a.grad[123] = float("nan")
    for s in (a, b):
        p = _plan(tb, s)
        tb.tb_adamw_step(p, 1, inv_loss_scale=1 / 65536.0, **HP)
        p.close()
    torch.cuda.synchronize()
    assert torch.isnan(a.theta[123]) and torch.isnan(a.m[123]) and torch.isnan(a.v[123])
    keep = torch.ones(a.theta.numel(), dtype=torch.bool, device="cuda")
    keep[123] = False
    for k in ("theta", "m", "v", "copy"):
        assert torch.equal(getattr(a, k)[keep], getattr(b, k)[keep]), k


def test_step_argument_errors(tb, synth):
    st = synth.make_adamw_state([("a", (64,))], seed=7, device="cuda")
    p = _plan(tb, st)
    with pytest.raises(tb.TbError):
        tb.tb_adamw_step(p, 0, inv_loss_scale=1.0, **HP)
    with pytest.raises(tb.TbError):
        tb.tb_adamw_step(p, 1, inv_loss_scale=1.0, lr=1e-3, beta1=1.0, beta2=0.999, eps=1e-8,
                         weight_decay=0.0)
    with pytest.raises(tb.TbError):
        tb.tb_adamw_step(p, 1, inv_loss_scale=-1.0, **HP)
    p.close()


def test_plan_of_empty_tensors_is_a_no_op(tb):
    """A plan whose tensors all have n = 0: every call succeeds and launches nothing
    that could fail; the gradient norm of nothing is 0 with a clip factor of 1."""
    empty = [torch.empty(0, device="cuda") for _ in range(3)]
    g = [torch.empty(0, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    c = [torch.empty(0, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    plan = tb.tb_adamw_plan_create(empty[:2], empty[1:3], empty[:2], g, c)
    tb.tb_adamw_step(plan, 1, inv_loss_scale=1.0, **HP)
    out = torch.full((3,), float("nan"), device="cuda")
    ws = torch.empty(max(tb.tb_adamw_grad_norm_workspace_size(plan), 1), dtype=torch.uint8,
                     device="cuda")
    tb.tb_adamw_grad_norm(plan, 1.0, 1.0, out, ws)
    tb.tb_adamw_step_clipped(plan, 1, inv_loss_scale=1.0, clip=out, **HP)
    torch.cuda.synchronize()
    assert out.tolist() == [0.0, 1.0, 0.0]
    plan.close()
    # nothing left behind: a following call still reports success
    P = torch.full((4, 8), 0.125, device="cuda")
    dX = torch.empty_like(P)
    tb.tb_softmax_bwd(torch.ones_like(P), P, dX)
    torch.cuda.synchronize()
    assert torch.all(dX == 0)


def test_tile_counter_is_reset_on_every_path(tb, synth):
    """The step kernel's CTAs claim tiles from a counter in the plan that each call
    clears before its launch.  After every kind of call (a device step that returns early for t < 1,
    a step skipped for a non-finite gradient, plain, clipped and device steps) the next
    step must still visit every element: each step leaves every gradient element +0.
    Two tables: one with many more tiles than CTAs, one with a single tile."""
    for shapes in (synth.gpt2_small_shapes()[:30], [("a", (4096,)), ("b", (77,))]):
        st = synth.make_adamw_state(shapes, seed=71, device="cuda")
        plan = _plan(tb, st)
        k = len(st.sizes)
        clip = torch.zeros(3, device="cuda")
        ws = torch.empty(tb.tb_adamw_grad_norm_workspace_size(plan), dtype=torch.uint8,
                         device="cuda")
        inv = 1 / 65536.0

        def grads_zero():
            torch.cuda.synchronize()
            return all(bool((st.tensor("grad", i) == 0).all()) for i in range(k))

        def clipped(t):
            tb.tb_adamw_grad_norm(plan, inv, 1.0, clip, ws)
            tb.tb_adamw_step_clipped(plan, t, inv_loss_scale=inv, clip=clip, **HP)

        calls = [
            ("device step with t = 0", False,
             lambda: tb.tb_adamw_step_device(plan, torch.zeros(1, dtype=torch.int64, device="cuda"),
                                             inv_loss_scale=inv, **HP)),
            ("plain step", True, lambda: tb.tb_adamw_step(plan, 1, inv_loss_scale=inv, **HP)),
            ("clipped step", True, lambda: clipped(2)),
            ("skipped step", True, lambda: clipped(3)),
            ("device step", True,
             lambda: tb.tb_adamw_step_device(plan, torch.full((1,), 3, dtype=torch.int64, device="cuda"),
                                             inv_loss_scale=inv, **HP)),
            ("plain step again", True, lambda: tb.tb_adamw_step(plan, 4, inv_loss_scale=inv, **HP)),
        ]
        for i, (name, runs, call) in enumerate(calls):
            synth.fill_grads(st, i + 2)
            if name == "skipped step":
                st.tensor("grad", k - 1)[-1] = float("inf")
            before = st.theta.clone()
            call()
            if runs:
                assert grads_zero(), f"{name}: some gradient elements were not visited"
            else:
                assert not grads_zero() and torch.equal(st.theta, before), name
            if name == "skipped step":
                assert clip[2].item() == 1.0 and torch.equal(st.theta, before)
        assert tb.tb_device_error(reset=True) == 1      # from the t = 0 call
        plan.close()


def test_steps_of_one_plan_on_two_streams_ordered_by_events(tb, synth):
    """Steps of one plan alternate between two streams, each waiting for the other;
    the result equals the same steps on one stream, bit for bit."""
    shapes = synth.gpt2_small_shapes()[:16]
    a = synth.make_adamw_state(shapes, seed=72, device="cuda")
    b = synth.make_adamw_state(shapes, seed=72, device="cuda")
    pa, pb = _plan(tb, a), _plan(tb, b)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for t in range(1, 7):
        synth.fill_grads(a, t)
        synth.fill_grads(b, t)
        torch.cuda.synchronize()
        tb.tb_adamw_step(pa, t, inv_loss_scale=1 / 65536.0, **HP)
        s, other = (s1, s2) if t % 2 else (s2, s1)
        s.wait_stream(other)
        tb.tb_adamw_step(pb, t, inv_loss_scale=1 / 65536.0, stream=s, **HP)
        torch.cuda.synchronize()
    for key in ("theta", "m", "v", "copy", "grad"):
        assert torch.equal(getattr(a, key), getattr(b, key)), key
    pa.close()
    pb.close()


@pytest.mark.parametrize("hp", [
    dict(lr=1e-3, beta1=0.0, beta2=0.999, eps=1e-8, weight_decay=0.01),
    dict(lr=1e-3, beta1=0.9, beta2=0.0, eps=1e-8, weight_decay=0.01),
    dict(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=0.0, weight_decay=0.0),
    dict(lr=0.5, beta1=0.5, beta2=0.75, eps=1e-3, weight_decay=0.5),
], ids=["beta1=0", "beta2=0", "lr=0", "eps=0-no-decay", "large"])
def test_hyperparameter_edges(tb, synth, hp):
    """The ends of the accepted ranges (beta = 0 makes m or v the last gradient alone,
    lr = 0 leaves theta exactly as it was, eps = 0 divides by sqrt(v_hat) alone) and
    large values, against the oracle on every element over 5 steps."""
    st = synth.make_adamw_state([("a", (4096,)), ("b", (1000,)), ("c", (7,))], seed=81,
                                device="cuda")
    theta0 = st.theta.clone()
    err = _run(tb, synth, st, 5, _all_live(st), hp=hp)
    _assert_within_targets(err)
    if hp["lr"] == 0.0:
        assert torch.equal(st.theta, theta0)


def test_tile_counter_over_a_long_mix_of_calls(tb, synth):
    """200 calls on one plan, cycling through plain, clipped and device-counter steps and
    replays of a captured graph; after every call each gradient element is +0 (every tile
    was visited, so the counter started each launch at zero)."""
    st = synth.make_adamw_state(synth.gpt2_small_shapes()[:8], seed=73, device="cuda")
    plan = _plan(tb, st)
    k = len(st.sizes)
    inv = 1 / 65536.0
    clip = torch.zeros(3, device="cuda")
    ws = torch.empty(tb.tb_adamw_grad_norm_workspace_size(plan), dtype=torch.uint8, device="cuda")
    step = torch.zeros(1, dtype=torch.int64, device="cuda")

    def device_step():
        step.add_(1)
        tb.tb_adamw_grad_norm(plan, inv, 1.0, clip, ws)
        tb.tb_adamw_step_device(plan, step, inv_loss_scale=inv, clip=clip, **HP)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        device_step()                       # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        device_step()
    ity = torch.int16
    for i in range(200):
        synth.fill_grads(st, i + 2)
        kind = i % 4
        if kind == 0:
            tb.tb_adamw_step(plan, i + 1, inv_loss_scale=inv, **HP)
        elif kind == 1:
            tb.tb_adamw_grad_norm(plan, inv, 1.0, clip, ws)
            tb.tb_adamw_step_clipped(plan, i + 1, inv_loss_scale=inv, clip=clip, **HP)
        elif kind == 2:
            device_step()
        else:
            graph.replay()
        torch.cuda.synchronize()
        assert all(bool((st.tensor("grad", j).view(ity) == 0).all()) for j in range(k)), (i, kind)
    assert tb.tb_device_error(reset=True) == 0
    plan.close()
