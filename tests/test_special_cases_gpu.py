"""Special cases whose results are exact, so the kernels must reproduce them bit for bit
whatever their summation order:

* softmax backward of one-hot rows of P: the row's dot product is dY at the hot
  column, so every element of dX is exactly zero, +0 or -0 (dense and causal entry
  points);
* LayerNorm backward with gamma = 0: dxhat = 0, so dX is exactly zero while dgamma
  and dbeta still follow dY;
* LayerNorm and RMSNorm backward with dY = 0: every output is exactly zero;
* AdamW with zero gradients, no decay and eps > 0: the update is 0 / eps = 0, so
  theta stays as it was, m and v stay zero, and the copy is RNE(theta).
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import floored_rel, to_bits

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.bfloat16, torch.float16]
IDS = ["f32", "bf16", "f16"]


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


def _zero_bits(t):
    """Every element is +0 (the bit pattern)."""
    return bool((t.view(torch.int32 if t.element_size() == 4 else torch.int16) == 0).all())


def _zero(t):
    """Every element is +0 or -0 (a product of +0 and a negative value is -0); NaN fails."""
    return bool((t == 0).all())


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
@pytest.mark.parametrize("rows, cols", [(300, 1024), (77, 1000), (9, 20000), (513, 8)])
def test_softmax_one_hot_rows_give_exact_zero(tb, rows, cols, dtype):
    g = torch.Generator(device="cuda").manual_seed(rows + cols)
    hot = torch.randint(0, cols, (rows,), device="cuda", generator=g)
    P = torch.zeros(rows, cols, device="cuda", dtype=dtype)
    P[torch.arange(rows, device="cuda"), hot] = 1
    dY = torch.randn(rows, cols, device="cuda", generator=g).to(dtype)
    dX = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd(dY, P, dX)
    torch.cuda.synchronize()
    assert _zero(dX)
    # causal: row r open on its first r % cols + 1 columns, the hot column inside them
    hot_c = torch.minimum(hot, torch.arange(rows, device="cuda") % cols)
    Pc = torch.zeros_like(P)
    Pc[torch.arange(rows, device="cuda"), hot_c] = 1
    dXc = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd_causal(dY, Pc, dXc, period=cols)
    torch.cuda.synchronize()
    assert _zero(dXc)


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
@pytest.mark.parametrize("rows, D", [(1000, 768), (333, 4096), (37, 10000)])
def test_layernorm_zero_gamma_gives_zero_dx(tb, synth, rows, D, dtype):
    x, dY, mean, rstd, _ = synth.layernorm_inputs(rows, D, dtype, seed=D, device="cuda")
    gamma = torch.zeros(D, device="cuda")
    dX = torch.full_like(x, float("nan"))
    dg = torch.full((D,), float("nan"), device="cuda")
    db = torch.full((D,), float("nan"), device="cuda")
    ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, dtype), dtype=torch.uint8,
                     device="cuda")
    tb.tb_layernorm_bwd(dY, x, mean, rstd, gamma, dX, dg, db, ws)
    torch.cuda.synchronize()
    assert _zero(dX)
    args = [t.double().cpu().numpy() for t in (dY, x, mean, rstd, gamma)]
    _, rdg, rdb = oracle.layernorm_bwd_f64(*args)
    assert floored_rel(dg.double().cpu().numpy(), rdg) <= 1e-3
    assert floored_rel(db.double().cpu().numpy(), rdb) <= 1e-3


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_norms_of_zero_dy_are_zero(tb, synth, dtype):
    rows, D = 2048, 4096
    x, _, mean, rstd, gamma = synth.layernorm_inputs(rows, D, dtype, seed=3, device="cuda")
    dY = torch.zeros_like(x)
    dX = torch.full_like(x, float("nan"))
    dg = torch.full((D,), float("nan"), device="cuda")
    db = torch.full((D,), float("nan"), device="cuda")
    ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, dtype), dtype=torch.uint8,
                     device="cuda")
    tb.tb_layernorm_bwd(dY, x, mean, rstd, gamma, dX, dg, db, ws)
    xr, _, inv, gr = synth.rmsnorm_inputs(rows, D, dtype, seed=4, device="cuda")
    rdX = torch.full_like(xr, float("nan"))
    rdg = torch.full((D,), float("nan"), device="cuda")
    rws = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(rows, D, dtype), dtype=torch.uint8,
                      device="cuda")
    tb.tb_rmsnorm_bwd(torch.zeros_like(xr), xr, inv, gr, rdX, rdg, rws)
    torch.cuda.synchronize()
    for t in (dX, dg, db, rdX, rdg):
        assert _zero(t)


def test_adamw_zero_gradients_without_decay_leave_theta(tb, synth):
    st = synth.make_adamw_state(synth.gpt2_small_shapes()[:12], seed=82, device="cuda")
    k = len(st.sizes)
    plan = tb.tb_adamw_plan_create(*[[st.tensor(a, i) for i in range(k)]
                                     for a in ("theta", "m", "v", "grad", "copy")])
    theta0 = st.theta.clone()
    for t in (1, 2, 3):
        st.grad.zero_()
        tb.tb_adamw_step(plan, t, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                         inv_loss_scale=1 / 65536.0)
    torch.cuda.synchronize()
    plan.close()
    for i in range(k):
        th = st.tensor("theta", i)
        assert torch.equal(th, theta0.narrow(0, st.offsets[i], st.sizes[i]))
        assert _zero_bits(st.tensor("m", i)) and _zero_bits(st.tensor("v", i))
        want = oracle.encode16(th.double().cpu().numpy(), "bf16")
        assert np.array_equal(to_bits(st.tensor("copy", i)), want)
