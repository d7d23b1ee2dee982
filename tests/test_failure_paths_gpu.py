"""Failure detection without a GPU fault.

* The LayerNorm ring kernel's waits on its own bulk copies are bounded: the
  self-test entry runs it with the copies withheld, so every wait runs out after
  a short limit; the kernel reports TB_ERR_TIMEOUT through the device error
  word and returns, and the context stays usable for the next call.
* A destroyed AdamW plan is rejected by every call that takes a plan, without
  being dereferenced.
* A stale value in an AdamW plan's tile counter (what a launch that stopped
  part-way would leave) is planted from the host; the next step still updates and
  zeroes every element, bit for bit as a plan whose counter was never touched.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tolerance import floored_rel

pytestmark = pytest.mark.gpu

TB_ERR_INVALID_VALUE, TB_ERR_TIMEOUT = 1, 9


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


def test_bounded_wait_runs_out_and_the_context_stays_usable(tb, synth):
    assert tb.tb_device_error(reset=True) in (0, TB_ERR_TIMEOUT)
    tb.tb_layernorm_bwd_selftest_timeout(wait_limit_ns=2_000_000)
    assert tb.tb_device_error(reset=True) == TB_ERR_TIMEOUT
    assert tb.tb_device_error(reset=True) == 0
    # the next call runs normally and is correct
    x, dY, mean, rstd, gamma = synth.layernorm_inputs(64, 256, torch.float32, seed=31, device="cuda")
    dX = torch.empty_like(x)
    dg = torch.empty(256, device="cuda")
    db = torch.empty(256, device="cuda")
    ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(64, 256, torch.float32), dtype=torch.uint8,
                     device="cuda")
    tb.tb_layernorm_bwd(dY, x, mean, rstd, gamma, dX, dg, db, ws)
    torch.cuda.synchronize()
    assert tb.tb_device_error(reset=True) == 0
    args = [t.double().cpu().numpy() for t in (dY, x, mean, rstd, gamma)]
    rdx, rdg, rdb = oracle.layernorm_bwd_f64(*args)
    assert floored_rel(dX.double().cpu().numpy(), rdx) <= 1e-4
    assert floored_rel(dg.double().cpu().numpy(), rdg) <= 1e-3
    assert floored_rel(db.double().cpu().numpy(), rdb) <= 1e-3


def test_selftest_rejects_a_limit_out_of_range(tb):
    for bad in (0, 999, 1_000_000_001):
        with pytest.raises(tb.TbError) as e:
            tb.tb_layernorm_bwd_selftest_timeout(wait_limit_ns=bad)
        assert e.value.code == TB_ERR_INVALID_VALUE


def test_destroyed_plan_is_rejected(tb, synth):
    st = synth.make_adamw_state([("a", (4096,))], seed=32, device="cuda")
    plan = tb.tb_adamw_plan_create([st.theta.narrow(0, 0, 4096)], [st.m.narrow(0, 0, 4096)],
                                   [st.v.narrow(0, 0, 4096)], [st.grad.narrow(0, 0, 4096)],
                                   [st.copy.narrow(0, 0, 4096)])
    stale = plan.handle
    lib = tb._binding.lib
    hp = tb._binding.tb_adamw_hparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert lib.tb_adamw_step(stale, 1, ctypes.byref(hp), 1.0, None) == 0
    torch.cuda.synchronize()
    plan.close()
    theta = st.theta.clone()
    assert lib.tb_adamw_step(stale, 2, ctypes.byref(hp), 1.0, None) == TB_ERR_INVALID_VALUE
    size = ctypes.c_size_t(0)
    assert lib.tb_adamw_grad_norm_workspace_size(stale, ctypes.byref(size)) == TB_ERR_INVALID_VALUE
    assert lib.tb_adamw_plan_destroy(stale) == TB_ERR_INVALID_VALUE
    clip = torch.zeros(3, device="cuda")
    assert lib.tb_adamw_step_clipped(stale, 2, ctypes.byref(hp), 1.0, clip.data_ptr(),
                                     None) == TB_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert torch.equal(theta, st.theta)     # nothing ran
    # a pointer that was never a plan
    assert lib.tb_adamw_step(ctypes.c_void_p(0x1000), 1, ctypes.byref(hp), 1.0,
                             None) == TB_ERR_INVALID_VALUE


def test_stale_tile_counter_is_cleared_before_the_next_step(tb, synth):
    # 3 tensors, 8.4 M params: about 520 tiles of 16,384 elements, more than the
    # persistent grid, so CTAs claim tiles from the counter
    shapes = [("a", (4096, 1024)), ("b", (4099,)), ("c", (1024, 4095))]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    runs = []
    for stale in (None, 1, 300, 2 ** 40):
        st = synth.make_adamw_state(shapes, seed=33, device="cuda")
        k = len(shapes)
        plan = tb.tb_adamw_plan_create(*[[st.tensor(a, i) for i in range(k)]
                                         for a in ("theta", "m", "v", "grad", "copy")])
        for t in (1, 2):
            synth.fill_grads(st, t)
            if stale is not None:
                tb.tb_adamw_selftest_stale_counter(plan, stale)
            tb.tb_adamw_step(plan, t, inv_loss_scale=1.0 / 65536.0, **hp)
            torch.cuda.synchronize()
            for i in range(k):
                assert int(torch.count_nonzero(st.tensor("grad", i))) == 0, (stale, t, i)
        runs.append((st.theta.clone(), st.m.clone(), st.v.clone(), st.copy.clone()))
        plan.close()
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)
