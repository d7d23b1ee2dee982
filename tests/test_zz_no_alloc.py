"""LayerNorm backward without any allocation (tb_layernorm_bwd_noalloc).

Some callers cannot allocate device memory where they run the backward -- code
inside a framework that owns all device memory through its own pool, or a step
loop that must not call cudaMalloc/cudaFree because those can synchronise with
the device.  They have no workspace to pass, so this entry point keeps its
scratch in a fixed array inside the library.  These checks call it through the
C ABI and compare it with the workspace entry point, twice in a row (the second
call finds the previous call's partial sums still in the shared array), within
the tolerances the other LayerNorm tests use, and then the second call's output
with the CPU oracle under the same rules.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import floored_rel, layernorm_dx_err_bound, lowp_check, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


def _with_workspace(tb, x, dY, mean, rstd, gamma):
    rows, D = x.shape
    dX = torch.empty_like(x)
    dg = torch.empty(D, device=x.device)
    db = torch.empty(D, device=x.device)
    ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, x.dtype), dtype=torch.uint8,
                     device=x.device)
    tb.tb_layernorm_bwd(dY, x, mean, rstd, gamma, dX, dg, db, ws)
    return dX, dg, db


def _without_allocation(tb, x, dY, mean, rstd, gamma):
    D = x.shape[1]
    dX = torch.full_like(x, float("nan"))
    dg = torch.full((D,), float("nan"), device=x.device)
    db = torch.full((D,), float("nan"), device=x.device)
    tb.tb_layernorm_bwd_noalloc(dY, x, mean, rstd, gamma, dX, dg, db)
    return dX, dg, db


def _close(a, b):
    (dxa, dga, dba), (dxb, dgb, dbb) = a, b
    assert floored_rel(dga.double().cpu().numpy(), dgb.double().cpu().numpy()) <= 1e-3
    assert floored_rel(dba.double().cpu().numpy(), dbb.double().cpu().numpy()) <= 1e-3
    if dxa.dtype == torch.float32:
        assert floored_rel(dxa.double().cpu().numpy(), dxb.double().cpu().numpy()) <= 1e-4
    else:
        kind = "bf16" if dxa.dtype == torch.bfloat16 else "f16"
        ok, _, _ = lowp_check(to_bits(dxa), dxb.double().cpu().numpy(), kind)
        assert ok.all()


@pytest.mark.parametrize("rows, D, dtype", [
    (16384, 4096, torch.bfloat16),   # partials fit with the usual grid: bitwise equal
    (4096, 8192, torch.float32),     # rows split over a two-CTA cluster
    (1024, 12288, torch.bfloat16),   # rows split over a three-CTA cluster: bitwise equal
    (300, 1004, torch.float16),      # 2,008-byte rows, not a multiple of 16 bytes: plain-load path
    (512, 12300, torch.bfloat16),    # plain path; partials of 2 CTAs/SM exceed 16 MiB: fewer CTAs
], ids=["16384x4096-bf16", "4096x8192-f32", "1024x12288-bf16", "300x1004-f16", "512x12300-bf16"])
def test_matches_workspace_entry_point_twice(tb, synth, rows, D, dtype):
    args = synth.layernorm_inputs(rows, D, dtype, seed=rows + D, device="cuda", dy_std=1e-2)
    ref = _with_workspace(tb, *args)
    for _ in range(2):
        got = _without_allocation(tb, *args)
        torch.cuda.synchronize()
        _close(got, ref)
    if (rows, D) in ((16384, 4096), (1024, 12288)):
        for u, w in zip(got, ref):
            assert torch.equal(u, w)
    # and against the oracle directly (float64 LayerNorm backward on the same inputs)
    x, dY, mean, rstd, gamma = (t.double().cpu().numpy() for t in args)
    rdx, rdg, rdb = oracle.layernorm_bwd_f64(dY, x, mean, rstd, gamma)
    dX, dg, db = got
    assert floored_rel(dg.double().cpu().numpy(), rdg) <= 1e-3
    assert floored_rel(db.double().cpu().numpy(), rdb) <= 1e-3
    if dX.dtype == torch.float32:
        assert floored_rel(dX.double().cpu().numpy(), rdx) <= 1e-4
    else:
        kind = "bf16" if dX.dtype == torch.bfloat16 else "f16"
        ok, _, _ = lowp_check(to_bits(dX), rdx, kind,
                              layernorm_dx_err_bound(x, dY, mean, rstd, gamma))
        assert ok.all()
    assert tb.tb_device_error(reset=True) == 0


def test_rejects_rows_longer_than_the_scratch_holds(tb):
    D = (16 << 20) // 8 + 16            # one CTA would need 2*D floats > 16 MiB
    x = torch.zeros(1, D, device="cuda")
    mean = torch.zeros(1, device="cuda")
    g = torch.ones(D, device="cuda")
    with pytest.raises(tb.TbError) as ei:
        tb.tb_layernorm_bwd_noalloc(x, x.clone(), mean, mean.clone(), g, torch.empty_like(x),
                                    torch.empty(D, device="cuda"), torch.empty(D, device="cuda"))
    assert ei.value.code == 5           # TB_ERR_WORKSPACE
