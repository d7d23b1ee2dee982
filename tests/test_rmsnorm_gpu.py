"""GPU parity of the RMSNorm backward against the CPU oracle.

Same targets as the LayerNorm backward: fp32 dX within 1e-4 floored relative
error, 16-bit dX within one 16-bit ulp of the oracle rounded to nearest even
(or the fp32 arithmetic's own bound where it cancels), dgamma within 1e-3
floored relative.  Sizes: 1024 x 256 fp32, 16,384 x 4,096 bf16 (the Llama-7B
hidden size, every element), a sweep of D over the ring and plain paths with
ragged row counts, zero rows, determinism and the workspace check.
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import floored_rel, lowp_check, to_bits, within_bound

pytestmark = pytest.mark.gpu

KIND = {torch.bfloat16: "bf16", torch.float16: "f16"}


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


def run(tb, x, dY, rs, gamma, ws_bytes=None):
    rows, D = x.shape
    dX = torch.full_like(x, float("nan"))
    dg = torch.full((D,), float("nan"), device=x.device)
    need = tb.tb_rmsnorm_bwd_workspace_size(rows, D, x.dtype)
    ws = torch.empty(max(need if ws_bytes is None else ws_bytes, 1), dtype=torch.uint8,
                     device=x.device)
    tb.tb_rmsnorm_bwd(dY, x, rs, gamma, dX, dg, ws)
    return dX, dg


def _err_bound(x, dY, rs, gamma):
    """Bound on |dX_fp32 - dX_exact|: a few roundings per term, the row sum at most
    D/32 + 64 rounded additions."""
    D = x.shape[1]
    xh = x * rs[:, None]
    dxh = dY * gamma[None, :]
    sb = np.sum(np.abs(dxh * xh), axis=1, keepdims=True) / D
    mb = np.abs(np.sum(dxh * xh, axis=1, keepdims=True)) / D
    u = 2.0 ** -24
    return rs[:, None] * (4 * u * (np.abs(dxh) + np.abs(xh) * mb) + (D / 32 + 64) * u * np.abs(xh) * sb)


def check(x, dY, rs, gamma, dX, dg):
    """fp32 dX must meet the 1e-4 floored relative target.  Only for D <= 2 may it
    instead sit within the derived fp32 error bound: at D = 1 the exact dX is
    proportional to eps (x_hat is +-1 up to eps) and cancels far below its terms."""
    xn, dYn = x.double().cpu().numpy(), dY.double().cpu().numpy()
    rn, gn = rs.double().cpu().numpy(), gamma.double().cpu().numpy()
    rdx, rdg = oracle.rmsnorm_bwd_f64(dYn, xn, rn, gn)
    assert floored_rel(dg.double().cpu().numpy(), rdg) <= 1e-3
    if dX.dtype == torch.float32:
        got = dX.double().cpu().numpy()
        e = floored_rel(got, rdx)
        if x.shape[1] > 2:
            assert e <= 1e-4, f"dX floored relative error {e}"
        elif e > 1e-4:
            ok = within_bound(got, rdx, _err_bound(xn, dYn, rn, gn))
            assert ok.all(), f"dX floored relative error {e}, {(~ok).sum()} beyond the fp32 bound"
    else:
        ok, _, dmax = lowp_check(to_bits(dX), rdx, KIND[dX.dtype], _err_bound(xn, dYn, rn, gn))
        assert ok.all(), f"{(~ok).sum()} dX elements off (max ulp distance {dmax})"


def test_small_fp32(tb, synth):
    args = synth.rmsnorm_inputs(1024, 256, torch.float32, seed=0, device="cuda")
    check(*args, *run(tb, *args))


def test_llama_hidden_bf16(tb, synth):
    """16,384 rows x D=4096 bf16, dY ~ N(0, 1e-2); every element compared."""
    args = synth.rmsnorm_inputs(16384, 4096, torch.bfloat16, seed=1, device="cuda", dy_std=1e-2)
    out = run(tb, *args)
    torch.cuda.synchronize()
    check(*args, *out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16],
                         ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("D", [1, 3, 8, 100, 256, 1000, 2048, 4096, 4104, 8192, 12288, 16384,
                               25600, 65536])
def test_feature_dim_sweep(tb, synth, D, dtype):
    for rows in (1, 7, 300):
        args = synth.rmsnorm_inputs(rows, D, dtype, seed=D + rows, device="cuda")
        check(*args, *run(tb, *args))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("D", [100, 1004, 4100, 8191, 8196])
def test_plain_path_shapes(tb, synth, D, dtype):
    """Odd row lengths and buffers one element off alignment: the register row
    kernel up to 8,192 columns, the last-resort kernel beyond."""
    for rows, shift in ((7, 1), (300, 0)):
        x0, dY0, rs, gamma = synth.rmsnorm_inputs(rows, D, dtype, seed=7 * D + rows, device="cuda")
        if shift:
            x = torch.empty(rows * D + shift, dtype=dtype, device="cuda")[shift:].view(rows, D)
            dY = torch.empty(rows * D + shift, dtype=dtype, device="cuda")[shift:].view(rows, D)
            x.copy_(x0)
            dY.copy_(dY0)
        else:
            x, dY = x0, dY0
        check(x, dY, rs, gamma, *run(tb, x, dY, rs, gamma))


def test_zero_rows_write_zero_dgamma(tb):
    D = 64
    x = torch.empty(0, D, device="cuda")
    rs = torch.empty(0, device="cuda")
    dX, dg = run(tb, x, x.clone(), rs, torch.ones(D, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(dg == 0)


def test_deterministic_bitwise(tb, synth):
    args = synth.rmsnorm_inputs(16384, 4096, torch.bfloat16, seed=2, device="cuda", dy_std=1e-2)
    a = run(tb, *args)
    b = run(tb, *args)
    torch.cuda.synchronize()
    for u, w in zip(a, b):
        assert torch.equal(u, w)


def test_workspace_too_small_is_rejected(tb, synth):
    args = synth.rmsnorm_inputs(512, 1024, torch.bfloat16, seed=3, device="cuda")
    need = tb.tb_rmsnorm_bwd_workspace_size(512, 1024, torch.bfloat16)
    with pytest.raises(tb.TbError) as ei:
        run(tb, *args, ws_bytes=16)     # the query may return more than one path needs
    assert ei.value.code == 5
