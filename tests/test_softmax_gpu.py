"""GPU parity of the softmax backward against the CPU oracle.

Targets: fp32 dX within 1e-5 absolute of the float64 oracle; 16-bit dX within
one 16-bit ulp of the oracle's exact result rounded to nearest even (or, for
outputs that cancel far below their terms, within the fp32 arithmetic's own
error bound -- see tests/tolerance.py).  Covers the tiny config (1024 x 128
fp32, every element), the attention config (98,304 x 1,024 causal, fp32 and
bf16, every element), a sweep of row lengths across every kernel path with a
ragged row count, unaligned buffers (two-pass path) and empty inputs, and the
causal variant (reads only the open columns) on the attention config and on
shapes that exercise every path with row offsets and wrap-around periods,
including the folded pairs (rows q and period-1-q of a causal block on one warp
or one CTA) on every instance the host can pick, with odd periods, partial last
blocks and large offsets.
"""
import numpy as np
import pytest
import torch

import oracle
from tolerance import lowp_check, to_bits

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


def _err_bound(P, dY):
    """Bound on |dX_fp32 - dX_exact| for the kernel's fp32 arithmetic: the dot
    product (at most cols/32 + 16 rounded additions on any path, each below
    2^-24 of sum|P*dY|), the subtraction and the final multiply."""
    cols = P.shape[1]
    S = np.sum(np.abs(P * dY), axis=1, keepdims=True)
    dot = np.sum(P * dY, axis=1, keepdims=True)
    k = cols / 32 + 64
    return np.abs(P) * (k * 2.0 ** -24 * S + 2.0 ** -22 * (np.abs(dY) + np.abs(dot)))


def check(dX, P, dY):
    """Compares the GPU result with the float64 oracle on the same inputs."""
    Pn = P.double().cpu().numpy()
    dYn = dY.double().cpu().numpy()
    ref = oracle.softmax_bwd_f64(dYn, Pn)
    if dX.dtype == torch.float32:
        err = np.max(np.abs(dX.double().cpu().numpy() - ref)) if ref.size else 0.0
        assert err <= 1e-5, f"max abs error {err}"
    else:
        ok, n_err, dmax = lowp_check(to_bits(dX), ref, KIND[dX.dtype], _err_bound(Pn, dYn))
        assert ok.all(), f"{(~ok).sum()} elements off (max ulp distance {dmax})"


def test_tiny_config_fp32(tb, synth):
    P, dY = synth.softmax_inputs(1024, 128, torch.float32, seed=0, device="cuda")
    dX = torch.empty_like(P)
    tb.tb_softmax_bwd(dY, P, dX)
    check(dX, P, dY)


COLS = [1, 2, 3, 4, 5, 8, 16, 31, 33, 64, 127, 128, 255, 256, 1000, 1023, 1024, 1025, 2048,
        2049, 2056, 3072, 4096, 6144, 8192, 8200, 16384, 16392, 20000]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16],
                         ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("cols", COLS)
def test_row_length_sweep(tb, synth, cols, dtype):
    P, dY = synth.softmax_inputs(37, cols, dtype, seed=cols, device="cuda")
    dX = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd(dY, P, dX)
    check(dX, P, dY)


# Shapes with more row groups than a persistent grid has CTAs (152 SMs x 3), in both grid
# regimes: one CTA per row group when a CTA carries at least 40 KB of traffic, else the
# persistent grid striding over the groups.
@pytest.mark.parametrize("rows, cols, dtype, period", [
    (4000, 1024, torch.float32, 0),        # warp per row, 96 KB per CTA: one CTA per group
    (4000, 128, torch.float32, 0),         # warp per row, 12 KB per CTA: persistent
    (4000, 512, torch.bfloat16, 512),      # causal, about 16 KB per CTA: persistent
    (4000, 1024, torch.float32, 1024),     # causal, about 66 KB per CTA: one CTA per group
    (2000, 4096, torch.float32, 0),        # CTA per row, 48 KB: one CTA per row
    (2000, 2048, torch.float32, 0),        # CTA per row, 24 KB: persistent
    (2000, 4096, torch.bfloat16, 4096),    # CTA per row, causal, about 16 KB: persistent
], ids=["group-oneshot", "group-persistent", "causal-bf16-persistent", "causal-f32-oneshot",
        "cta-oneshot", "cta-persistent", "cta-causal-persistent"])
def test_both_grid_regimes(tb, synth, rows, cols, dtype, period):
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=rows + cols, device="cuda",
                                 causal_period=period or None)
    dX = torch.full_like(P, float("nan"))
    if period:
        tb.tb_softmax_bwd_causal(dY, P, dX, period=period)
    else:
        tb.tb_softmax_bwd(dY, P, dX)
    check(dX, P, dY)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_unaligned_buffers_take_two_pass_path(tb, synth, dtype):
    rows, cols = 19, 1024
    P0, dY0 = synth.softmax_inputs(rows, cols, dtype, seed=9, device="cuda")
    bufP = torch.empty(rows * cols + 1, dtype=dtype, device="cuda")
    bufY = torch.empty(rows * cols + 1, dtype=dtype, device="cuda")
    bufX = torch.empty(rows * cols + 1, dtype=dtype, device="cuda")
    P = bufP[1:].view(rows, cols)
    dY = bufY[1:].view(rows, cols)
    dX = bufX[1:].view(rows, cols)
    P.copy_(P0)
    dY.copy_(dY0)
    tb.tb_softmax_bwd(dY, P, dX)
    check(dX, P, dY)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_attention_config_full_size(tb, synth, dtype):
    """B=8, H=12, S=1024: 98,304 rows x 1,024 causal columns; every element compared."""
    rows, cols = 8 * 12 * 1024, 1024
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=2, device="cuda", causal_period=1024)
    # the causal structure: row r sees columns j <= r mod 1024, masked entries exactly 0
    assert torch.all(P[5, 6:] == 0) and torch.all(P[5, :6] > 0)
    dX = torch.empty_like(P)
    tb.tb_softmax_bwd(dY, P, dX)
    torch.cuda.synchronize()
    for r0 in range(0, rows, 16384):
        check(dX[r0:r0 + 16384], P[r0:r0 + 16384], dY[r0:r0 + 16384])
    # masked positions give exactly zero
    assert torch.all(dX[5, 6:] == 0)


def test_empty_inputs_are_noops(tb):
    for shape in ((0, 16), (16, 0), (0, 0)):
        P = torch.empty(shape, device="cuda")
        tb.tb_softmax_bwd(P, P.clone(), P.clone())


def test_aliasing_rejected(tb, synth):
    P, dY = synth.softmax_inputs(8, 64, torch.float32, seed=3, device="cuda")
    with pytest.raises(tb.TbError):
        tb.tb_softmax_bwd(dY, P, dY)


def test_deterministic(tb, synth):
    P, dY = synth.softmax_inputs(4096, 1024, torch.bfloat16, seed=4, device="cuda")
    a, b = torch.empty_like(P), torch.empty_like(P)
    tb.tb_softmax_bwd(dY, P, a)
    tb.tb_softmax_bwd(dY, P, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ----------------------------------------------------------------------------- causal variant
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_causal_variant_attention_config(tb, synth, dtype):
    """tb_softmax_bwd_causal on the 98,304 x 1,024 causal block stack: same values as the
    oracle (and as the dense kernel), every element."""
    rows, cols = 8 * 12 * 1024, 1024
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=5, device="cuda", causal_period=1024)
    dX = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd_causal(dY, P, dX, period=1024)
    dense = torch.empty_like(P)
    tb.tb_softmax_bwd(dY, P, dense)
    torch.cuda.synchronize()
    assert torch.equal(dX, dense)          # +0 == -0 under torch.equal's value comparison
    for r0 in range(0, rows, 24576):
        check(dX[r0:r0 + 24576], P[r0:r0 + 24576], dY[r0:r0 + 24576])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16],
                         ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("rows, cols, period, offset", [
    (300, 128, 128, 0), (300, 1024, 256, 768), (77, 1000, 1000, 0), (64, 33, 33, 0),
    (129, 4096, 4096, 0), (50, 20000, 20000, 0), (40, 2048, 16, 5), (10, 512, 4, 600)])
def test_causal_variant_shapes(tb, synth, rows, cols, period, offset, dtype):
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=rows + cols, device="cuda",
                                 causal_period=period, causal_offset=offset)
    dX = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd_causal(dY, P, dX, period=period, offset=offset)
    check(dX, P, dY)


# Folded pairs (16-bit causal rows of 65..256 vectors with period <= rows: rows q and
# period-1-q of a block on one warp).  Odd periods (a middle row without a partner),
# partial last blocks, period 1, period == rows, periods longer than the row, offsets,
# both grid regimes, more pairs than a persistent grid holds, every slot count (4, 6
# and 10 vectors a lane) and both sum orders; and shapes beside them (shorter rows,
# pairs that would need more slots) that stay on the one-row kernel.
PAIRS = [(2500, 1024, 1024, 0), (2049, 1024, 1023, 3), (1000, 768, 333, 0), (640, 1024, 640, 0),
         (600, 520, 1, 7), (20000, 1024, 256, 0), (20000, 528, 528, 0), (1100, 1016, 1016, 5),
         (2100, 2048, 2048, 0), (3000, 2048, 1024, 0), (1500, 2048, 1500, 0), (2100, 1040, 1040, 0),
         (4100, 2048, 2048, 9), (3000, 1536, 1536, 0),
         (777, 256, 256, 0), (1000, 512, 333, 0), (1500, 1024, 1500, 0), (300, 1024, 256, 768),
         (300, 2048, 256, 1800)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("rows, cols, period, offset", PAIRS)
def test_causal_folded_pairs(tb, synth, rows, cols, period, offset, dtype):
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=7 * rows + period, device="cuda",
                                 causal_period=period, causal_offset=offset)
    dX = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd_causal(dY, P, dX, period=period, offset=offset)
    # vectors of 8 columns that hold no open column are written as +0
    r = torch.arange(rows, device="cuda")[:, None] % period
    c = torch.arange(cols, device="cuda")[None, :]
    closed = (c // 8) * 8 >= r + 1 + offset
    assert torch.all(dX.view(torch.int16)[closed] == 0)
    check(dX, P, dY)
    # each row summed in the dense kernel's order (its extra terms are exact zeros)
    dense = torch.empty_like(P)
    tb.tb_softmax_bwd(dY, P, dense)
    torch.cuda.synchronize()
    assert torch.equal(dX, dense)


# Folded pairs on the CTA path (causal rows of 257..2048 vectors: 16-bit rows of 2,056..16,384
# columns, fp32 of 1,028..8,192; rows q and period-1-q of a block on one CTA of 128, 256 or
# 512 threads).  Every instance that can be chosen (128 threads with 2, 4 or 6 slots a
# thread, 256 with 4, 6, 8 or 10, 512 with 6), full blocks plus partial ones, odd periods
# with offsets, periods shorter than the row, row lengths that are not a multiple of the CTA,
# and period 1.  CTAs of fewer than 512 threads group each row's sum differently from the
# dense kernel, so the check is the oracle's, plus bitwise repeatability.
CTA_PAIRS = [(4500, 4096, 4096, 0), (4500, 6144, 4095, 3), (3000, 8192, 2048, 0),
             (2100, 4104, 2000, 7), (600, 4112, 1, 0), (3000, 2560, 2560, 0),
             (5700, 6144, 5600, 0), (2053, 8192, 2048, 3100), (1030, 12288, 1024, 5000),
             (1027, 16384, 1024, 7700), (1027, 16384, 1024, 9000)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16],
                         ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("rows, cols, period, offset", CTA_PAIRS)
def test_causal_folded_pairs_cta(tb, synth, rows, cols, period, offset, dtype):
    if cols * torch.tensor([], dtype=dtype).element_size() > 2048 * 16:
        pytest.skip("rows of more than 2048 vectors take the two-pass kernel")
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=3 * rows + period, device="cuda",
                                 causal_period=period, causal_offset=offset)
    dX = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd_causal(dY, P, dX, period=period, offset=offset)
    E = 16 // P.element_size()
    r = torch.arange(rows, device="cuda")[:, None] % period
    c = torch.arange(cols, device="cuda")[None, :]
    closed = (c // E) * E >= r + 1 + offset
    itype = torch.int32 if dtype == torch.float32 else torch.int16
    assert torch.all(dX.view(itype)[closed] == 0)
    again = torch.full_like(P, float("nan"))
    tb.tb_softmax_bwd_causal(dY, P, again, period=period, offset=offset)
    torch.cuda.synchronize()
    assert torch.equal(dX.view(itype), again.view(itype))
    step = max(1, (1 << 23) // cols)
    for r0 in range(0, rows, step):
        check(dX[r0:r0 + step], P[r0:r0 + step], dY[r0:r0 + step])


def test_causal_variant_rejects_bad_period(tb, synth):
    P, dY = synth.softmax_inputs(8, 64, torch.float32, seed=3, device="cuda")
    with pytest.raises(tb.TbError):
        tb.tb_softmax_bwd_causal(dY, P, torch.empty_like(P), period=0)


def test_causal_variant_huge_offset_opens_every_column(tb, synth):
    """An offset far beyond cols (up to the int64 limit) leaves no column masked: the
    result is the dense one, bit for bit."""
    P, dY = synth.softmax_inputs(100, 1000, torch.float32, seed=7, device="cuda")
    dense = torch.empty_like(P)
    tb.tb_softmax_bwd(dY, P, dense)
    for offset in (1000, 2**40, 2**63 - 1):
        dX = torch.full_like(P, float("nan"))
        tb.tb_softmax_bwd_causal(dY, P, dX, period=2**62, offset=offset)
        torch.cuda.synchronize()
        assert torch.equal(dX, dense), offset
