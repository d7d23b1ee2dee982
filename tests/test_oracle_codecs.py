"""Pins for the oracle's 16-bit float codecs.

The codecs are written from the binary16 / bfloat16 bit layouts; they are pinned
by brute force over every 16-bit pattern against library conversions (numpy's
float16 and torch's bfloat16), and by hand-picked rounding ties.
"""
import numpy as np
import pytest
import torch


ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_decode_bf16_all_patterns(orc):
    got = orc.decode16(ALL, "bf16")
    ref = torch.from_numpy(ALL.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_decode_f16_all_patterns(orc):
    got = orc.decode16(ALL, "f16")
    ref = ALL.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_encode_roundtrips_every_pattern(orc):
    for kind in ("bf16", "f16"):
        vals = orc.decode16(ALL, kind)
        ok = ~np.isnan(vals)
        back = orc.encode16(vals[ok], kind)
        assert np.array_equal(back, ALL[ok]), kind


def _random_floats(n, seed):
    rng = np.random.default_rng(seed)
    # mixture of magnitudes: normal range, tiny (subnormal for bf16/f16), huge (overflow)
    exps = rng.integers(-140, 130, n)
    mant = rng.random(n) + 0.5
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    with np.errstate(over="ignore"):    # the huge ones overflow to +-inf on purpose
        return (sign * np.ldexp(mant, exps)).astype(np.float32)


def test_encode_bf16_matches_torch_rne(orc):
    x = _random_floats(200_000, 1)
    got = orc.encode16(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_encode_f16_matches_numpy_rne(orc):
    rng = np.random.default_rng(2)
    x = np.concatenate([_random_floats(100_000, 3).astype(np.float64) * 1e-4,
                        rng.standard_normal(100_000) * 3e4,
                        rng.standard_normal(100_000)])
    got = orc.encode16(x, "f16")
    with np.errstate(over="ignore"):    # values beyond fp16's range round to +-inf
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("x, bits", [
    (1.0 + 2.0 ** -8, 0x3F80),          # tie between 1 and 1+2^-7 -> even (1.0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),      # tie between 1+2^-7 and 1+2^-6 -> even (1+2^-6)
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),  # just above the tie -> up
    (-0.0, 0x8000),
    (2.0 ** 127 * (2 - 2.0 ** -7), 0x7F7F),  # largest finite bf16
    (2.0 ** 127 * (2 - 2.0 ** -8), 0x7F80),  # halfway to 2^128: tie -> even = inf
    (2.0 ** -133, 0x0001),              # smallest bf16 subnormal
    (2.0 ** -134, 0x0000),              # half of it: tie -> even (zero)
])
def test_encode_bf16_ties_and_edges(orc, x, bits):
    assert int(orc.encode16(np.array([x]), "bf16")[0]) == bits
