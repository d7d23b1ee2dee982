"""Pins for the oracle's stand-alone casts (the training loop's unscale and copy-back casts).

Both casts have a plain definition that library routines implement exactly:
fp16/bf16 -> fp32 times a scale is one fp32 rounding of an exact product
(torch's own fp32 multiply on the widened values), fp32 -> 16-bit is round to
nearest even (torch's conversion).
"""
import numpy as np
import torch


def _values(n, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n) * np.exp(rng.uniform(-20, 20, n))).astype(np.float32)


def test_cast_to_f32_matches_torch_bitwise(orc):
    for kind, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        bits = orc.encode16(_values(100_000, 1).astype(np.float64), kind)
        t = torch.from_numpy(bits.view(np.int16).copy()).view(tdt)
        for scale in (1.0, 1 / 1024.0, 1 / 65536.0, 0.3):
            ref = (t.float() * torch.tensor(scale, dtype=torch.float32)).numpy()
            got = orc.cast_to_f32(bits, kind, scale)
            nan = np.isnan(ref)
            assert np.array_equal(np.isnan(got), nan)
            assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    x = _values(10_000, 2)
    np.testing.assert_array_equal(orc.cast_to_f32(x, "f32", 0.5), x * np.float32(0.5))


def test_cast_from_f32_matches_torch_rne(orc):
    x = _values(200_000, 3)
    for kind, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        ref = torch.from_numpy(x).to(tdt).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(orc.cast_from_f32(x, kind), ref)
