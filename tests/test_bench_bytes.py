"""The algorithmic byte counts behind the benchmark's GB/s, checked on CPU.

Every count is recomputed here by walking the buffers a kernel reads and writes
once each (pure Python on small shapes), so a wrong factor in bench.py's
formulas -- and with it every reported bandwidth -- shows up here.
"""
import bench


def test_adamw_bytes_per_parameter():
    # per parameter: read grad (bf16) + theta, m, v (fp32); write theta, m, v, copy (bf16), grad
    reads = 2 + 4 + 4 + 4
    writes = 4 + 4 + 4 + 2 + 2
    for n in (1, 7, 124_439_808, 6_738_415_616):
        assert bench.adamw_bytes(n) == (reads + writes) * n


def test_softmax_bytes():
    for rows, cols, es in ((3, 5, 4), (98_304, 1_024, 2)):
        assert bench.softmax_bytes(rows, cols, es) == (2 + 1) * rows * cols * es


def test_layernorm_and_rmsnorm_bytes():
    for rows, D, es in ((3, 8, 4), (16_384, 4_096, 2)):
        elems = rows * D * es
        ln = 2 * elems + elems + rows * (4 + 4) + D * (4 + 4 + 4)      # x, dY; dX; mean, inv_std; gamma, dgamma, dbeta
        rms = 2 * elems + elems + rows * 4 + D * (4 + 4)                # x, dY; dX; inv_rms; gamma, dgamma
        assert bench.layernorm_bytes(rows, D, es) == ln
        assert bench.rmsnorm_bytes(rows, D, es) == rms


def test_causal_softmax_bytes_brute_force():
    for rows, cols, period, offset, es in ((40, 13, 10, 0, 4), (64, 64, 16, 3, 2), (30, 24, 7, 50, 2),
                                           (2_048, 1_024, 1_024, 0, 4)):
        per_vec = 16 // es
        total = 0
        for r in range(rows):
            open_cols = min(cols, r % period + 1 + offset)
            vectors = -(-open_cols // per_vec)
            total += 2 * vectors * 16                  # the vectors of P and dY holding an open column
            total += cols * es                         # all of dX
        assert bench.causal_softmax_bytes(rows, cols, period, offset, es) == total


def test_full_step_bytes():
    n = 6_738_415_616
    rows, cols = 98_304, 1_024
    expect = (bench.adamw_bytes(n) + bench.softmax_bytes(rows, cols, 4) + bench.softmax_bytes(rows, cols, 2)
              + bench.layernorm_bytes(16_384, 4_096, 2))
    assert bench.FULL_STEP_BYTES == expect == 204_367_241_216
