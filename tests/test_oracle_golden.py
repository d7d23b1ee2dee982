"""The oracle still reproduces its stored small-case outputs (tests/golden).

The fixture was written by tests/golden/make_golden.py, which calls only the
oracle.  Besides guarding against drift, a few entries are checked here against
values worked out by hand from the definitions.
"""
import json
import os

import numpy as np

GOLD = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")


def _load():
    with open(GOLD) as f:
        return json.load(f)


def test_adamw_matches_fixture(orc):
    g = _load()["adamw"]
    theta = np.array(g["theta0"])
    m = np.zeros_like(theta)
    v = np.zeros_like(theta)
    for st in g["steps"]:
        copy, gz = orc.adamw_step_f64(theta, m, v, np.array(st["grad_f16_bits"], np.uint16),
                                      "f16", 1.0 / g["loss_scale"], st["t"], **g["hparams"])
        assert theta.tolist() == st["theta"]
        assert m.tolist() == st["m"] and v.tolist() == st["v"]
        assert [int(c) for c in copy] == st["copy_bf16_bits"]
        assert [int(z) for z in gz] == st["grad_after"] == [0, 0, 0, 0]


def test_adamw_fixture_step1_by_hand():
    """Step 1: theta_1 = theta_0 - lr*sign(g)*|g|/(|g|+eps) - lr*wd*theta_0."""
    g = _load()["adamw"]
    lr, eps, wd = (float(np.float32(g["hparams"][k])) for k in ("lr", "eps", "weight_decay"))
    th0 = np.array(g["theta0"])
    gg = np.array([1.0, -0.5, 0.0, 2.0])
    expect = th0 - lr * gg / (np.abs(gg) + eps) - lr * wd * th0
    np.testing.assert_allclose(g["steps"][0]["theta"], expect, rtol=1e-15)


def test_softmax_fixture_by_hand(orc):
    s = _load()["softmax_bwd"]
    # row 0: dot = 0.25*1 + 0.25*(-1) + 0.5*2 = 1 -> dX = P*(dY-1) = [0, -0.5, 0.5]
    # row 1: one-hot -> dot = -2 -> dX = [0, 0, 0]
    assert s["dX"] == [[0.0, -0.5, 0.5], [0.0, 0.0, 0.0]]
    got = orc.softmax_bwd_f64(np.array(s["dY"]), np.array(s["P"]))
    assert got.tolist() == s["dX"]


def test_layernorm_fixture(orc):
    c = _load()["layernorm_bwd"]
    dX, dg, db = orc.layernorm_bwd_f64(np.array(c["dY"]), np.array(c["x"]),
                                       np.array(c["mean"]), np.array(c["inv_std"]),
                                       np.array(c["gamma"]))
    assert dX.tolist() == c["dX"] and dg.tolist() == c["dgamma"] and db.tolist() == c["dbeta"]
    # dbeta is the column sum of dY, by hand
    assert c["dbeta"] == [1.5, 0.0, 1.0, 0.25]
