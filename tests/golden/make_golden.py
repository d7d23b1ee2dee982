"""Writes tests/golden/oracle_small.json from the CPU oracle alone.

The pages print no worked numeric example for these kernels, so the stored
values here are the oracle's own outputs on tiny hand-written inputs, kept to
catch any later change in the oracle's arithmetic (a change must then name the
passage that justifies it).  The inputs are chosen so that a reader can check
the numbers by hand:

* AdamW, three steps of one element per gradient pattern (fp16 gradients,
  loss scale 1024, lr 1e-3, betas 0.9/0.999, eps 1e-8, weight decay 0.01);
* softmax backward on the rows P = [0.25, 0.25, 0.5] and one-hot rows;
* LayerNorm backward on x = [1, 2, 3, 6] with gamma = [1, 2, 0.5, 1].

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def adamw_case():
    theta = np.array([0.5, -0.25, 0.0, 0.125])
    m = np.zeros(4)
    v = np.zeros(4)
    grads = [[1024.0, -512.0, 0.0, 2048.0],   # g = 1, -0.5, 0, 2 after unscaling
             [1024.0, 512.0, 0.0, -2048.0],
             [0.5, -0.5, 1.0, 0.0]]
    steps = []
    for t, g in enumerate(grads, start=1):
        gb = oracle.encode16(np.array(g), "f16")
        copy, gz = oracle.adamw_step_f64(theta, m, v, gb, "f16", 1.0 / 1024.0, t, **HP)
        steps.append({"t": t, "grad_f16_bits": [int(b) for b in gb],
                      "theta": theta.tolist(), "m": m.tolist(), "v": v.tolist(),
                      "copy_bf16_bits": [int(c) for c in copy],
                      "grad_after": [int(z) for z in gz]})
    return {"hparams": HP, "loss_scale": 1024.0, "theta0": [0.5, -0.25, 0.0, 0.125],
            "steps": steps}


def softmax_case():
    P = np.array([[0.25, 0.25, 0.5], [0.0, 1.0, 0.0]])
    dY = np.array([[1.0, -1.0, 2.0], [3.0, -2.0, 5.0]])
    return {"P": P.tolist(), "dY": dY.tolist(), "dX": oracle.softmax_bwd_f64(dY, P).tolist()}


def layernorm_case():
    x = np.array([[1.0, 2.0, 3.0, 6.0], [0.0, -1.0, 1.0, 4.0]])
    dY = np.array([[0.5, -1.0, 2.0, 0.25], [1.0, 1.0, -1.0, 0.0]])
    gamma = np.array([1.0, 2.0, 0.5, 1.0])
    eps = 1e-5
    mu = x.mean(axis=1)
    rs = 1.0 / np.sqrt(((x - mu[:, None]) ** 2).mean(axis=1) + eps)
    dX, dg, db = oracle.layernorm_bwd_f64(dY, x, mu, rs, gamma)
    return {"x": x.tolist(), "dY": dY.tolist(), "gamma": gamma.tolist(), "eps": eps,
            "mean": mu.tolist(), "inv_std": rs.tolist(),
            "dX": dX.tolist(), "dgamma": dg.tolist(), "dbeta": db.tolist()}


if __name__ == "__main__":
    out = {"adamw": adamw_case(), "softmax_bwd": softmax_case(),
           "layernorm_bwd": layernorm_case()}
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", os.path.join(HERE, "oracle_small.json"))
