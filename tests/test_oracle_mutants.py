"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake (a dropped term, a
wrong sign, a wrong operand), compiles the copy on the CPU and runs the pins of
the affected method through it.  At least one pin has to fail for every mutant.
"""
import numpy as np
import pytest

import test_oracle_adamw as A
import test_oracle_cast as CA
import test_oracle_gradclip as GC
import test_oracle_layernorm as L
import test_oracle_rmsnorm as RN
import test_oracle_softmax as S

ADAMW_PINS = [A.test_step1_closed_form, A.test_constant_gradient_no_decay,
              A.test_zero_gradient_is_pure_decay, A.test_matches_torch_adamw_float64]
SOFTMAX_PINS = [S.test_one_hot_rows_give_exact_zero, S.test_uniform_rows_give_centered_dy,
                S.test_rows_sum_to_zero, S.test_central_finite_differences,
                S.test_matches_torch_autograd_float64]
LN_PINS = [L.test_dbeta_is_column_sum, L.test_dgamma_is_column_sum_of_dy_xhat, L.test_rows_of_dx_sum_to_zero,
           L.test_dx_orthogonal_to_xhat_when_eps_zero, L.test_d_equals_one_is_degenerate,
           L.test_central_finite_differences, L.test_matches_torch_autograd_float64]

RMS_PINS = [RN.test_dgamma_is_column_sum_of_dy_xhat, RN.test_dx_orthogonal_to_xhat_when_eps_zero,
            RN.test_central_finite_differences, RN.test_matches_torch_rms_norm_autograd_float64]

CLIP_PINS = [GC.test_norm_matches_numpy_over_several_tensors, GC.test_norm_special_cases,
             GC.test_clip_factor_closed_forms, GC.test_clipped_step_matches_torch_clip_then_adamw,
             GC.test_skip_leaves_state_and_zeroes_gradient]

CAST_PINS = [CA.test_cast_to_f32_matches_torch_bitwise, CA.test_cast_from_f32_matches_torch_rne]

MUTANTS = [
    ("cast: scale ignored", "out[i] = (float)(x * (double)scale);", "out[i] = (float)x;", CAST_PINS),
    ("cast: product rounded twice through half",
     "out[i] = (float)(x * (double)scale);", "out[i] = (float)(float)x * scale * 1.0000001f;", CAST_PINS),
    ("gradclip: norm misses the loss-scale removal",
     "        g *= inv_loss_scale;\n        s += g * g;", "        s += g * g;", CLIP_PINS),
    ("gradclip: clip factor inverted",
     "return max_norm / norm;", "return norm / max_norm;", CLIP_PINS),
    ("gradclip: clipping on norm >= max_norm only when below",
     "if (max_norm > 0.0 && norm > max_norm)", "if (max_norm > 0.0 && norm < max_norm)", CLIP_PINS),
    ("gradclip: clip not applied in the step",
     "* inv_loss_scale * clip;", "* inv_loss_scale;", CLIP_PINS),
    ("gradclip: non-finite gradient not flagged",
     "if (!isfinite(g)) *nonfinite = 1;", "", CLIP_PINS),
    ("rmsnorm: projection term dropped",
     "dxr[j] = rs * (dxhat - xhat * mean_dxhat_xhat);", "dxr[j] = rs * dxhat;", RMS_PINS),
    ("rmsnorm: projection term sign flipped",
     "dxr[j] = rs * (dxhat - xhat * mean_dxhat_xhat);",
     "dxr[j] = rs * (dxhat + xhat * mean_dxhat_xhat);", RMS_PINS),
    ("rmsnorm: gamma not applied",
     "sum_dxhat_xhat += (dyr[j] * gamma[j]) * (xr[j] * rs);",
     "sum_dxhat_xhat += dyr[j] * (xr[j] * rs);", RMS_PINS),
    ("adamw: decay added instead of subtracted",
     "- lr * wd * th;", "+ lr * wd * th;", ADAMW_PINS),
    ("adamw: first-moment bias correction dropped",
     "double m_hat = m[i] / bc1;", "double m_hat = m[i];", ADAMW_PINS),
    ("adamw: eps inside the square root",
     "(sqrt(v_hat) + eps)", "sqrt(v_hat + eps)", ADAMW_PINS),
    ("adamw: second moment takes g instead of g^2",
     "(1.0 - b2) * (g * g);", "(1.0 - b2) * g;", ADAMW_PINS),
    ("adamw: decay on the updated theta",
     "- lr * wd * th;", "- lr * wd * (th - lr * m_hat / (sqrt(v_hat) + eps));", ADAMW_PINS),
    ("adamw: second-moment bias correction dropped",
     "double v_hat = v[i] / bc2;", "double v_hat = v[i];", ADAMW_PINS),
    ("adamw: working copy rounded from the pre-update theta",
     "copy[i] = orc_encode16_rne(theta[i], copy_kind);", "copy[i] = orc_encode16_rne(th, copy_kind);",
     ADAMW_PINS),
    ("adamw: loss scale not removed",
     "* inv_loss_scale;\n        /* first", ";\n        /* first", ADAMW_PINS),
    ("softmax: dot added instead of subtracted",
     "dx[j] = p[j] * (dy[j] - dot);", "dx[j] = p[j] * (dy[j] + dot);", SOFTMAX_PINS),
    ("softmax: dot of dY with itself",
     "for (int64_t j = 0; j < cols; ++j) dot += p[j] * dy[j];\n        for (int64_t j = 0; j < cols; ++j) dx[j] = p[j] * (dy[j] - dot);\n    }\n}\n\nvoid orc_softmax_bwd_f32",
     "for (int64_t j = 0; j < cols; ++j) dot += dy[j] * dy[j];\n        for (int64_t j = 0; j < cols; ++j) dx[j] = p[j] * (dy[j] - dot);\n    }\n}\n\nvoid orc_softmax_bwd_f32",
     SOFTMAX_PINS),
    ("softmax: every row reads the first row of P",
     "const double* p = P + r * cols;", "const double* p = P;", SOFTMAX_PINS),
    ("softmax: P factor dropped",
     "dx[j] = p[j] * (dy[j] - dot);", "dx[j] = (dy[j] - dot);", SOFTMAX_PINS),
    ("layernorm: mean of dxhat dropped",
     "dxr[j] = rs * (dxhat - mean_dxhat - xhat * mean_dxhat_xhat);\n            dgamma[j] += dyr[j] * xhat;\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     "dxr[j] = rs * (dxhat - xhat * mean_dxhat_xhat);\n            dgamma[j] += dyr[j] * xhat;\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     LN_PINS),
    ("layernorm: xhat term sign flipped",
     "dxr[j] = rs * (dxhat - mean_dxhat - xhat * mean_dxhat_xhat);\n            dgamma[j] += dyr[j] * xhat;\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     "dxr[j] = rs * (dxhat - mean_dxhat + xhat * mean_dxhat_xhat);\n            dgamma[j] += dyr[j] * xhat;\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     LN_PINS),
    ("layernorm: gamma not applied to dY",
     "double dxhat = dyr[j] * gamma[j];\n            sum_dxhat += dxhat;",
     "double dxhat = dyr[j];\n            sum_dxhat += dxhat;", LN_PINS),
    ("layernorm: dbeta accumulates dxhat",
     "dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     "dbeta[j] += dxhat;\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32", LN_PINS),
    ("layernorm: dgamma from the raw x instead of xhat",
     "dgamma[j] += dyr[j] * xhat;\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     "dgamma[j] += dyr[j] * xr[j];\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     LN_PINS),
    ("layernorm: projection sum takes dY instead of dxhat",
     "sum_dxhat_xhat += dxhat * xhat;", "sum_dxhat_xhat += dyr[j] * xhat;", LN_PINS),
    ("layernorm: inv_std factor dropped from dX",
     "dxr[j] = rs * (dxhat - mean_dxhat - xhat * mean_dxhat_xhat);\n            dgamma[j] += dyr[j] * xhat;\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     "dxr[j] = (dxhat - mean_dxhat - xhat * mean_dxhat_xhat);\n            dgamma[j] += dyr[j] * xhat;\n            dbeta[j] += dyr[j];\n        }\n    }\n}\n\nvoid orc_layernorm_bwd_f32",
     LN_PINS),
]


@pytest.mark.parametrize("desc, old, new, pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_kill_mutant(orc, tmp_path, desc, old, new, pins):
    src = open(orc.source_path()).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {desc}"
    mutated = src.replace(old, new, 1)
    so = orc.compile_variant(mutated, str(tmp_path), "mutant")
    failures = 0
    with orc.swapped_library(so):
        for pin in pins:
            args = {"orc": orc}
            try:
                if pin is A.test_step1_closed_form:
                    pin(orc, "f16", 1024.0)
                else:
                    pin(**args)
            except AssertionError:
                failures += 1
    assert failures >= 1, f"no pin caught: {desc}"
