"""The Python binding rejects arguments that the C entry points cannot check
themselves (they receive bare pointers): tensors of the wrong size or dtype for
the sizes the kernels index them by, and tensors that are not on the current
CUDA device.  Every check raises before any pointer reaches libtb, so these
tests run without a GPU.
"""
import pytest
import torch


@pytest.fixture(scope="module")
def tb():
    import __graft_entry__
    __graft_entry__.build()
    import ln_backward_gb300
    return ln_backward_gb300


def _ln_args(rows=4, D=8):
    x = torch.zeros(rows, D)
    return dict(dY=x.clone(), x=x, mean=torch.zeros(rows), inv_std=torch.ones(rows),
                gamma=torch.ones(D), dX=torch.empty_like(x), dgamma=torch.empty(D),
                dbeta=torch.empty(D))


@pytest.mark.parametrize("name, bad", [("mean", torch.zeros(3)), ("inv_std", torch.ones(5)),
                                       ("gamma", torch.ones(7)), ("dgamma", torch.empty(9)),
                                       ("dbeta", torch.empty(4)),
                                       ("mean", torch.zeros(4, dtype=torch.float64))])
def test_layernorm_statistics_and_gamma_sizes(tb, name, bad):
    a = _ln_args()
    a[name] = bad
    with pytest.raises(ValueError, match=name):
        tb.tb_layernorm_bwd(workspace=None, **a)
    with pytest.raises(ValueError, match=name):
        tb.tb_layernorm_bwd_noalloc(**a)


@pytest.mark.parametrize("name, bad", [("inv_rms", torch.ones(3)), ("gamma", torch.ones(9)),
                                       ("dgamma", torch.empty(7, dtype=torch.bfloat16))])
def test_rmsnorm_sizes(tb, name, bad):
    x = torch.zeros(4, 8)
    a = dict(dY=x.clone(), x=x, inv_rms=torch.ones(4), gamma=torch.ones(8), dX=torch.empty_like(x),
             dgamma=torch.empty(8))
    a[name] = bad
    with pytest.raises(ValueError, match=name):
        tb.tb_rmsnorm_bwd(workspace=None, **a)


def test_adamw_plan_sizes_and_dtypes(tb):
    p = [torch.zeros(10), torch.zeros(6)]
    m = [torch.zeros(10), torch.zeros(6)]
    v = [torch.zeros(10), torch.zeros(6)]
    g = [torch.zeros(10, dtype=torch.bfloat16), torch.zeros(6, dtype=torch.bfloat16)]
    c = [torch.zeros(10, dtype=torch.bfloat16), torch.zeros(6, dtype=torch.bfloat16)]
    bad_cases = {
        "m[1]": (p, [m[0], torch.zeros(5)], v, g, c),
        "v[0]": (p, m, [torch.zeros(10, dtype=torch.float16), v[1]], g, c),
        "grads[1]": (p, m, v, [g[0], torch.zeros(6, dtype=torch.float16)], c),   # mixed dtypes
        "grads[0]": (p, m, v, [torch.zeros(11, dtype=torch.bfloat16), g[1]], c),
        "copies[1]": (p, m, v, g, [c[0], torch.zeros(7, dtype=torch.bfloat16)]),
        "params[0]": ([torch.zeros(10, dtype=torch.bfloat16), p[1]], m, v, g, c),
    }
    for name, args in bad_cases.items():
        with pytest.raises(ValueError, match=name.replace("[", r"\[").replace("]", r"\]")):
            tb.tb_adamw_plan_create(*args)
    with pytest.raises(ValueError, match="same dtype"):
        tb.tb_adamw_plan_create(p, m, v, g, [c[0], torch.zeros(6, dtype=torch.float16)])


def test_tensors_must_be_cuda_tensors(tb):
    """Well-formed arguments in host memory: refused before their pointers are used."""
    P = torch.full((4, 8), 0.125)
    with pytest.raises(ValueError, match="CUDA"):
        tb.tb_softmax_bwd(P.clone(), P, torch.empty_like(P))
    with pytest.raises(ValueError, match="CUDA"):
        tb.tb_layernorm_bwd(workspace=None, **_ln_args())
    with pytest.raises(ValueError, match="CUDA"):
        tb.tb_cast_to_f32(torch.zeros(8, dtype=torch.bfloat16), torch.empty(8))
