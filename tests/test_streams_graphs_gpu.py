"""Stream semantics of the C ABI: calls on different streams run concurrently
without interfering, and the softmax / LayerNorm / RMSNorm calls can be captured
into a CUDA graph and replayed on new data with results bitwise equal to eager
calls (every call is stream-ordered, allocates nothing and does not synchronise).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


def _ln_bufs(tb, rows, D, dtype):
    ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, dtype), dtype=torch.uint8,
                     device="cuda")
    return (torch.empty(rows, D, dtype=dtype, device="cuda"), torch.empty(D, device="cuda"),
            torch.empty(D, device="cuda"), ws)


def test_concurrent_streams_match_serial(tb, synth):
    P, dY = synth.softmax_inputs(8192, 1024, torch.bfloat16, seed=41, device="cuda")
    x, ldY, mu, rs, g = synth.layernorm_inputs(4096, 4096, torch.bfloat16, seed=42, device="cuda")
    # serial reference
    ref_sm = torch.empty_like(P)
    tb.tb_softmax_bwd(dY, P, ref_sm)
    rdx, rdg, rdb, rws = _ln_bufs(tb, 4096, 4096, torch.bfloat16)
    tb.tb_layernorm_bwd(ldY, x, mu, rs, g, rdx, rdg, rdb, rws)
    torch.cuda.synchronize()
    # the same two calls, each on its own stream, several times over
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    out_sm = torch.empty_like(P)
    dx, dg, db, ws = _ln_bufs(tb, 4096, 4096, torch.bfloat16)
    torch.cuda.synchronize()
    for _ in range(5):
        tb.tb_softmax_bwd(dY, P, out_sm, stream=s1)
        tb.tb_layernorm_bwd(ldY, x, mu, rs, g, dx, dg, db, ws, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(out_sm, ref_sm)
    assert torch.equal(dx, rdx) and torch.equal(dg, rdg) and torch.equal(db, rdb)
    assert tb.tb_device_error() == 0


def test_cuda_graph_capture_and_replay(tb, synth):
    rows_sm, rows_ln, D = 4096, 2048, 4096
    P, dY = synth.softmax_inputs(rows_sm, 1024, torch.float32, seed=43, device="cuda")
    x, ldY, mu, rs, g = synth.layernorm_inputs(rows_ln, D, torch.bfloat16, seed=44, device="cuda")
    rx, rdY, rinv, rg = synth.rmsnorm_inputs(rows_ln, D, torch.bfloat16, seed=45, device="cuda")
    dX = torch.empty_like(P)
    ldx, ldg, ldb, lws = _ln_bufs(tb, rows_ln, D, torch.bfloat16)
    rdx = torch.empty_like(rx)
    rdg = torch.empty(D, device="cuda")
    rws = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(rows_ln, D, torch.bfloat16), dtype=torch.uint8,
                      device="cuda")

    def calls(stream=None):
        tb.tb_softmax_bwd(dY, P, dX, stream=stream)
        tb.tb_layernorm_bwd(ldY, x, mu, rs, g, ldx, ldg, ldb, lws, stream=stream)
        tb.tb_rmsnorm_bwd(rdY, rx, rinv, rg, rdx, rdg, rws, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls()                      # warm-up outside capture (per-device queries are cached)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()

    # new input data in the same buffers, then replay
    P2, dY2 = synth.softmax_inputs(rows_sm, 1024, torch.float32, seed=53, device="cuda")
    P.copy_(P2)
    dY.copy_(dY2)
    x2, ldY2, mu2, rs2, _ = synth.layernorm_inputs(rows_ln, D, torch.bfloat16, seed=54, device="cuda")
    for dst, src in ((x, x2), (ldY, ldY2), (mu, mu2), (rs, rs2)):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    got = [t.clone() for t in (dX, ldx, ldg, ldb, rdx, rdg)]
    calls()                          # eager on the same data
    torch.cuda.synchronize()
    want = (dX, ldx, ldg, ldb, rdx, rdg)
    for a, b in zip(got, want):
        assert torch.equal(a, b)
    assert tb.tb_device_error() == 0
