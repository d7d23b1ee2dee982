"""Stream semantics of the C ABI: calls on different streams run concurrently
without interfering, and the softmax / LayerNorm / RMSNorm calls can be captured
into a CUDA graph and replayed on new data with results bitwise equal to eager
calls (every call is stream-ordered, allocates nothing and does not synchronise).

The softmax, LayerNorm and RMSNorm kernels are launched as programmatic
dependents of the work before them; the stream-order tests below check, with no
synchronisation between the calls, that they still read what the previous kernel
wrote and write nothing that the previous kernel was still reading -- against
torch kernels and against their own earlier calls sharing one workspace.
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


def test_concurrent_cluster_split_calls_match_serial(tb, synth):
    """Two cluster-split LayerNorm calls (16,384 bf16 columns: four-CTA clusters) and
    an RMSNorm call on split fp32 rows, each on its own stream and overlapping on the
    GPU: the clusters of different calls share the SMs, and every result is bitwise
    equal to the serial call's."""
    D, rows = 16384, 1024
    a = synth.layernorm_inputs(rows, D, torch.bfloat16, seed=90, device="cuda", dy_std=1e-2)
    b = synth.layernorm_inputs(rows, D, torch.bfloat16, seed=91, device="cuda", dy_std=1e-2)
    rx, rdY, rinv, rg = synth.rmsnorm_inputs(rows, 12288, torch.float32, seed=92, device="cuda")
    rws_size = tb.tb_rmsnorm_bwd_workspace_size(rows, 12288, torch.float32)

    def rms_bufs():
        return (torch.empty_like(rx), torch.empty(12288, device="cuda"),
                torch.empty(rws_size, dtype=torch.uint8, device="cuda"))

    ref_a, ref_b = _ln_bufs(tb, rows, D, torch.bfloat16), _ln_bufs(tb, rows, D, torch.bfloat16)
    ref_r = rms_bufs()
    tb.tb_layernorm_bwd(a[1], a[0], a[2], a[3], a[4], *ref_a)
    tb.tb_layernorm_bwd(b[1], b[0], b[2], b[3], b[4], *ref_b)
    tb.tb_rmsnorm_bwd(rdY, rx, rinv, rg, *ref_r)
    torch.cuda.synchronize()
    out_a, out_b = _ln_bufs(tb, rows, D, torch.bfloat16), _ln_bufs(tb, rows, D, torch.bfloat16)
    out_r = rms_bufs()
    streams = [torch.cuda.Stream() for _ in range(3)]
    torch.cuda.synchronize()
    for _ in range(5):
        tb.tb_layernorm_bwd(a[1], a[0], a[2], a[3], a[4], *out_a, stream=streams[0])
        tb.tb_layernorm_bwd(b[1], b[0], b[2], b[3], b[4], *out_b, stream=streams[1])
        tb.tb_rmsnorm_bwd(rdY, rx, rinv, rg, *out_r, stream=streams[2])
    torch.cuda.synchronize()
    for got, want in ((out_a, ref_a), (out_b, ref_b), (out_r, ref_r)):
        for u, w in zip(got[:-1], want[:-1]):     # outputs, not the workspaces
            assert torch.equal(u, w)
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


@pytest.mark.parametrize("D, dtype", [(1004, torch.bfloat16), (2048, torch.bfloat16),
                                      (8192, torch.bfloat16), (16384, torch.bfloat16),
                                      (12288, torch.float32)],
                         ids=["fallback-bf16", "ring-bf16", "wide-ring-bf16", "split-bf16",
                              "split-f32"])
def test_norm_row_paths_replay_from_a_graph(tb, synth, D, dtype):
    """LayerNorm and RMSNorm backward on each row path (the register fallback, the
    ring, the 512-thread ring, the cluster-split kernel) captured in a CUDA graph,
    replayed on new data, bitwise equal to eager calls."""
    rows = 300
    x, ldY, mu, rs, g = synth.layernorm_inputs(rows, D, dtype, seed=70 + D, device="cuda")
    ldx, ldg, ldb, lws = _ln_bufs(tb, rows, D, dtype)
    rdx = torch.empty_like(x)
    rdg = torch.empty(D, device="cuda")
    rws = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(rows, D, dtype), dtype=torch.uint8,
                      device="cuda")

    def calls():
        tb.tb_layernorm_bwd(ldY, x, mu, rs, g, ldx, ldg, ldb, lws)
        tb.tb_rmsnorm_bwd(ldY, x, rs, g, rdx, rdg, rws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls()                      # warm-up outside capture (per-device queries are cached)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    x2, ldY2, mu2, rs2, _ = synth.layernorm_inputs(rows, D, dtype, seed=80 + D, device="cuda")
    for dst, src in ((x, x2), (ldY, ldY2), (mu, mu2), (rs, rs2)):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    got = [t.clone() for t in (ldx, ldg, ldb, rdx, rdg)]
    calls()
    torch.cuda.synchronize()
    for a, b in zip(got, (ldx, ldg, ldb, rdx, rdg)):
        assert torch.equal(a, b)
    assert tb.tb_device_error() == 0


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _clone_state(st):
    import copy
    c = copy.copy(st)
    for k in ("theta", "m", "v", "grad", "copy"):
        setattr(c, k, getattr(st, k).clone())
    return c


def _plan(tb, st):
    k = len(st.sizes)
    return tb.tb_adamw_plan_create(*[[st.tensor(a, i) for i in range(k)]
                                     for a in ("theta", "m", "v", "grad", "copy")])


def _close(a, b):
    """fp32 state agreeing to 1e-6 relative (the device forms 1 - beta^t with CUDA's
    pow and the host with the C library's; both round to fp32, so they differ at
    most in a rare last bit of the bias correction)."""
    return torch.allclose(a, b, rtol=1e-6, atol=1e-12)


def test_device_step_counter_matches_host_steps(tb, synth):
    a = synth.make_adamw_state(synth.gpt2_small_shapes()[:12], seed=61, device="cuda")
    b = _clone_state(a)
    pa, pb = _plan(tb, a), _plan(tb, b)
    step = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in range(1, 6):
        synth.fill_grads(a, t)
        b.grad.copy_(a.grad)
        tb.tb_adamw_step(pa, t, inv_loss_scale=1 / 65536.0, **HP)
        step.add_(1)
        tb.tb_adamw_step_device(pb, step, inv_loss_scale=1 / 65536.0, **HP)
    torch.cuda.synchronize()
    for k in ("theta", "m", "v"):
        assert _close(getattr(a, k), getattr(b, k)), k
    assert torch.equal(b.grad, torch.zeros_like(b.grad))
    assert tb.tb_device_error() == 0
    pa.close()
    pb.close()


def test_whole_optimizer_step_replayed_from_a_cuda_graph(tb, synth):
    """Counter increment, gradient norm and clipped update captured once and replayed
    for three steps, against the same three steps called eagerly with host steps."""
    shapes = synth.gpt2_small_shapes()[:12]
    a = synth.make_adamw_state(shapes, seed=62, device="cuda")
    b = _clone_state(a)
    pa, pb = _plan(tb, a), _plan(tb, b)
    max_norm = 0.05
    grads = []
    for t in range(1, 4):
        synth.fill_grads(a, t)
        grads.append(a.grad.clone())
    # eager reference on a, host step counter
    clip_a = torch.zeros(3, device="cuda")
    ws_a = torch.empty(tb.tb_adamw_grad_norm_workspace_size(pa), dtype=torch.uint8, device="cuda")
    for t in range(1, 4):
        a.grad.copy_(grads[t - 1])
        tb.tb_adamw_grad_norm(pa, 1 / 65536.0, max_norm, clip_a, ws_a)
        tb.tb_adamw_step_clipped(pa, t, inv_loss_scale=1 / 65536.0, clip=clip_a, **HP)
    # graph on b: everything per step lives on the device
    step = torch.zeros(1, dtype=torch.int64, device="cuda")
    clip_b = torch.zeros(3, device="cuda")
    ws_b = torch.empty(tb.tb_adamw_grad_norm_workspace_size(pb), dtype=torch.uint8, device="cuda")

    def one_step():
        step.add_(1)
        tb.tb_adamw_grad_norm(pb, 1 / 65536.0, max_norm, clip_b, ws_b)
        tb.tb_adamw_step_device(pb, step, inv_loss_scale=1 / 65536.0, clip=clip_b, **HP)

    # warm up on a throw-away copy of the state so that b itself starts untouched
    w = _clone_state(b)
    pw = _plan(tb, w)
    ws_w = torch.empty_like(ws_b)
    tb.tb_adamw_grad_norm(pw, 1 / 65536.0, max_norm, clip_b, ws_w)
    tb.tb_adamw_step_device(pw, torch.ones(1, dtype=torch.int64, device="cuda"),
                            inv_loss_scale=1 / 65536.0, clip=clip_b, **HP)
    torch.cuda.synchronize()
    pw.close()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        one_step()
    for t in range(1, 4):
        b.grad.copy_(grads[t - 1])
        graph.replay()
    torch.cuda.synchronize()
    assert step.item() == 3
    assert _close(clip_a, clip_b)
    for k in ("theta", "m", "v"):
        assert _close(getattr(a, k), getattr(b, k)), k
    assert tb.tb_device_error() == 0
    pa.close()
    pb.close()


def test_device_step_below_one_updates_nothing(tb, synth):
    st = synth.make_adamw_state([("a", (4096,))], seed=63, device="cuda")
    plan = _plan(tb, st)
    before = st.theta.clone()
    tb.tb_adamw_step_device(plan, torch.zeros(1, dtype=torch.int64, device="cuda"),
                            inv_loss_scale=1.0, **HP)
    torch.cuda.synchronize()
    assert torch.equal(st.theta, before)
    assert tb.tb_device_error(reset=True) == 1        # TB_ERR_INVALID_VALUE
    assert tb.tb_device_error(reset=True) == 0
    plan.close()


def test_programmatic_launch_keeps_stream_order_softmax(tb, synth):
    rows, cols = 8192, 1024
    P1, dY1 = synth.softmax_inputs(rows, cols, torch.bfloat16, seed=51, device="cuda")
    P2, dY2 = synth.softmax_inputs(rows, cols, torch.bfloat16, seed=52, device="cuda")
    ref1, ref2 = torch.empty_like(P1), torch.empty_like(P1)
    tb.tb_softmax_bwd(dY1, P1, ref1)
    tb.tb_softmax_bwd(dY2, P2, ref2)
    torch.cuda.synchronize()
    assert not torch.equal(ref1, ref2)
    P, dY, dX = P1.clone(), dY1.clone(), torch.empty_like(P1)
    snaps = []
    for _ in range(4):
        tb.tb_softmax_bwd(dY, P, dX)
        snaps.append(dX.clone())          # a torch kernel reads dX ...
        P.copy_(P2)                       # ... and torch kernels rewrite the inputs
        dY.copy_(dY2)
        tb.tb_softmax_bwd(dY, P, dX)      # must read the new inputs, and write dX only
        snaps.append(dX.clone())          # after the clone above has read it
        P.copy_(P1)
        dY.copy_(dY1)
    torch.cuda.synchronize()
    for i, snap in enumerate(snaps):
        assert torch.equal(snap, ref1 if i % 2 == 0 else ref2), i


@pytest.mark.parametrize("op", ["layernorm", "rmsnorm"])
def test_programmatic_launch_keeps_stream_order_norms(tb, synth, op):
    """Back-to-back calls on different inputs share one workspace: a call's row kernel
    must not overwrite the column partials before the previous call's column reduction
    has read them, and must read inputs a torch kernel has just rewritten."""
    rows, D = 4096, 4096
    if op == "layernorm":
        a = synth.layernorm_inputs(rows, D, torch.bfloat16, seed=53, device="cuda", dy_std=1e-2)
        b = synth.layernorm_inputs(rows, D, torch.bfloat16, seed=54, device="cuda", dy_std=1e-2)
        ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, torch.bfloat16),
                         dtype=torch.uint8, device="cuda")

        def call(inp, outs):
            x, dY, mu, rs, g = inp
            tb.tb_layernorm_bwd(dY, x, mu, rs, g, *outs, ws)

        def outs_new():
            return (torch.empty(rows, D, dtype=torch.bfloat16, device="cuda"),
                    torch.empty(D, device="cuda"), torch.empty(D, device="cuda"))
    else:
        a = synth.rmsnorm_inputs(rows, D, torch.bfloat16, seed=55, device="cuda", dy_std=1e-2)
        b = synth.rmsnorm_inputs(rows, D, torch.bfloat16, seed=56, device="cuda", dy_std=1e-2)
        ws = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(rows, D, torch.bfloat16),
                         dtype=torch.uint8, device="cuda")

        def call(inp, outs):
            x, dY, inv, g = inp
            tb.tb_rmsnorm_bwd(dY, x, inv, g, *outs, ws)

        def outs_new():
            return (torch.empty(rows, D, dtype=torch.bfloat16, device="cuda"),
                    torch.empty(D, device="cuda"))
    ref_a, ref_b = outs_new(), outs_new()
    call(a, ref_a)
    torch.cuda.synchronize()
    call(b, ref_b)
    torch.cuda.synchronize()
    assert not torch.equal(ref_a[1], ref_b[1])
    # alternate the two problems with no synchronisation: each call's own outputs, and
    # one input tensor set that torch kernels rewrite between the calls
    own = [(outs_new(), outs_new()) for _ in range(3)]
    shared = [(outs_new(), outs_new()) for _ in range(3)]
    cur = tuple(t.clone() for t in a)
    torch.cuda.synchronize()
    for oa, ob in own:
        call(a, oa)
        call(b, ob)
    for oa, ob in shared:
        call(cur, oa)
        for t, src in zip(cur, b):
            t.copy_(src)
        call(cur, ob)
        for t, src in zip(cur, a):
            t.copy_(src)
    torch.cuda.synchronize()
    for oa, ob in own + shared:
        for u, w in zip(oa, ref_a):
            assert torch.equal(u, w)
        for u, w in zip(ob, ref_b):
            assert torch.equal(u, w)
    assert tb.tb_device_error(reset=True) == 0
