"""Guard regions around every output: no entry point writes outside its buffers.

Each output (and each workspace) is carved out of a larger byte buffer whose
margins are filled with a fixed byte pattern; after the call the margins must
still hold it.  Shapes are ragged on purpose (row lengths that are not a
multiple of a vector, row counts that are not a multiple of a CTA's rows,
tensors whose sizes are not a multiple of the 8-element unit) and some outputs
start one element past a 16-byte boundary, so every tail loop and every scalar
path runs next to a margin.  The values themselves are checked by the parity
tests; here only the margins are.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

PAD = 4096          # bytes of margin on each side
PATTERN = 0xA5


@pytest.fixture(scope="module")
def tb():
    import ln_backward_gb300
    return ln_backward_gb300


@pytest.fixture(scope="module")
def synth():
    from ln_backward_gb300 import synth
    return synth


class Guarded:
    """A tensor of `shape`/`dtype` that starts `shift` bytes past a 16-byte
    boundary inside a byte buffer with PAD-byte margins of PATTERN."""

    def __init__(self, shape, dtype, shift=0, fill=None):
        es = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        self.lo = PAD + shift
        self.nbytes = n * es
        self.buf = torch.full((self.lo + self.nbytes + PAD,), PATTERN, dtype=torch.uint8,
                              device="cuda")
        self.t = self.buf.narrow(0, self.lo, self.nbytes).view(dtype).view(*shape)
        if fill is not None:
            self.t.copy_(fill)

    def margins_intact(self):
        torch.cuda.synchronize()
        head = self.buf[:self.lo]
        tail = self.buf[self.lo + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


SOFTMAX_SHAPES = [(333, 1000, torch.float32, 0), (77, 2050, torch.bfloat16, 0),
                  (1000, 128, torch.float16, 2), (9, 20000, torch.float32, 4),
                  (513, 8, torch.bfloat16, 0), (3, 33000, torch.bfloat16, 0),
                  (100, 3000, torch.float32, 0)]


@pytest.mark.parametrize("rows, cols, dtype, shift", SOFTMAX_SHAPES)
def test_softmax_bwd_stays_in_bounds(tb, synth, rows, cols, dtype, shift):
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=11, device="cuda")
    dX = Guarded((rows, cols), dtype, shift)
    tb.tb_softmax_bwd(dY, P, dX.t)
    assert dX.margins_intact()
    dXc = Guarded((rows, cols), dtype, shift)
    tb.tb_softmax_bwd_causal(dY, P, dXc.t, period=max(1, cols // 3), offset=1)
    assert dXc.margins_intact()


LN_SHAPES = [(1000, 768, torch.bfloat16, 0), (333, 4096, torch.float32, 0),
             (50, 8192, torch.float16, 0), (37, 10000, torch.bfloat16, 0),
             (129, 1000, torch.float32, 4), (65, 264, torch.bfloat16, 2), (1, 8, torch.float32, 0)]


@pytest.mark.parametrize("rows, D, dtype, shift", LN_SHAPES)
def test_layernorm_bwd_stays_in_bounds(tb, synth, rows, D, dtype, shift):
    x, dY, mean, rstd, gamma = synth.layernorm_inputs(rows, D, dtype, seed=12, device="cuda")
    need = tb.tb_layernorm_bwd_workspace_size(rows, D, dtype)
    dX = Guarded((rows, D), dtype, shift)
    dg = Guarded((D,), torch.float32, 4 if shift else 0)
    db = Guarded((D,), torch.float32)
    ws = Guarded((need,), torch.uint8)
    tb.tb_layernorm_bwd(dY, x, mean, rstd, gamma, dX.t, dg.t, db.t, ws.t)
    for g in (dX, dg, db, ws):
        assert g.margins_intact()
    # the entry point without a workspace
    dX2, dg2, db2 = Guarded((rows, D), dtype, shift), Guarded((D,), torch.float32), \
        Guarded((D,), torch.float32)
    tb.tb_layernorm_bwd_noalloc(dY, x, mean, rstd, gamma, dX2.t, dg2.t, db2.t)
    for g in (dX2, dg2, db2):
        assert g.margins_intact()


@pytest.mark.parametrize("rows, D, dtype, shift", LN_SHAPES)
def test_rmsnorm_bwd_stays_in_bounds(tb, synth, rows, D, dtype, shift):
    x, dY, inv, gamma = synth.rmsnorm_inputs(rows, D, dtype, seed=13, device="cuda")
    need = tb.tb_rmsnorm_bwd_workspace_size(rows, D, dtype)
    dX = Guarded((rows, D), dtype, shift)
    dg = Guarded((D,), torch.float32)
    ws = Guarded((need,), torch.uint8)
    tb.tb_rmsnorm_bwd(dY, x, inv, gamma, dX.t, dg.t, ws.t)
    for g in (dX, dg, ws):
        assert g.margins_intact()


@pytest.mark.parametrize("src_dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n, shift", [(1, 0), (8191, 0), (100_003, 4), (65_536, 0)])
def test_casts_stay_in_bounds(tb, src_dtype, n, shift):
    src = (torch.randn(n, device="cuda") * 100).to(src_dtype)
    dst = Guarded((n,), torch.float32, shift)
    tb.tb_cast_to_f32(src, dst.t, scale=0.5)
    assert dst.margins_intact()
    if src_dtype != torch.float32:
        back = Guarded((n,), src_dtype, shift // 2)
        tb.tb_cast_from_f32(dst.t, back.t)
        assert back.margins_intact()


SENT32 = 0x7FA5A5A5          # a NaN payload no kernel produces
SENT16 = 0x7DA5              # an fp16 NaN payload (a huge finite bf16); not produced here
ADAMW_SIZES = [1, 7, 8, 9, 1000, 8193, 65_541, 3, 300_007]
GAP = 37                     # elements between tensors (so most tensors start misaligned)


def _arena(total, dtype, sentinel):
    itype = torch.int32 if dtype == torch.float32 else torch.int16
    return torch.full((total,), sentinel, dtype=itype, device="cuda").view(dtype)


@pytest.mark.parametrize("grad_dtype, with_copy", [(torch.bfloat16, True), (torch.float16, True),
                                                   (torch.float32, False)])
def test_adamw_touches_only_its_tensors(tb, grad_dtype, with_copy):
    offs, o = [], GAP
    for n in ADAMW_SIZES:
        offs.append(o)
        o += n + GAP
    total = o
    theta = _arena(total, torch.float32, SENT32)
    m = _arena(total, torch.float32, SENT32)
    v = _arena(total, torch.float32, SENT32)
    grad = _arena(total, grad_dtype, SENT32 if grad_dtype == torch.float32 else SENT16)
    copy = _arena(total, torch.bfloat16, SENT16)
    gen = torch.Generator(device="cuda").manual_seed(21)
    for off, n in zip(offs, ADAMW_SIZES):
        theta[off:off + n] = torch.randn(n, device="cuda", generator=gen) * 0.02
        m[off:off + n] = 0
        v[off:off + n] = 0
        copy[off:off + n] = 0
    live = torch.zeros(total, dtype=torch.bool, device="cuda")
    for off, n in zip(offs, ADAMW_SIZES):
        live[off:off + n] = True
    before = {k: t.clone() for k, t in (("theta", theta), ("m", m), ("v", v), ("grad", grad),
                                        ("copy", copy))}

    def views(t):
        return [t.narrow(0, off, n) for off, n in zip(offs, ADAMW_SIZES)]

    plan = tb.tb_adamw_plan_create(views(theta), views(m), views(v), views(grad),
                                   views(copy) if with_copy else [None] * len(offs))
    clip = torch.zeros(3, device="cuda")
    ws = torch.empty(tb.tb_adamw_grad_norm_workspace_size(plan), dtype=torch.uint8, device="cuda")
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    for t in (1, 2):
        for off, n in zip(offs, ADAMW_SIZES):
            grad[off:off + n] = (torch.randn(n, device="cuda", generator=gen) * 65.536).to(grad_dtype)
        tb.tb_adamw_step(plan, t, inv_loss_scale=1 / 65536.0, **hp)
    for off, n in zip(offs, ADAMW_SIZES):
        grad[off:off + n] = (torch.randn(n, device="cuda", generator=gen) * 65.536).to(grad_dtype)
    tb.tb_adamw_grad_norm(plan, 1 / 65536.0, 1.0, clip, ws)
    tb.tb_adamw_step_clipped(plan, 3, inv_loss_scale=1 / 65536.0, clip=clip, **hp)
    torch.cuda.synchronize()
    plan.close()
    for k, t in (("theta", theta), ("m", m), ("v", v), ("grad", grad), ("copy", copy)):
        itype = torch.int32 if t.element_size() == 4 else torch.int16
        gap_now = t.view(itype)[~live]
        gap_before = before[k].view(itype)[~live]
        assert torch.equal(gap_now, gap_before), f"{k}: a gap between tensors was written"
    # and the live elements did change where they must
    assert not torch.equal(theta.view(torch.int32)[live], before["theta"].view(torch.int32)[live])
    # the same steps on the same values packed without gaps give the same results, so
    # no read of a gap (filled with NaN payloads) reached a result
    n_live = int(live.sum())
    packed = {k: before[k][live].clone() for k in before}
    poffs, o = [], 0
    for n in ADAMW_SIZES:
        poffs.append(o)
        o += n

    def pviews(t):
        return [t.narrow(0, off, n) for off, n in zip(poffs, ADAMW_SIZES)]

    gen = torch.Generator(device="cuda").manual_seed(21)
    for off, n in zip(offs, ADAMW_SIZES):             # replay the generator draws of the state
        torch.randn(n, device="cuda", generator=gen)
    plan = tb.tb_adamw_plan_create(pviews(packed["theta"]), pviews(packed["m"]), pviews(packed["v"]),
                                   pviews(packed["grad"]),
                                   pviews(packed["copy"]) if with_copy else [None] * len(offs))
    clip2 = torch.zeros(3, device="cuda")
    ws2 = torch.empty(tb.tb_adamw_grad_norm_workspace_size(plan), dtype=torch.uint8, device="cuda")
    for t in (1, 2):
        parts = [(torch.randn(n, device="cuda", generator=gen) * 65.536).to(grad_dtype) for n in ADAMW_SIZES]
        packed["grad"].copy_(torch.cat(parts))
        tb.tb_adamw_step(plan, t, inv_loss_scale=1 / 65536.0, **hp)
    parts = [(torch.randn(n, device="cuda", generator=gen) * 65.536).to(grad_dtype) for n in ADAMW_SIZES]
    packed["grad"].copy_(torch.cat(parts))
    tb.tb_adamw_grad_norm(plan, 1 / 65536.0, 1.0, clip2, ws2)
    tb.tb_adamw_step_clipped(plan, 3, inv_loss_scale=1 / 65536.0, clip=clip2, **hp)
    torch.cuda.synchronize()
    plan.close()
    assert packed["theta"].numel() == n_live
    for k, t in (("theta", theta), ("m", m), ("v", v), ("grad", grad), ("copy", copy)):
        itype = torch.int32 if t.element_size() == 4 else torch.int16
        assert torch.equal(t.view(itype)[live], packed[k].view(itype)), f"{k}: differs from the packed run"


def test_grad_norm_outputs_stay_in_bounds(tb, synth):
    st = synth.make_adamw_state([("a", (1001,)), ("b", (64, 65))], seed=14, device="cuda")
    k = len(st.sizes)
    plan = tb.tb_adamw_plan_create(*[[st.tensor(a, i) for i in range(k)]
                                     for a in ("theta", "m", "v", "grad", "copy")])
    need = tb.tb_adamw_grad_norm_workspace_size(plan)
    out = Guarded((3,), torch.float32)
    ws = Guarded((need,), torch.uint8)
    tb.tb_adamw_grad_norm(plan, 1 / 65536.0, 1.0, out.t, ws.t)
    assert out.margins_intact() and ws.margins_intact()
    plan.close()


# ----------------------------------------------------------------------------- input guards
# Each input is placed twice at the same offset from a 16-byte boundary: once between
# margins of 0xFF bytes (a NaN in fp32, bf16 and fp16) and once between finite margins
# (0xA5 bytes).  Both runs take the same code path, so a read past an input's end or
# before its start that reached a result would make the two differ; every result must
# be equal bit for bit.
POISON = 0xFF


class Poisoned(Guarded):
    def __init__(self, values, shift=0, poison=True):
        super().__init__(tuple(values.shape), values.dtype, shift)
        if poison:
            self.buf.fill_(POISON)
        self.t.copy_(values)


def _both(values, shift=0):
    """The same values between finite margins and between NaN margins."""
    return Poisoned(values, shift, poison=False).t, Poisoned(values, shift).t


@pytest.mark.parametrize("rows, cols, dtype, shift", SOFTMAX_SHAPES)
def test_softmax_reads_only_its_inputs(tb, synth, rows, cols, dtype, shift):
    P, dY = synth.softmax_inputs(rows, cols, dtype, seed=15, device="cuda")
    (fP, gP), (fdY, gdY) = _both(P, shift), _both(dY, shift)
    ref, out = torch.empty_like(P), torch.empty_like(P)
    tb.tb_softmax_bwd(fdY, fP, ref)
    tb.tb_softmax_bwd(gdY, gP, out)
    refc, outc = torch.empty_like(P), torch.empty_like(P)
    tb.tb_softmax_bwd_causal(fdY, fP, refc, period=max(1, cols // 3), offset=1)
    tb.tb_softmax_bwd_causal(gdY, gP, outc, period=max(1, cols // 3), offset=1)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(outc, refc)


@pytest.mark.parametrize("rows, D, dtype, shift", LN_SHAPES)
def test_layernorm_and_rmsnorm_read_only_their_inputs(tb, synth, rows, D, dtype, shift):
    x, dY, mean, rstd, gamma = synth.layernorm_inputs(rows, D, dtype, seed=16, device="cuda")
    pairs = [_both(dY, shift), _both(x, shift), _both(mean), _both(rstd), _both(gamma)]
    outs = []
    for side in (0, 1):
        dX, dg, db = torch.empty_like(x), torch.empty(D, device="cuda"), torch.empty(D, device="cuda")
        ws = torch.empty(tb.tb_layernorm_bwd_workspace_size(rows, D, dtype), dtype=torch.uint8,
                         device="cuda")
        tb.tb_layernorm_bwd(*[p[side] for p in pairs], dX, dg, db, ws)
        outs.append((dX, dg, db))
    xr, dYr, inv, gr = synth.rmsnorm_inputs(rows, D, dtype, seed=17, device="cuda")
    pairs = [_both(dYr, shift), _both(xr, shift), _both(inv), _both(gr)]
    for side in (0, 1):
        dX, dg = torch.empty_like(xr), torch.empty(D, device="cuda")
        ws = torch.empty(tb.tb_rmsnorm_bwd_workspace_size(rows, D, dtype), dtype=torch.uint8,
                         device="cuda")
        tb.tb_rmsnorm_bwd(*[p[side] for p in pairs], dX, dg, ws)
        outs.append((dX, dg))
    torch.cuda.synchronize()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    for a, b in zip(outs[2], outs[3]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("src_dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n, shift", [(1, 0), (8191, 0), (100_003, 4)])
def test_casts_read_only_their_inputs(tb, src_dtype, n, shift):
    src = (torch.randn(n, device="cuda") * 100).to(src_dtype)
    sh = shift if src_dtype == torch.float32 else shift // 2
    fs, gs = _both(src, sh)
    ref, out = torch.empty(n, device="cuda"), torch.empty(n, device="cuda")
    tb.tb_cast_to_f32(fs, ref, scale=0.5)
    tb.tb_cast_to_f32(gs, out, scale=0.5)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    if src_dtype != torch.float32:
        fr, gr = _both(ref, shift)
        r16, o16 = torch.empty(n, dtype=src_dtype, device="cuda"), torch.empty(n, dtype=src_dtype, device="cuda")
        tb.tb_cast_from_f32(fr, r16)
        tb.tb_cast_from_f32(gr, o16)
        torch.cuda.synchronize()
        assert torch.equal(o16.view(torch.int16), r16.view(torch.int16))
