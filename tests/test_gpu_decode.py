"""GPU parity of the decode step (m3_step) against the fp64 oracle, through
the C ABI: the fast kernel's shapes (P in {32, 64, 128}, N a multiple of 8,
R in {1, 2, 4}) with fp32 and bf16 inputs, missing optional inputs, the
generic kernel on element-aligned inputs, and the full decode workload (b256 h32
P64 N64) over consecutive steps checked on sampled (batch, head) units."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, max_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def run_chain(m3, shape, seed, steps, with_prev=True, with_lam=True, with_theta=True, sel=None):
    inp = inputs.make_decode_inputs(shape, seed)
    d = {k: v.cuda() for k, v in inp.items()}
    state = d["state0"].clone()
    ys = []
    for s in range(steps):
        y = torch.empty_like(d["x"][s + 1])
        m3.m3_step(state, d["x"][s + 1], d["dt"][s + 1], d["A"], d["B"][s + 1], d["C"][s + 1],
                   d["lam"][s + 1] if with_lam else None, d["theta"][s + 1] if with_theta else None,
                   d["B"][s] if with_prev else None, d["x"][s] if with_prev else None, y)
        ys.append(y)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    yg = torch.stack(ys, 1).float().cpu()          # [b, steps, h, R, P]
    st = state.cpu()
    tok = lambda a: a[1:steps + 1].transpose(0, 1)  # [steps, b, ...] -> [b, steps, ...]
    args = dict(x=tok(inp["x"]), dt=tok(inp["dt"]), A=inp["A"], B=tok(inp["B"]), C=tok(inp["C"]),
                lam=tok(inp["lam"]) if with_lam else None, theta=tok(inp["theta"]) if with_theta else None,
                h0=inp["state0"], prevB=inp["B"][0] if with_prev else None,
                prevx=inp["x"][0] if with_prev else None)
    if sel is not None:
        bsel, hsel = sel
        pick = lambda a, hax: None if a is None else a[bsel][:, hsel] if hax == 1 else a[bsel][:, :, hsel]
        args = dict(x=pick(args["x"], 2), dt=pick(args["dt"], 2), A=args["A"][hsel], B=pick(args["B"], 2),
                    C=pick(args["C"], 2), lam=pick(args["lam"], 2), theta=pick(args["theta"], 2),
                    h0=pick(args["h0"], 1), prevB=pick(args["prevB"], 1), prevx=pick(args["prevx"], 1))
        yg = yg[bsel][:, :, hsel]
        st = st[bsel][:, hsel]
    if with_prev:
        yr, fr = oracle.scan(args["x"], args["dt"], args["A"], args["B"], args["C"], args["lam"], args["theta"],
                             h0=args["h0"], prevB=args["prevB"], prevx=args["prevx"])
    else:
        # every call was given no previous token: no beta term at any step, so
        # the reference is a chain of single oracle steps without a carry
        fr, ys_r = args["h0"], []
        for t in range(steps):
            at = lambda a: None if a is None else a[:, t]
            yt, fr = oracle.step(fr, at(args["x"]), at(args["dt"]), args["A"], at(args["B"]), at(args["C"]),
                                 at(args["lam"]), at(args["theta"]))
            ys_r.append(yt)
        yr = np.stack(ys_r, 1)
    return max_rel(yg, yr), max_rel(st, fr)


FAST = [(32, 8), (64, 64), (128, 16), (64, 32), (32, 64)]   # (P, N)


@pytest.mark.parametrize("P,N", FAST, ids=lambda v: str(v))
@pytest.mark.parametrize("R", [1, 2, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fast_step_shapes(m3, P, N, R, dtype):
    shape = inputs.DecodeShape(batch=3, heads=5, headdim=P, dstate=N, rank=R, steps=6, dtype=dtype)
    ey, es = run_chain(m3, shape, 100 + P + N + R, 6)
    assert ey <= TOL[dtype] and es <= TOL[dtype], (ey, es)


# 8192 (b, h) units, several waves of CTAs for every fast shape; sampled units
# are checked against the oracle.
@pytest.mark.parametrize("P,N", [pn for pn in FAST if (pn[0] // 4) * (pn[1] // 8) >= 32], ids=lambda v: str(v))
@pytest.mark.parametrize("R", [1, 2, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fast_step_many_units(m3, P, N, R, dtype):
    shape = inputs.DecodeShape(batch=256, heads=32, headdim=P, dstate=N, rank=R, steps=3, dtype=dtype)
    ey, es = run_chain(m3, shape, 200 + P + N + R, 3, sel=([0, 131, 255], [0, 13, 31]))
    assert ey <= TOL[dtype] and es <= TOL[dtype], (ey, es)


def test_fast_step_many_units_optional_inputs(m3):
    shape = inputs.DecodeShape(batch=256, heads=32, headdim=64, dstate=64, rank=2, steps=3, dtype="f32")
    ey, es = run_chain(m3, shape, 9, 3, with_prev=False, with_lam=False, with_theta=False,
                       sel=([1, 254], [2, 30]))
    assert ey <= 1e-4 and es <= 1e-4, (ey, es)


@pytest.mark.parametrize("prev,lam,theta", [(False, True, True), (True, False, True), (True, True, False),
                                            (False, False, False)])
def test_fast_step_optional_inputs(m3, prev, lam, theta):
    shape = inputs.DecodeShape(batch=2, heads=3, headdim=64, dstate=64, rank=2, steps=4, dtype="f32")
    ey, es = run_chain(m3, shape, 7, 4, with_prev=prev, with_lam=lam, with_theta=theta)
    assert ey <= 1e-4 and es <= 1e-4, (ey, es)


def test_unaligned_inputs_take_generic_kernel(m3):
    """Inputs that are only element-aligned (not 16-byte) still step correctly
    (the generic kernel); a state that is not 16-byte aligned is rejected."""
    shape = inputs.DecodeShape(batch=2, heads=2, headdim=64, dstate=64, rank=1, steps=1, dtype="f32")
    inp = inputs.make_decode_inputs(shape, 3)
    d = {k: v.cuda() for k, v in inp.items()}
    xbuf = torch.empty(d["x"][1].numel() + 1, device="cuda")
    x1 = xbuf[1:].view_as(d["x"][1])
    x1.copy_(d["x"][1])
    state = d["state0"].clone()
    y = torch.empty_like(d["x"][1])
    m3.m3_step(state, x1, d["dt"][1], d["A"], d["B"][1], d["C"][1], d["lam"][1], d["theta"][1],
               d["B"][0], d["x"][0], y)
    torch.cuda.synchronize()
    yr, fr = oracle.step(inp["state0"], inp["x"][1], inp["dt"][1], inp["A"], inp["B"][1], inp["C"][1],
                         inp["lam"][1], inp["theta"][1], inp["B"][0], inp["x"][0])
    assert max_rel(y.cpu(), yr) <= 1e-4 and max_rel(state.cpu(), fr) <= 1e-4
    sbuf = torch.empty(d["state0"].numel() + 1, device="cuda")
    bad_state = sbuf[1:].view_as(d["state0"])
    with pytest.raises(m3.M3Error) as e:
        m3.m3_step(bad_state, d["x"][1], d["dt"][1], d["A"], d["B"][1], d["C"][1], d["lam"][1], d["theta"][1],
                   d["B"][0], d["x"][0], y)
    assert e.value.status == m3.M3_ERR_ALIGN


@pytest.mark.parametrize("R", [1, 4])
def test_decode_workload_full_size(m3, R):
    """The decode workload (b256 h32 P64 N64, fp32 state and inputs) at full
    size, the launch the bench times, over 16 consecutive steps; checked on
    sampled (batch, head) units."""
    shape = inputs.DecodeShape(**{**inputs.WORKLOADS[inputs.DECODE].__dict__, "rank": R, "steps": 16})
    ey, es = run_chain(m3, shape, 4, 16, sel=([0, 100, 255], [0, 17, 31]))
    assert ey <= 1e-4 and es <= 1e-4, (ey, es)


@pytest.mark.parametrize("R", [1, 4])
def test_decode_sweep_1024_steps_in_graph(m3, R):
    """The decode sweep the bench times: b256 h32 P64 N64 fp32, 1024 consecutive
    m3_step calls captured in one CUDA graph.  y and the state are checked
    against the oracle after every 64th step and at step 1024, on 12 sampled
    (batch, head) units; the oracle runs the same 1024 tokens in 64-token
    segments, each started from its own previous segment's final state."""
    steps, seg = 1024, 64
    shape = inputs.DecodeShape(**{**inputs.WORKLOADS[inputs.DECODE].__dict__, "rank": R, "steps": steps})
    inp = inputs.make_decode_inputs(shape, 4 + R, device="cuda")
    bsel, hsel = [0, 37, 128, 255], [0, 11, 31]
    state = inp["state0"].clone()
    ys = torch.empty_like(inp["x"][1:])
    snaps = torch.empty((steps // seg,) + tuple(state.shape), device="cuda")
    dims = m3.step_dims(inp["x"][0], inp["B"][0])
    stream = torch.cuda.Stream()

    def sweep():
        for s in range(steps):
            m3.m3_step(state, inp["x"][s + 1], inp["dt"][s + 1], inp["A"], inp["B"][s + 1], inp["C"][s + 1],
                       inp["lam"][s + 1], inp["theta"][s + 1], inp["B"][s], inp["x"][s], ys[s], stream=stream,
                       dims=dims)
            if (s + 1) % seg == 0:
                snaps[(s + 1) // seg - 1].copy_(state)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        sweep()                                         # uncaptured warm-up, as the bench does
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sweep()
    state.copy_(inp["state0"])
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK

    sel = lambda a: a[:, bsel][:, :, hsel].cpu()        # [S, b, h, ...] -> sampled units
    x, dt, B, C, lam, th = (sel(inp[k]) for k in ("x", "dt", "B", "C", "lam", "theta"))
    A = inp["A"][hsel].cpu()
    h = inp["state0"][bsel][:, hsel].cpu()
    yg = ys[:, bsel][:, :, hsel].cpu()                  # [steps, b', h', R, P]
    sg = snaps[:, bsel][:, :, hsel].cpu()
    worst = (0.0, 0.0)
    for k in range(steps // seg):
        t0, t1 = k * seg + 1, (k + 1) * seg + 1         # tokens of this segment
        tok = lambda a: a[t0:t1].transpose(0, 1)
        yr, h = oracle.scan(tok(x), tok(dt), A, tok(B), tok(C), tok(lam), tok(th), h0=h,
                            prevB=B[t0 - 1], prevx=x[t0 - 1])
        ey = max_rel(yg[t0 - 1:t1 - 1].transpose(0, 1), yr)
        es = max_rel(sg[k], h)
        worst = (max(worst[0], ey), max(worst[1], es))
        assert ey <= 1e-4 and es <= 1e-4, (k, ey, es)
    print(f"R{R} 1024 steps: worst segment y {worst[0]:.2e} state {worst[1]:.2e}")


@pytest.mark.parametrize("R,dtype", [(4, "f32"), (1, "bf16")])
def test_decode_step_every_unit(m3, R, dtype):
    """One decode step of b256 h32 P64 N64 checked on every (batch, head) unit:
    the persistent kernel walks many units per CTA, so an indexing mistake would
    show on some units only."""
    shape = inputs.DecodeShape(batch=256, heads=32, headdim=64, dstate=64, rank=R, steps=2, dtype=dtype)
    ey, es = run_chain(m3, shape, 300 + R, 2)
    assert ey <= TOL[dtype] and es <= TOL[dtype], (ey, es)
