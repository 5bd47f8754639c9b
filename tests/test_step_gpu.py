"""Single-token decode steps against the float64 oracle run with L = 1 (the
oracle is the same sequential loop; one step of it is the definition of a
decode step), chained steps against the oracle over the whole sequence, and
in-place state updates.  Metric max|gpu - ref| / max|ref| on the output and
on the state separately: <= 1e-4 with fp32 I/O, <= 1e-2 with bf16 I/O."""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_err
from selective_state_space_chunked_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 1e-2}


@pytest.fixture(scope="module")
def lr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_chunked_gb300 import build
    build.build()
    from selective_state_space_chunked_gb300 import binding
    return binding


def cuda(p):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in p.items()}


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("with_z", [True, False])
def test_selective_step_matches_oracle(lr, io, with_z):
    p = wl.selective_inputs(3, 1, 96, seed=31, io=io, with_h0=True)
    z = p["z"] if with_z else None
    d = cuda(p)
    y, h = lr.selective_scan_step(d["x"][:, 0], d["dt"][:, 0], d["Bm"][:, 0], d["Cm"][:, 0],
                                  d["A_log"], z=None if z is None else d["z"][:, 0],
                                  Dskip=d["Dskip"], h=d["h0"])
    yr, hr = oracle.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=z,
                                   Dskip=p["Dskip"], h0=p["h0"])
    assert rel_err(y.float().cpu()[:, None], yr) <= TOL[io]
    assert rel_err(h.cpu(), hr) <= TOL[io]


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_rglru_step_matches_oracle(lr, io):
    p = wl.rglru_inputs(3, 1, 64, seed=32, io=io, with_h0=True)
    d = cuda(p)
    y, h = lr.rglru_scan_step(d["x"][:, 0], d["r"][:, 0], d["i"][:, 0], d["a_log"], d["c"], h=d["h0"])
    yr, hr = oracle.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    assert rel_err(y.float().cpu()[:, None], yr) <= TOL[io]
    assert rel_err(h.cpu(), hr) <= TOL[io]


@pytest.mark.parametrize("io,dk,dv,H", [("bf16", 128, 128, 2), ("f32", 128, 128, 2),
                                        ("f32", 64, 32, 3), ("bf16", 40, 24, 1)])
def test_hgrn2_step_matches_oracle(lr, io, dk, dv, H):
    g = torch.Generator().manual_seed(33)
    B = 2
    q, k = (torch.randn(B, 1, H * dk, generator=g) / dk ** 0.5 for _ in range(2))
    v = torch.randn(B, 1, H * dv, generator=g) / dv ** 0.5
    gate = 0.2 + 0.8 * torch.sigmoid(torch.randn(B, 1, H * dv, generator=g) + 2)
    S0 = 0.1 * torch.randn(B, H, dv, dk, generator=g)
    dt = torch.float32 if io == "f32" else torch.bfloat16
    q, k, v, gate = (t.to(dt) for t in (q, k, v, gate))
    o, S = lr.hgrn2_step(q[:, 0].cuda(), k[:, 0].cuda(), v[:, 0].cuda(), gate[:, 0].cuda(), H,
                         S=S0.cuda())
    orf, Srf = oracle.hgrn2(q, k, v, gate, H, S0=S0)
    assert rel_err(o.float().cpu()[:, None], orf) <= TOL[io]
    assert rel_err(S.cpu(), Srf) <= TOL[io]


@pytest.mark.parametrize("B,D", [(1, 8), (3, 40)])
def test_selective_step_partial_last_block(lr, B, D):
    """Four lanes per channel: 4*B*D threads that do not fill the last
    128-thread block (the idle lanes still join the readout shuffles), and
    the zero initial state."""
    p = wl.selective_inputs(B, 1, D, seed=36 + D, io="f32", with_h0=False)
    d = cuda(p)
    y, h = lr.selective_scan_step(d["x"][:, 0], d["dt"][:, 0], d["Bm"][:, 0], d["Cm"][:, 0],
                                  d["A_log"], z=d["z"][:, 0], Dskip=d["Dskip"], h=None)
    yr, hr = oracle.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                                   Dskip=p["Dskip"])
    assert rel_err(y.float().cpu()[:, None], yr) <= TOL["f32"]
    assert rel_err(h.cpu(), hr) <= TOL["f32"]


def test_chained_steps_follow_the_sequence_in_place(lr):
    """20 steps with the state updated in place equal the oracle over L = 20."""
    L = 20
    p = wl.selective_inputs(2, L, 64, seed=34, io="f32", with_h0=True)
    d = cuda(p)
    h = d["h0"].clone()
    ys = []
    for t in range(L):
        y, hn = lr.selective_scan_step(d["x"][:, t], d["dt"][:, t], d["Bm"][:, t], d["Cm"][:, t],
                                       d["A_log"], z=d["z"][:, t], Dskip=d["Dskip"], h=h, h_out=h)
        assert hn is h
        ys.append(y)
    yr, hr = oracle.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                                   Dskip=p["Dskip"], h0=p["h0"])
    assert rel_err(torch.stack(ys, 1).cpu(), yr) <= 1e-4
    assert rel_err(h.cpu(), hr) <= 1e-4

    pr = wl.rglru_inputs(2, L, 64, seed=35, io="f32", with_h0=True)
    d = cuda(pr)
    h = d["h0"].clone()
    ys = [lr.rglru_scan_step(d["x"][:, t], d["r"][:, t], d["i"][:, t], d["a_log"], d["c"], h=h,
                             h_out=h)[0] for t in range(L)]
    yr, hr = oracle.rglru_scan(pr["x"], pr["r"], pr["i"], pr["a_log"], pr["c"], h0=pr["h0"])
    assert rel_err(torch.stack(ys, 1).cpu(), yr) <= 1e-4
    assert rel_err(h.cpu(), hr) <= 1e-4

    ph = wl.hgrn2_inputs(1, L, 2, 128, seed=36)
    d = cuda(ph)
    S = torch.zeros(1, 2, 128, 128, device="cuda")
    os_ = [lr.hgrn2_step(d["q"][:, t], d["k"][:, t], d["v"][:, t], d["g"][:, t], 2, S=S, S_out=S)[0]
           for t in range(L)]
    orf, Srf = oracle.hgrn2(ph["q"], ph["k"], ph["v"], ph["g"], 2)
    assert rel_err(torch.stack(os_, 1).float().cpu(), orf) <= 1e-2
    assert rel_err(S.cpu(), Srf) <= 1e-2


def test_step_zero_state_equals_explicit_zeros(lr):
    p = wl.rglru_inputs(2, 1, 64, seed=37, io="bf16")
    d = cuda(p)
    y0, h0 = lr.rglru_scan_step(d["x"][:, 0], d["r"][:, 0], d["i"][:, 0], d["a_log"], d["c"])
    y1, h1 = lr.rglru_scan_step(d["x"][:, 0], d["r"][:, 0], d["i"][:, 0], d["a_log"], d["c"],
                                h=torch.zeros(2, 64, device="cuda"))
    assert torch.equal(y0, y1) and torch.equal(h0, h1)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_minmax_steps_equal_the_scan_bit_for_bit(lr, io):
    """Chained in-place MinMax steps reproduce the oracle's sequence exactly."""
    dt = torch.float32 if io == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(38)
    r = torch.randn(2, 25, 64, generator=g).to(dt)
    s = (torch.randn(2, 25, 64, generator=g) - 1).to(dt)
    x0 = torch.randn(2, 64, generator=g).to(dt).float()
    x = x0.cuda()
    ys = [lr.minmax_scan_step(r[:, t].cuda(), s[:, t].cuda(), x=x, x_out=x)[0] for t in range(25)]
    yr, xr = oracle.minmax_scan(r, s, x0)
    assert np.array_equal(torch.stack(ys, 1).double().cpu().numpy(), yr)
    assert np.array_equal(x.double().cpu().numpy(), xr)


def test_steps_at_the_benchmark_decode_shapes(lr):
    """One step of each form at the shapes the benchmark's decode line times
    (RG-LRU B=8 D=2560, selective B=4 D=4096, HGRN2 B=4 H=16 d=128, bf16),
    from a random carried state, against the oracle's one-step scan."""
    p = wl.rglru_inputs(8, 1, 2560, seed=41, io="bf16", with_h0=True)
    d = cuda(p)
    y, h = lr.rglru_scan_step(d["x"][:, 0], d["r"][:, 0], d["i"][:, 0], d["a_log"], d["c"], h=d["h0"])
    yr, hr = oracle.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    assert rel_err(y.float().cpu()[:, None], yr) <= TOL["bf16"] and rel_err(h.cpu(), hr) <= TOL["bf16"]

    p = wl.selective_inputs(4, 1, 4096, seed=42, io="bf16", with_h0=True)
    d = cuda(p)
    y, h = lr.selective_scan_step(d["x"][:, 0], d["dt"][:, 0], d["Bm"][:, 0], d["Cm"][:, 0], d["A_log"],
                                  z=d["z"][:, 0], Dskip=d["Dskip"], h=d["h0"])
    yr, hr = oracle.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                                   Dskip=p["Dskip"], h0=p["h0"])
    assert rel_err(y.float().cpu()[:, None], yr) <= TOL["bf16"] and rel_err(h.cpu(), hr) <= TOL["bf16"]

    p = wl.hgrn2_inputs(4, 1, 16, 128, seed=43, io="bf16", with_S0=True)
    S0 = 0.1 * p["S0"]
    o, S = lr.hgrn2_step(p["q"][:, 0].cuda(), p["k"][:, 0].cuda(), p["v"][:, 0].cuda(), p["g"][:, 0].cuda(),
                         16, S=S0.cuda())
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], 16, S0=S0)
    assert rel_err(o.float().cpu()[:, None], orf) <= TOL["bf16"] and rel_err(S.cpu(), Srf) <= TOL["bf16"]
