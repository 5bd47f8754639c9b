"""Scans whose gates arrive before their activation ([RGLRU] forward's
sigmoid on r and i, [HGRN2] g = lb + (1 - lb) sigmoid(f)): the kernel applies
the activation; the oracle gets the activated gates computed in float64 from
the same input bits.  Tolerances as for the plain scans."""
import pytest
import torch

import oracle
from conftest import rel_err
from selective_state_space_chunked_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 1e-2}
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def lr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_chunked_gb300 import build
    build.build()
    from selective_state_space_chunked_gb300 import binding
    return binding


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("B,L,D", [(2, 300, 128), (1, 77, 64)])
def test_rglru_preact_matches_oracle(lr, io, B, L, D):
    g = torch.Generator().manual_seed(B * 100 + L)
    x, r_pre, i_pre = (torch.randn(B, L, D, generator=g).to(DT[io]) for _ in range(3))
    a = 0.9 + 0.099 * torch.rand(D, generator=g)
    a_log = torch.log(a)
    h0 = torch.randn(B, D, generator=g)
    y, hf = lr.rglru_scan(x.cuda(), r_pre.cuda(), i_pre.cuda(), a_log.cuda(), 8.0, h0=h0.cuda(),
                          gates_preact=True)
    yr, hr = oracle.rglru_scan(x, torch.sigmoid(r_pre.double()), torch.sigmoid(i_pre.double()),
                               a_log, 8.0, h0=h0)
    assert rel_err(y.float().cpu(), yr) <= TOL[io]
    assert rel_err(hf.cpu(), hr) <= TOL[io]


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_rglru_preact_with_time_splits(lr, io):
    """L = 900 leaves a ragged last tile (4 rows of a 64-step bf16 tile, 4 of
    a 32-step f32 tile); the aggregate pass must treat the padded rows as
    identity steps although sigmoid(0) = 1/2."""
    g = torch.Generator().manual_seed(3)
    x, r_pre, i_pre = (torch.randn(1, 900, 64, generator=g).to(DT[io]) for _ in range(3))
    a_log = torch.log(0.9 + 0.099 * torch.rand(64, generator=g))
    lr.lr_set_split_override(3)
    try:
        y, hf = lr.rglru_scan(x.cuda(), r_pre.cuda(), i_pre.cuda(), a_log.cuda(), 8.0,
                              gates_preact=True)
    finally:
        lr.lr_set_split_override(0)
    yr, hr = oracle.rglru_scan(x, torch.sigmoid(r_pre.double()), torch.sigmoid(i_pre.double()),
                               a_log, 8.0)
    assert rel_err(y.float().cpu(), yr) <= TOL[io] and rel_err(hf.cpu(), hr) <= TOL[io]


@pytest.mark.parametrize("B,L,H,lb", [(1, 256, 2, 0.2), (2, 130, 1, 0.5), (1, 1000, 2, 0.2)])
def test_hgrn2_preact_matches_oracle(lr, B, L, H, lb):
    p = wl.hgrn2_inputs(B, L, H, 128, seed=B + L)
    f = torch.randn(B, L, H * 128, generator=torch.Generator().manual_seed(L)).add(2.0).to(torch.bfloat16)
    o, Sf = lr.hgrn2(p["q"].cuda(), p["k"].cuda(), p["v"].cuda(), f.cuda(), H=H, gate_lb=lb)
    torch.cuda.synchronize()
    assert lr.status() == 0
    gate = lb + (1.0 - lb) * torch.sigmoid(f.double())
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], gate, H)
    assert rel_err(o.float().cpu(), orf) <= 1e-2
    assert rel_err(Sf.cpu(), Srf) <= 1e-2


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_rglru_preact_saturated_gates(lr, io):
    """Pre-activations far into both tails (|v| up to 1e4): the sigmoids
    saturate to 0 and 1 -- the fast form's clamped exponentials must agree
    with the exact sigmoid there too."""
    g = torch.Generator().manual_seed(21)
    B, L, D = 2, 333, 128
    x = torch.randn(B, L, D, generator=g).to(DT[io])
    r_pre = (30.0 * torch.randn(B, L, D, generator=g)).to(DT[io])
    i_pre = (30.0 * torch.randn(B, L, D, generator=g)).to(DT[io])
    r_pre[:, ::7] = 1e4
    i_pre[:, 3::11] = -1e4
    a_log = torch.log(0.9 + 0.099 * torch.rand(D, generator=g))
    h0 = torch.randn(B, D, generator=g)
    y, hf = lr.rglru_scan(x.cuda(), r_pre.cuda(), i_pre.cuda(), a_log.cuda(), 8.0, h0=h0.cuda(),
                          gates_preact=True)
    yr, hr = oracle.rglru_scan(x, torch.sigmoid(r_pre.double()), torch.sigmoid(i_pre.double()),
                               a_log, 8.0, h0=h0)
    assert torch.isfinite(y.float()).all() and torch.isfinite(hf).all()
    assert rel_err(y.float().cpu(), yr) <= TOL[io]
    assert rel_err(hf.cpu(), hr) <= TOL[io]
