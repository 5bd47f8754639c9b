"""The scans the benchmark times beside its step (its `extra` entries), at
the benchmark's full sizes and in the same launch configuration, checked on
sampled channels or heads that the oracle computes independently: MinMax
(exact), RG-LRU and HGRN2 with their gates before the activation, and HGRN2
with fp32 I/O on the step-by-step kernel."""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_err
from selective_state_space_chunked_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_chunked_gb300 import build
    build.build()
    from selective_state_space_chunked_gb300 import binding
    return binding


def test_minmax_bf16_B8_L4096_D2560_sampled_exact(lr):
    B, L, D = 8, 4096, 2560
    g = torch.Generator(device="cuda").manual_seed(11)
    r = torch.randn(B, L, D, device="cuda", generator=g).to(torch.bfloat16)
    s = (torch.randn(B, L, D, device="cuda", generator=g) - 1.0).to(torch.bfloat16)
    x0 = torch.randn(B, D, device="cuda", generator=g).to(torch.bfloat16).float()
    y, xf = lr.minmax_scan(r, s, x0)
    torch.cuda.synchronize()
    assert lr.status() == 0
    rng = np.random.default_rng(3)
    for b in (0, B - 1):
        ds = torch.from_numpy(np.concatenate([np.sort(rng.choice(D, 40, replace=False)), [0, D - 1]])).cuda()
        yr, xr = oracle.minmax_scan(r[b:b + 1][:, :, ds].cpu(), s[b:b + 1][:, :, ds].cpu(), x0[b:b + 1, ds].cpu())
        assert np.array_equal(y[b:b + 1][:, :, ds].double().cpu().numpy(), yr)
        assert np.array_equal(xf[b:b + 1, ds].double().cpu().numpy(), xr)


def test_rglru_preact_bf16_B8_L4096_D2560_sampled(lr):
    cfg = wl.WORKLOADS["rglru_bf16"]
    p = wl.make_inputs(cfg, device="cuda")
    y, hf = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"], gates_preact=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    for b in (0, cfg.B - 1):
        ds = torch.from_numpy(np.concatenate([np.sort(rng.choice(cfg.D, 40, replace=False)), [0, cfg.D - 1]])).cuda()
        sub = {k: p[k][b:b + 1][:, :, ds].cpu() for k in ("x", "r", "i")}
        yr, hr = oracle.rglru_scan(sub["x"], torch.sigmoid(sub["r"].double()), torch.sigmoid(sub["i"].double()),
                                   p["a_log"][ds].cpu(), p["c"], h0=p["h0"][b:b + 1, ds].cpu())
        assert rel_err(y[b:b + 1][:, :, ds].float().cpu(), yr) <= 1e-2
        assert rel_err(hf[b:b + 1, ds].cpu(), hr) <= 1e-2


def test_hgrn2_preact_bf16_B4_L4096_H16_sampled(lr):
    cfg = wl.WORKLOADS["hgrn2_bf16"]
    p = wl.make_inputs(cfg, device="cuda")
    o, Sf = lr.hgrn2(p["q"], p["k"], p["v"], p["g"], H=cfg.H, gate_lb=0.2)
    torch.cuda.synchronize()
    assert lr.status() == 0
    for b, h in ((0, 0), (3, 15)):
        sl = slice(h * 128, (h + 1) * 128)
        sub = {n: p[n][b:b + 1, :, sl].cpu() for n in ("q", "k", "v", "g")}
        gate = 0.2 + 0.8 * torch.sigmoid(sub["g"].double())
        orf, Srf = oracle.hgrn2(sub["q"], sub["k"], sub["v"], gate, 1)
        assert rel_err(o[b:b + 1, :, sl].float().cpu(), orf) <= 1e-2
        assert rel_err(Sf[b:b + 1, h:h + 1].cpu(), Srf) <= 1e-2


def test_hgrn2_f32_B4_L4096_H16_general_kernel_sampled(lr):
    cfg = wl.WORKLOADS["hgrn2_bf16"]
    p = wl.make_inputs(cfg, device="cuda")
    pf = {n: p[n].float() for n in ("q", "k", "v", "g")}
    del p
    o, Sf = lr.hgrn2(pf["q"], pf["k"], pf["v"], pf["g"], H=cfg.H)
    torch.cuda.synchronize()
    assert lr.status() == 0
    for b, h in ((1, 3), (2, 12)):
        sl = slice(h * 128, (h + 1) * 128)
        sub = {n: pf[n][b:b + 1, :, sl].cpu() for n in ("q", "k", "v", "g")}
        orf, Srf = oracle.hgrn2(sub["q"], sub["k"], sub["v"], sub["g"], 1)
        assert rel_err(o[b:b + 1, :, sl].cpu(), orf) <= 1e-4
        assert rel_err(Sf[b:b + 1, h:h + 1].cpu(), Srf) <= 1e-4
