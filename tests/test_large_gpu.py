"""Calls past 2^31 elements: every scan at a size whose element offsets
overflow 32-bit integers (the C ABI takes each of B, L and the width up to
INT_MAX, so a call's total can exceed 2^31).

The sequence lengths are ragged (not a multiple of any kernel's tile), and
the outputs are compared with the float64 oracle on the last batch row, where
the offsets are largest, for sampled channels (RG-LRU, selective, MinMax) or
the last head (HGRN2).  Tolerances as everywhere: 1e-2 relative for bf16 I/O,
bit-exact for MinMax.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_err
from selective_state_space_chunked_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

INT32_ELEMS = 2 ** 31


@pytest.fixture(scope="module")
def lr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_chunked_gb300 import build
    build.build()
    from selective_state_space_chunked_gb300 import binding
    return binding


@pytest.fixture(autouse=True)
def _free(lr):
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    assert lr.status() == 0


def channels(D, seed):
    rng = np.random.default_rng(seed)
    ds = np.concatenate([rng.choice(D, 6, replace=False), [0, D // 2 - 1, D - 1]])
    return torch.from_numpy(np.unique(ds)).cuda()


def test_rglru_past_int32_elements(lr):
    B, L, D = 2, 2 ** 19 + 37, 2560
    assert B * L * D > INT32_ELEMS
    p = wl.rglru_inputs(B, L, D, seed=51, io="bf16", with_h0=True, device="cuda")
    y, hf = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    torch.cuda.synchronize()
    b, ds = B - 1, channels(D, 1)
    sub = {k: p[k][b:b + 1][:, :, ds].cpu() for k in ("x", "r", "i")}
    yr, hr = oracle.rglru_scan(sub["x"], sub["r"], sub["i"], p["a_log"][ds].cpu(), p["c"],
                               h0=p["h0"][b:b + 1, ds].cpu())
    assert rel_err(y[b:b + 1][:, :, ds].float().cpu(), yr) <= 1e-2
    assert rel_err(hf[b:b + 1, ds].cpu(), hr) <= 1e-2


def test_selective_past_int32_elements(lr):
    B, L, D = 2, 2 ** 18 + 1000, 4096
    assert B * L * D > INT32_ELEMS
    p = wl.selective_inputs(B, L, D, seed=52, io="bf16", with_h0=True, device="cuda")
    y, hf = lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                              Dskip=p["Dskip"], h0=p["h0"])
    torch.cuda.synchronize()
    b, ds = B - 1, channels(D, 2)
    sub = {k: p[k][b:b + 1][:, :, ds].cpu() for k in ("x", "dt", "z")}
    yr, hr = oracle.selective_scan(sub["x"], sub["dt"], p["Bm"][b:b + 1].cpu(),
                                   p["Cm"][b:b + 1].cpu(), p["A_log"][ds].cpu(), z=sub["z"],
                                   Dskip=p["Dskip"][ds].cpu(), h0=p["h0"][b:b + 1, ds].cpu())
    assert rel_err(y[b:b + 1][:, :, ds].float().cpu(), yr) <= 1e-2
    assert rel_err(hf[b:b + 1, ds].cpu(), hr) <= 1e-2


def test_hgrn2_past_int32_elements(lr):
    B, L, H, d = 8, 2 ** 17 + 40, 16, 128
    assert B * L * H * d > INT32_ELEMS
    p = wl.hgrn2_inputs(B, L, H, d, seed=53, io="bf16", device="cuda")
    o, Sf = lr.hgrn2(p["q"], p["k"], p["v"], p["g"], H=H)
    torch.cuda.synchronize()
    b, h = B - 1, H - 1
    cols = slice(h * d, (h + 1) * d)
    sub = {k: p[k][b:b + 1, :, cols].cpu() for k in ("q", "k", "v", "g")}
    orf, sr = oracle.hgrn2(sub["q"], sub["k"], sub["v"], sub["g"], H=1)
    assert rel_err(o[b:b + 1, :, cols].float().cpu(), orf) <= 1e-2
    assert rel_err(Sf[b:b + 1, h:h + 1].cpu(), sr) <= 1e-2


def test_minmax_past_int32_elements_bit_exact(lr):
    B, L, D = 2, 2 ** 19 + 37, 2560
    assert B * L * D > INT32_ELEMS
    g = torch.Generator(device="cuda").manual_seed(54)
    r = torch.randn(B, L, D, device="cuda", generator=g).to(torch.bfloat16)
    s = (torch.randn(B, L, D, device="cuda", generator=g) - 1.0).to(torch.bfloat16)
    x0 = torch.randn(B, D, device="cuda", generator=g).to(torch.bfloat16).float()  # representable
    y, xf = lr.minmax_scan(r, s, x0)
    torch.cuda.synchronize()
    b, ds = B - 1, channels(D, 3)
    yr, xr = oracle.minmax_scan(r[b:b + 1][:, :, ds].cpu(), s[b:b + 1][:, :, ds].cpu(),
                                x0[b:b + 1, ds].cpu())
    assert np.array_equal(y[b:b + 1][:, :, ds].double().cpu().numpy(), yr)
    assert np.array_equal(xf[b:b + 1, ds].double().cpu().numpy(), xr)
