"""Host-buffer entry points on the GPU: the sequence runs through the device
in chunks (here forced short: 100 steps, so chunk boundaries fall off the
kernels' tiles, and 64) with the state carried across; results against the
oracle and against the device-buffer call, with pinned and pageable inputs,
caller-given and library-allocated outputs."""
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


@pytest.fixture(params=[100, 64])
def chunk(lr, request):
    prev = lr.lr_set_host_chunk_steps(request.param)
    yield request.param
    lr.lr_set_host_chunk_steps(prev)


def pinned(d):
    return {k: (v.pin_memory() if torch.is_tensor(v) else v) for k, v in d.items()}


def cuda(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_rglru_host_path(lr, chunk, io):
    p = pinned(wl.rglru_inputs(2, 333, 64, seed=21, io=io, with_h0=True))
    y, hf = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    assert y.device.type == "cpu" and hf.device.type == "cpu"
    yr, hr = oracle.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    assert rel_err(y.float(), yr) <= TOL[io] and rel_err(hf, hr) <= TOL[io]
    d = cuda(p)
    yd, hd = lr.rglru_scan(d["x"], d["r"], d["i"], d["a_log"], d["c"], h0=d["h0"])
    assert rel_err(y.float(), yd.float().cpu()) <= 1e-5 and rel_err(hf, hd.cpu()) <= 1e-5


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selective_host_path(lr, chunk, io):
    p = pinned(wl.selective_inputs(2, 250, 64, seed=22, io=io, with_h0=True))
    y, hf = lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                              Dskip=p["Dskip"], h0=p["h0"])
    yr, hr = oracle.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                                   Dskip=p["Dskip"], h0=p["h0"])
    assert rel_err(y.float(), yr) <= TOL[io] and rel_err(hf, hr) <= TOL[io]


def test_selective_host_path_without_optional_tensors(lr, chunk):
    p = pinned(wl.selective_inputs(1, 180, 32, seed=23, io="f32"))
    y, hf = lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"])
    yr, hr = oracle.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"])
    assert rel_err(y, yr) <= 1e-4 and rel_err(hf, hr) <= 1e-4


@pytest.mark.parametrize("io,dk", [("bf16", 128), ("f32", 64)])
def test_hgrn2_host_path(lr, chunk, io, dk):
    """bf16 128 x 128: every chunk on the tensor-core kernel; fp32: the
    step-by-step kernel."""
    p = pinned(wl.hgrn2_inputs(1, 300, 2, dk, seed=24, io=io, with_S0=True))
    S0 = 0.1 * p["S0"]
    o, Sf = lr.hgrn2(p["q"], p["k"], p["v"], p["g"], H=2, S0=S0)
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], 2, S0=S0)
    assert lr.status() == 0
    assert rel_err(o.float(), orf) <= TOL[io] and rel_err(Sf, Srf) <= TOL[io]


def test_minmax_host_path_is_bitwise(lr, chunk):
    g = torch.Generator().manual_seed(25)
    r = torch.randn(2, 333, 64, generator=g).to(torch.bfloat16).pin_memory()
    s = (torch.randn(2, 333, 64, generator=g) - 1.0).to(torch.bfloat16).pin_memory()
    x0 = torch.randn(2, 64, generator=g).to(torch.bfloat16).float()   # representable in the output
    y, xf = lr.minmax_scan(r, s, x0)
    yd, xd = lr.minmax_scan(r.cuda(), s.cuda(), x0.cuda())
    assert torch.equal(y, yd.cpu()) and torch.equal(xf, xd.cpu())
    yr, xr = oracle.minmax_scan(r, s, x0)
    assert np.array_equal(y.double().numpy(), yr) and np.array_equal(xf.double().numpy(), xr)


def test_host_path_with_pageable_inputs_and_given_outputs(lr, chunk):
    p = wl.rglru_inputs(1, 257, 32, seed=26, io="f32", with_h0=True)   # pageable
    y = torch.full((1, 257, 32), float("nan"))
    hf = torch.full((1, 32), float("nan"))
    ry, rh = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"], out=(y, hf))
    assert ry is y and rh is hf
    yr, hr = oracle.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    assert rel_err(y, yr) <= 1e-4 and rel_err(hf, hr) <= 1e-4


def test_host_path_rejects_a_small_workspace(lr, chunk):
    p = pinned(wl.rglru_inputs(1, 200, 32, seed=27, io="bf16"))
    need = lr.lr_rglru_scan_fwd_host_workspace_size(1, 200, 32, lr.LR_BF16)
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lr.LrError) as e:
        lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], workspace=ws)
    assert e.value.code == lr.LR_ERR_WORKSPACE


def test_host_path_calls_from_two_threads_match_sequential(lr, chunk):
    """Host-buffer calls on one device are serialised inside the library
    (its streams and the staging workspace are shared); two Python threads
    calling at once get the same results as one after the other."""
    import threading
    inputs = [pinned(wl.rglru_inputs(1, 400, 64, seed=30 + k, io="bf16", with_h0=True)) for k in range(3)]
    ref = [lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"]) for p in inputs]
    got = [None] * len(inputs)
    errors = []

    def run(k):
        try:
            p = inputs[k]
            got[k] = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
        except Exception as e:   # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(k,)) for k in range(len(inputs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for (y, hf), (yr, hr) in zip(got, ref):
        assert torch.equal(y, yr) and torch.equal(hf, hr)


def test_queued_host_calls_match_the_synchronous_calls(lr, chunk):
    """RG-LRU, selective, HGRN2 and MinMax host-buffer calls queued with
    ``sync_host=False`` (two with their own workspace, two with one the
    binding allocates), then one ``host_sync()``: the calls overlap on the
    library's streams and every output and final state matches the
    synchronous call's (the same kernels over the same chunks); each call's
    device status is clear."""
    rg = pinned(wl.rglru_inputs(2, 333, 64, seed=41, io="bf16", with_h0=True))
    se = pinned(wl.selective_inputs(2, 250, 64, seed=42, io="f32", with_h0=True))
    hg = pinned(wl.hgrn2_inputs(1, 300, 2, 128, seed=43, io="bf16", with_S0=True))
    g = torch.Generator().manual_seed(44)
    mr = torch.randn(2, 333, 64, generator=g).to(torch.bfloat16).pin_memory()
    ms = (torch.randn(2, 333, 64, generator=g) - 1.0).to(torch.bfloat16).pin_memory()
    calls = [
        lambda **kw: lr.rglru_scan(rg["x"], rg["r"], rg["i"], rg["a_log"], rg["c"], h0=rg["h0"], **kw),
        lambda **kw: lr.selective_scan(se["x"], se["dt"], se["Bm"], se["Cm"], se["A_log"], z=se["z"],
                                       Dskip=se["Dskip"], h0=se["h0"], **kw),
        lambda **kw: lr.hgrn2(hg["q"], hg["k"], hg["v"], hg["g"], H=2, S0=0.1 * hg["S0"], **kw),
        lambda **kw: lr.minmax_scan(mr, ms, **kw),
    ]
    sync = [c() for c in calls]
    sizes = [lr.lr_rglru_scan_fwd_host_workspace_size(2, 333, 64, lr.LR_BF16),
             lr.lr_selective_scan_fwd_host_workspace_size(2, 250, 64, 16, lr.LR_F32)]
    wss = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in sizes] + [None, None]
    queued = []
    for c, ws in zip(calls, wss):
        queued.append(c(workspace=ws, sync_host=False))
        if ws is None:
            wss[len(queued) - 1] = lr._tls.ws   # the workspace the binding allocated for the call
    lr.host_sync()
    for ws in wss:
        assert lr.status(ws) == 0
    for (a, b), (ra, rb) in zip(queued, sync):
        assert rel_err(a.float(), ra.float()) <= 1e-6 and rel_err(b, rb) <= 1e-6
    assert torch.equal(queued[3][0], sync[3][0]) and torch.equal(queued[3][1], sync[3][1])
    yr, hr = oracle.rglru_scan(rg["x"], rg["r"], rg["i"], rg["a_log"], rg["c"], h0=rg["h0"])
    assert rel_err(queued[0][0].float(), yr) <= TOL["bf16"] and rel_err(queued[0][1], hr) <= TOL["bf16"]
