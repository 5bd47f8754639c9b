"""The RG-LRU entry point for callers that cannot allocate device memory.

lr_rglru_scan_fwd_noalloc takes no workspace: its look-back scratch and its
call status live in an array built into the library.  These tests call it
through the C ABI on problems small enough that the scan splits time across
thread blocks (so the built-in scratch is really used) and compare it, on two
calls in a row with different inputs, with

* lr_rglru_scan_fwd given a caller-allocated workspace: the same kernel with
  the same split plan.  With two time splits the second split's carry is
  always the first split's final state, so both entry points round alike and
  must agree bit for bit -- a leftover of the previous call in the shared
  scratch would show here.  With the automatic split count the look-back may
  compose a different number of descriptors from run to run (a different
  rounding order), so that case is compared within the tolerance;
* the float64 oracle, within the parity tolerance (1e-4 fp32, 1e-2 bf16).

The file is named to be collected last.
"""
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
    binding.lr_set_split_override(0)
    binding.lr_test_withhold_split(-1, 1000)
    return binding


def _noalloc(lr, p):
    B, L, D = p["x"].shape
    y = torch.empty_like(p["x"])
    hf = torch.empty(B, D, dtype=torch.float32, device="cuda")
    io = lr.LR_BF16 if p["x"].dtype == torch.bfloat16 else lr.LR_F32
    stream = torch.cuda.current_stream().cuda_stream
    rc = lr.lr_rglru_scan_fwd_noalloc(
        p["x"].data_ptr(), p["r"].data_ptr(), p["i"].data_ptr(), p["a_log"].data_ptr(),
        float(p["c"]), p["h0"].data_ptr() if p["h0"] is not None else None,
        y.data_ptr(), hf.data_ptr(), B, L, D, io, stream)
    assert rc == 0, lr.lr_status_string(rc)
    # the call's device-side status sits in the built-in scratch
    assert lr.lr_check_status(None, stream) == 0
    return y, hf


def _with_workspace(lr, p):
    return lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])


@pytest.mark.parametrize("splits", [2, 0])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_noalloc_matches_workspace_entry_and_oracle_two_calls(lr, io, splits):
    B, L, D = 2, 2000, 128
    prev = lr.lr_set_split_override(splits)
    try:
        plan_ws = lr.lr_rglru_scan_workspace_size(B, L, D, lr.LR_BF16 if io == "bf16" else lr.LR_F32)
        assert plan_ws > 256   # the plan splits time: look-back scratch beyond the status bytes
        for seed in (11, 12):   # two calls in a row, different inputs
            host = wl.rglru_inputs(B, L, D, seed=seed, io=io, with_h0=True)
            p = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in host.items()}
            y0, h0 = _noalloc(lr, p)
            y1, h1 = _with_workspace(lr, p)
            torch.cuda.synchronize()
            assert lr.status() == 0
            if splits == 2:
                assert torch.equal(y0, y1) and torch.equal(h0, h1)
            else:
                assert rel_err(y0.float().cpu(), y1.float().cpu()) <= TOL[io]
                assert rel_err(h0.cpu(), h1.cpu()) <= TOL[io]
            yr, hr = oracle.rglru_scan(host["x"], host["r"], host["i"], host["a_log"], host["c"],
                                       h0=host["h0"])
            assert rel_err(y0.float().cpu(), yr) <= TOL[io]
            assert rel_err(h0.cpu(), hr) <= TOL[io]
    finally:
        lr.lr_set_split_override(prev)


def test_noalloc_rejects_problems_beyond_builtin_scratch(lr):
    p = {k: (v.cuda() if torch.is_tensor(v) else v)
         for k, v in wl.rglru_inputs(4, 8192, 256, seed=1, io="bf16").items()}
    # 16 blocks x 128 splits (one 64-step tile each): ~1.6 MB of scratch
    prev = lr.lr_set_split_override(128)
    try:
        assert lr.lr_rglru_scan_workspace_size(4, 8192, 256, lr.LR_BF16) > (1 << 20)
        y = torch.empty_like(p["x"])
        rc = lr.lr_rglru_scan_fwd_noalloc(
            p["x"].data_ptr(), p["r"].data_ptr(), p["i"].data_ptr(), p["a_log"].data_ptr(),
            8.0, None, y.data_ptr(), None, 4, 8192, 256, lr.LR_BF16,
            torch.cuda.current_stream().cuda_stream)
        assert rc == lr.LR_ERR_WORKSPACE
    finally:
        lr.lr_set_split_override(prev)
