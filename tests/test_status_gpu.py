"""Device-side status per call.

Every call that can detect an error on the device (a bounded wait that ran
out) records its status in the first bytes of its own workspace, stamped
with the call, and lr_check_status(workspace, stream) reads and resets it.
So concurrent calls on different streams with different workspaces see their
own status, and a workspace's status always describes its latest call,
whatever the memory held before.  The error is made on the host side: the
test hook withholds one time split's carry, so the splits after it wait
~50 ms, give up, and report LR_ERR_TIMEOUT (no GPU fault is involved).
"""
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


@pytest.fixture(autouse=True)
def _knobs(lr):
    lr.lr_set_split_override(0)
    lr.lr_test_withhold_split(-1, 1000)
    lr.lr_set_selective_warmup(-1)
    yield
    lr.lr_set_split_override(0)
    lr.lr_test_withhold_split(-1, 1000)
    lr.lr_set_selective_warmup(-1)


def cuda(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


def rglru_ws(lr, B, L, D):
    return torch.empty(lr.lr_rglru_scan_workspace_size(B, L, D, lr.LR_F32), dtype=torch.uint8,
                       device="cuda")


def test_two_streams_two_workspaces_report_their_own_status(lr):
    host = wl.rglru_inputs(1, 512, 64, seed=3, io="f32", with_h0=True)
    p = cuda(host)
    lr.lr_set_split_override(4)
    ws_bad, ws_good = rglru_ws(lr, 1, 512, 64), rglru_ws(lr, 1, 512, 64)
    s_bad, s_good = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    lr.lr_test_withhold_split(1, 50)          # this call's successors time out ...
    with torch.cuda.stream(s_bad):
        lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"], workspace=ws_bad)
    lr.lr_test_withhold_split(-1, 1000)       # ... this one runs clean, concurrently
    with torch.cuda.stream(s_good):
        y, hf = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"],
                              workspace=ws_good)
    assert lr.status(ws_good, s_good) == lr.LR_OK
    assert lr.status(ws_bad, s_bad) == lr.LR_ERR_TIMEOUT
    assert lr.status(ws_bad, s_bad) == lr.LR_OK     # read and reset
    assert lr.status(ws_good, s_good) == lr.LR_OK
    yr, hr = oracle.rglru_scan(host["x"], host["r"], host["i"], host["a_log"], host["c"],
                               h0=host["h0"])
    assert rel_err(y.cpu(), yr) <= 1e-4 and rel_err(hf.cpu(), hr) <= 1e-4


def test_status_describes_the_latest_call_of_a_workspace(lr):
    p = cuda(wl.rglru_inputs(1, 512, 64, seed=4, io="f32", with_h0=True))
    lr.lr_set_split_override(4)
    ws = rglru_ws(lr, 1, 512, 64)
    ws.fill_(0xFF)                            # stale contents: no initialisation needed
    lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], workspace=ws)
    assert lr.status(ws) == lr.LR_OK
    lr.lr_test_withhold_split(1, 50)
    lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], workspace=ws)
    lr.lr_test_withhold_split(-1, 1000)
    lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], workspace=ws)
    assert lr.status(ws) == lr.LR_OK          # the clean call after the timed-out one
    lr.lr_test_withhold_split(1, 50)
    lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], workspace=ws)
    assert lr.status(ws) == lr.LR_ERR_TIMEOUT


def test_selective_timeout_beside_a_clean_hgrn2_call(lr):
    """The selective scan's look-back wait and HGRN2 report into their own
    workspaces on two streams."""
    q = cuda(wl.selective_inputs(1, 400, 32, seed=4, io="f32", with_h0=True))
    h = cuda(wl.hgrn2_inputs(1, 256, 2, 128, seed=5))
    lr.lr_set_split_override(4)
    lr.lr_set_selective_warmup(0)             # carries by look-back: the withheld one is waited for
    ws_sel = torch.empty(lr.lr_selective_scan_workspace_size(1, 400, 32, 16, lr.LR_F32),
                         dtype=torch.uint8, device="cuda")
    ws_hg = torch.empty(lr.lr_hgrn2_workspace_size(1, 256, 2, 128, 128, lr.LR_BF16),
                        dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    lr.lr_test_withhold_split(2, 50)
    with torch.cuda.stream(s1):
        lr.selective_scan(q["x"], q["dt"], q["Bm"], q["Cm"], q["A_log"], z=q["z"], Dskip=q["Dskip"],
                          h0=q["h0"], workspace=ws_sel)
    lr.lr_test_withhold_split(-1, 1000)
    with torch.cuda.stream(s2):
        lr.hgrn2(h["q"], h["k"], h["v"], h["g"], H=2, workspace=ws_hg)
    assert lr.status(ws_hg, s2) == lr.LR_OK
    assert lr.status(ws_sel, s1) == lr.LR_ERR_TIMEOUT
