"""Caller-provided result buffers (``out=``) of the three scans: GPU tensors
are written in place, host tensors receive a copy, and both equal the
default call bit for bit; a buffer of the wrong shape or dtype is rejected."""
import pytest
import torch

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


def calls(lr):
    p1 = wl.rglru_inputs(2, 100, 64, seed=21, io="bf16", with_h0=True)
    p2 = wl.selective_inputs(2, 100, 64, seed=22, io="bf16", with_h0=True)
    p3 = wl.hgrn2_inputs(1, 100, 2, 128, seed=23)
    return [
        (p1, lambda p, out: lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"],
                                          out=out)),
        (p2, lambda p, out: lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                                              Dskip=p["Dskip"], h0=p["h0"], out=out)),
        (p3, lambda p, out: lr.hgrn2(p["q"], p["k"], p["v"], p["g"], H=2, out=out)),
    ]


@pytest.fixture
def one_split(lr):
    # A single time split keeps the diagonal scans bit-reproducible: with
    # several, the look-back may combine carries in a different rounding
    # order from one run to the next.
    lr.lr_set_split_override(1)
    yield
    lr.lr_set_split_override(0)


def test_out_on_gpu_and_host_match_default(lr, one_split):
    for p, fn in calls(lr):
        dp = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in p.items()}
        ref = [t.cpu() for t in fn(dp, None)]
        dev_out = tuple(torch.empty_like(t, device="cuda") for t in ref)
        got = fn(dp, dev_out)
        assert all(g is d for g, d in zip(got, dev_out))
        torch.cuda.synchronize()
        host_out = tuple(torch.empty_like(t).pin_memory() for t in ref)
        got_h = fn(p, host_out)   # host inputs, host results
        assert all(g is h for g, h in zip(got_h, host_out))
        for r, d, h in zip(ref, dev_out, host_out):
            assert torch.equal(r, d.cpu()) and torch.equal(r, h)


def test_out_mismatch_rejected(lr):
    p, fn = calls(lr)[0]
    dp = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in p.items()}
    y, hf = fn(dp, None)
    with pytest.raises(ValueError):
        fn(dp, (torch.empty(y.shape[0], y.shape[1] + 1, y.shape[2], dtype=y.dtype, device="cuda"), hf))
    with pytest.raises(ValueError):
        fn(dp, (y.float(), hf))
    with pytest.raises(ValueError):
        fn(dp, (y, hf.cpu()))
