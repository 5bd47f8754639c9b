"""Parity of the CUDA MinMax scan with the float64 oracle.

The recurrence only selects among its arguments (min / max), so the GPU
result must equal the oracle bit for bit: every output is one of the inputs
or x0 (x0 is drawn representable in the I/O dtype).  Cases span several
tiles and blocks, ragged sequence and channel ends, both dtypes, forced time
splits (the look-back composes the page's operator), NaN propagation, zero
length, the bounded look-back wait, and the full-size shape B=8, L=4096,
D=2560 in bf16 checked on sampled channels.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def lr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_chunked_gb300 import build
    build.build()
    from selective_state_space_chunked_gb300 import binding
    binding.lr_set_split_override(0)
    binding.lr_test_withhold_split(-1, 1000)
    yield binding
    binding.lr_set_split_override(0)


def inputs(B, L, D, seed, io, with_x0=True):
    g = torch.Generator().manual_seed(seed)
    r = torch.randn(B, L, D, generator=g).to(DT[io])
    s = (torch.randn(B, L, D, generator=g) - 1.0).to(DT[io])
    x0 = torch.randn(B, D, generator=g).to(DT[io]).float() if with_x0 else None
    return r, s, x0


def check(lr, r, s, x0):
    y, xf = lr.minmax_scan(r.cuda(), s.cuda(), None if x0 is None else x0.cuda())
    torch.cuda.synchronize()
    assert lr.status() == 0
    yr, xr = oracle.minmax_scan(r, s, x0)
    yg = y.double().cpu().numpy()
    assert np.array_equal(yg, yr, equal_nan=True)
    assert np.array_equal(xf.double().cpu().numpy(), xr, equal_nan=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("B,L,D", [(2, 256, 128), (3, 77, 64), (1, 1, 8), (2, 300, 72),
                                   (1, 1000, 136)])
def test_minmax_oracle_sized(lr, io, B, L, D):
    check(lr, *inputs(B, L, D, seed=B * 1000 + L + D, io=io))


def test_minmax_default_zero_state(lr):
    check(lr, *inputs(2, 100, 64, seed=5, io="bf16", with_x0=False))


@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_minmax_forced_time_splits_lookback(lr, splits, io):
    lr.lr_set_split_override(splits)
    try:
        check(lr, *inputs(2, 700, 64, seed=splits, io=io))
    finally:
        lr.lr_set_split_override(0)


def test_minmax_nan_propagates(lr):
    r, s, x0 = inputs(1, 90, 64, seed=6, io="f32")
    r[0, 10, 3] = float("nan")
    s[0, 50, 9] = float("nan")
    check(lr, r, s, x0)
    lr.lr_set_split_override(3)
    try:
        check(lr, r, s, x0)
    finally:
        lr.lr_set_split_override(0)


def test_minmax_zero_length_returns_initial_state(lr):
    r, s, x0 = inputs(2, 0, 64, seed=7, io="bf16")
    y, xf = lr.minmax_scan(r.cuda(), s.cuda(), x0.cuda())
    assert y.shape == (2, 0, 64) and torch.equal(xf.cpu(), x0)


def test_minmax_bounded_lookback_wait_reports_timeout(lr):
    r, s, x0 = inputs(1, 512, 64, seed=8, io="f32")
    lr.lr_set_split_override(4)
    lr.lr_test_withhold_split(1, 50)
    try:
        lr.minmax_scan(r.cuda(), s.cuda(), x0.cuda())
        assert lr.status() == lr.LR_ERR_TIMEOUT
        assert lr.status() == 0
    finally:
        lr.lr_test_withhold_split(-1, 1000)
        lr.lr_set_split_override(0)
    check(lr, r, s, x0)


def test_minmax_full_size_sampled(lr):
    """B=8, L=4096, D=2560 in bf16 (the RG-LRU workload's shape), one launch;
    sampled channels of two batch rows against the oracle."""
    r, s, x0 = inputs(8, 4096, 2560, seed=9, io="bf16")
    y, xf = lr.minmax_scan(r.cuda(), s.cuda(), x0.cuda())
    torch.cuda.synchronize()
    assert lr.status() == 0
    for b in (0, 7):
        ch = torch.arange(0, 2560, 37)
        yr, xr = oracle.minmax_scan(r[b:b + 1, :, ch], s[b:b + 1, :, ch], x0[b:b + 1, ch])
        assert np.array_equal(y[b:b + 1, :, ch].double().cpu().numpy(), yr)
        assert np.array_equal(xf[b:b + 1, ch].double().cpu().numpy(), xr)
