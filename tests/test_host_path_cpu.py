"""Host-buffer entry points (lr_*_fwd_host) without a GPU: argument checks
that come before any CUDA call, and the empty sequence, whose final state is
the initial state (or zero) copied on the host -- no device is touched."""
import ctypes

import numpy as np
import pytest

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced (validation fails first)


@pytest.fixture(scope="module")
def lr():
    from selective_state_space_chunked_gb300 import build
    build.build()
    from selective_state_space_chunked_gb300 import binding
    return binding


def ptr(a):
    return a.ctypes.data


def test_host_entry_points_reject_bad_arguments(lr):
    bad_b = lr.lr_rglru_scan_fwd_host(FAKE, FAKE, FAKE, FAKE, 8.0, None, FAKE, None, -1, 4, 8, 1,
                                      FAKE, 1 << 20, None)
    assert bad_b == lr.LR_ERR_INVALID_ARG
    bad_n = lr.lr_selective_scan_fwd_host(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                          1, 4, 8, 8, 1, 1, FAKE, 1 << 20, None)
    assert bad_n == lr.LR_ERR_UNSUPPORTED
    odd = lr.lr_minmax_scan_fwd_host(FAKE + 4, FAKE, None, FAKE, None, 1, 4, 8, 1, FAKE, 1 << 20, None)
    assert odd == lr.LR_ERR_MISALIGNED
    big_dk = lr.lr_hgrn2_fwd_host(FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 4, 1, 513, 8, 64, 1,
                                  FAKE, 1 << 20, None)
    assert big_dk == lr.LR_ERR_UNSUPPORTED


def test_host_workspace_size_of_an_empty_problem_is_zero(lr):
    assert lr.lr_rglru_scan_fwd_host_workspace_size(0, 16, 8, 1) == 0
    assert lr.lr_selective_scan_fwd_host_workspace_size(2, 0, 8, 16, 1) == 0
    assert lr.lr_hgrn2_fwd_host_workspace_size(1, 0, 2, 64, 64, 1) == 0
    assert lr.lr_minmax_scan_fwd_host_workspace_size(1, 4, 0, 1) == 0


def test_host_chunk_knob_returns_previous_setting(lr):
    prev = lr.lr_set_host_chunk_steps(100)
    try:
        assert lr.lr_set_host_chunk_steps(64) == 100
    finally:
        lr.lr_set_host_chunk_steps(prev)
    assert lr.lr_set_host_chunk_steps(prev) == prev


@pytest.mark.parametrize("with_h0", [True, False])
def test_empty_sequence_copies_the_state_on_the_host(lr, with_h0):
    rng = np.random.default_rng(1)
    B, D, N, H, dk, dv = 2, 8, 16, 2, 4, 4
    # RG-LRU, MinMax: (B, D); selective: (B, D, N); HGRN2: (B, H, dv, dk)
    cases = [
        (lambda h0, hf: lr.lr_rglru_scan_fwd_host(FAKE, FAKE, FAKE, FAKE, 8.0, h0, FAKE, hf, B, 0, D, 1,
                                                  None, 0, None), (B, D)),
        (lambda h0, hf: lr.lr_minmax_scan_fwd_host(FAKE, FAKE, h0, FAKE, hf, B, 0, D, 1, None, 0, None),
         (B, D)),
        (lambda h0, hf: lr.lr_selective_scan_fwd_host(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, h0, FAKE,
                                                      hf, B, 0, D, N, 1, 1, None, 0, None), (B, D, N)),
        (lambda h0, hf: lr.lr_hgrn2_fwd_host(FAKE, FAKE, FAKE, FAKE, h0, FAKE, hf, B, 0, H, dk, dv, 64,
                                             1, None, 0, None), (B, H, dv, dk)),
    ]
    for call, shape in cases:
        h0 = rng.standard_normal(shape).astype(np.float32)
        hf = np.full(shape, 7.0, dtype=np.float32)
        assert call(ptr(h0) if with_h0 else None, ptr(hf)) == lr.LR_OK
        np.testing.assert_array_equal(hf, h0 if with_h0 else np.zeros(shape, np.float32))


def test_queued_host_entry_points_check_arguments_as_the_synchronous_ones(lr):
    """The *_async forms share the synchronous forms' argument checks, which
    return before anything is queued; the empty sequence copies the state on
    the host without queueing anything either."""
    assert lr.lr_rglru_scan_fwd_host_async(FAKE, FAKE, FAKE, FAKE, 8.0, None, FAKE, None, -1, 4, 8, 1,
                                           FAKE, 1 << 20, None) == lr.LR_ERR_INVALID_ARG
    assert lr.lr_selective_scan_fwd_host_async(FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                               1, 4, 8, 8, 1, 1, FAKE, 1 << 20, None) == lr.LR_ERR_UNSUPPORTED
    assert lr.lr_minmax_scan_fwd_host_async(FAKE + 4, FAKE, None, FAKE, None, 1, 4, 8, 1, FAKE, 1 << 20,
                                            None) == lr.LR_ERR_MISALIGNED
    assert lr.lr_hgrn2_fwd_host_async(FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 4, 1, 513, 8, 64, 1,
                                      FAKE, 1 << 20, None) == lr.LR_ERR_UNSUPPORTED
    h0 = np.arange(16, dtype=np.float32).reshape(2, 8)
    hf = np.zeros_like(h0)
    assert lr.lr_rglru_scan_fwd_host_async(FAKE, FAKE, FAKE, FAKE, 8.0, ptr(h0), FAKE, ptr(hf), 2, 0, 8, 1,
                                           None, 0, None) == lr.LR_OK
    np.testing.assert_array_equal(hf, h0)
