"""The C-ABI library loads, exports every symbol include/lrscan.h declares,
and rejects bad arguments before any CUDA call.

No test here launches anything: every call carries at least one invalid
argument, which the library's host-side validation catches first, so fake
pointers are never dereferenced.  Runs without a GPU.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lrscan.h")


@pytest.fixture(scope="module")
def lr():
    from selective_state_space_chunked_gb300 import build
    build.build()
    from selective_state_space_chunked_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lr_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_scans():
    names = declared_functions()
    for n in ("lr_selective_scan_fwd", "lr_rglru_scan_fwd", "lr_hgrn2_fwd",
              "lr_check_status", "lr_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lr):
    import ctypes
    so = ctypes.CDLL(lr.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(lr.SIGNATURES)


def test_status_strings_and_version(lr):
    assert lr.lr_status_string(0) == "LR_OK"
    for code in range(-7, 0):
        assert lr.lr_status_string(code).startswith("LR_ERR_")
    assert lr.lr_status_string(-99) == "unknown lrscan status"
    assert lr.lr_version() >= 10000


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced (validation fails first)


def sel_args(**kw):
    a = dict(x=FAKE, dt=FAKE, z=FAKE, Bm=FAKE, Cm=FAKE, A_log=FAKE, Dskip=FAKE,
             h0=FAKE, y=FAKE, h_final=FAKE, B=2, L=64, D=64, N=16, io=1,
             dt_softplus=1, workspace=None, ws_bytes=0, stream=None)
    a.update(kw)
    return a


def call_sel(lr, **kw):
    a = sel_args(**kw)
    return lr.lr_selective_scan_fwd(*a.values())


@pytest.mark.parametrize("field", ["x", "dt", "Bm", "Cm", "A_log", "y"])
def test_selective_null_required_pointer(lr, field):
    assert call_sel(lr, **{field: None}) == lr.LR_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), -1), (dict(L=-5), -1), (dict(D=-8), -1), (dict(io=7), -1),
    (dict(N=8), -2), (dict(D=60), -2), (dict(D=66, io=0), -2),
    (dict(L=1 << 40), -2),
    (dict(x=FAKE + 4), -3), (dict(Cm=FAKE + 8), -3), (dict(h0=FAKE + 2), -3),
    (dict(h_final=FAKE + 12), -3), (dict(z=FAKE + 1), -3),
])
def test_selective_validation_codes(lr, kw, code):
    assert call_sel(lr, **kw) == code


def rg_args(**kw):
    a = dict(x=FAKE, r=FAKE, i=FAKE, a_log=FAKE, c=8.0, h0=FAKE, y=FAKE,
             h_final=FAKE, B=2, L=64, D=64, io=1, workspace=None, ws_bytes=0,
             stream=None)
    a.update(kw)
    return a


def call_rg(lr, **kw):
    return lr.lr_rglru_scan_fwd(*rg_args(**kw).values())


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), -1), (dict(r=None), -1), (dict(i=None), -1),
    (dict(a_log=None), -1), (dict(y=None), -1), (dict(c=float("nan")), -1),
    (dict(c=float("inf")), -1), (dict(B=-1), -1), (dict(io=2), -1),
    (dict(D=12), -2), (dict(D=6, io=0), -2),
    (dict(r=FAKE + 8), -3), (dict(a_log=FAKE + 4), -3),
])
def test_rglru_validation_codes(lr, kw, code):
    assert call_rg(lr, **kw) == code


def hg_args(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, S0=FAKE, o=FAKE, S_final=FAKE,
             B=2, L=64, H=4, dk=128, dv=128, chunk=64, io=1, workspace=None,
             ws_bytes=0, stream=None)
    a.update(kw)
    return a


def call_hg(lr, **kw):
    return lr.lr_hgrn2_fwd(*hg_args(**kw).values())


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(g=None), -1), (dict(o=None), -1),
    (dict(H=0), -1), (dict(dk=0), -1), (dict(chunk=0), -1), (dict(B=-2), -1),
    (dict(dk=513), -2), (dict(dk=4096), -2),
    (dict(k=FAKE + 2), -3), (dict(S0=FAKE + 4), -3),
])
def test_hgrn2_validation_codes(lr, kw, code):
    assert call_hg(lr, **kw) == code


def test_workspace_size_of_empty_problems_is_the_call_status(lr):
    """Every call's device status lives in its workspace's first 256 bytes,
    so even an empty problem (nothing launched) asks for them; invalid
    arguments ask for nothing."""
    assert lr.lr_selective_scan_workspace_size(0, 10, 64, 16, 1) == 256
    assert lr.lr_selective_scan_workspace_size(1, 10, 64, 8, 1) == 0     # N != 16
    assert lr.lr_selective_scan_workspace_size(-1, 10, 64, 16, 1) == 0
    assert lr.lr_rglru_scan_workspace_size(1, 0, 64, 1) == 256
    assert lr.lr_minmax_scan_workspace_size(1, 4, 0, 1) == 256
    assert lr.lr_hgrn2_workspace_size(1, 0, 2, 128, 128, 1) == 256
    # HGRN2 adds one 8-byte redo mark per thread block (B * H * 2 blocks)
    assert lr.lr_hgrn2_workspace_size(2, 64, 3, 128, 128, 1) == 256 + 2 * 3 * 2 * 8
    assert lr.lr_hgrn2_workspace_size(1, 0, 0, 128, 128, 1) == 0         # H == 0


def test_hgrn2_needs_a_workspace_for_its_status(lr):
    """HGRN2 keeps its device status (LR_ERR_RANGE / LR_ERR_TIMEOUT) in the
    caller's workspace like the other scans: no workspace, no call."""
    rc = lr.lr_hgrn2_fwd(FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 4, 2, 128, 128, 64, 1,
                         None, 0, None)
    assert rc == lr.LR_ERR_WORKSPACE


def test_hidden_not_divisible_by_heads_raises_value_error(lr):
    import torch
    q = torch.zeros(1, 4, 100, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lr.hgrn2(q, q, q, q, H=3)


def test_package_has_no_cpu_fallback():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "selective_state_space_chunked_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


# ----------------------------------------------------------- decode steps
def call_sel_step(lr, **kw):
    a = dict(x=FAKE, dt=FAKE, z=FAKE, Bm=FAKE, Cm=FAKE, A_log=FAKE, Dskip=FAKE,
             h_in=FAKE, h_out=FAKE, y=FAKE, B=2, D=64, N=16, io=1, dt_softplus=1,
             stream=None)
    a.update(kw)
    return lr.lr_selective_scan_step(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), -1), (dict(Bm=None), -1), (dict(A_log=None), -1), (dict(h_out=None), -1),
    (dict(y=None), -1), (dict(B=-1), -1), (dict(io=3), -1),
    (dict(N=8), -2),
    (dict(h_in=FAKE + 4), -3), (dict(y=FAKE + 2), -3),
])
def test_selective_step_validation_codes(lr, kw, code):
    assert call_sel_step(lr, **kw) == code


def call_rg_step(lr, **kw):
    a = dict(x=FAKE, r=FAKE, i=FAKE, a_log=FAKE, c=8.0, h_in=FAKE, h_out=FAKE, y=FAKE,
             B=2, D=64, io=1, stream=None)
    a.update(kw)
    return lr.lr_rglru_scan_step(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(r=None), -1), (dict(h_out=None), -1), (dict(c=float("nan")), -1), (dict(D=-1), -1),
    (dict(i=FAKE + 8), -3),
])
def test_rglru_step_validation_codes(lr, kw, code):
    assert call_rg_step(lr, **kw) == code


def call_hg_step(lr, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, S_in=FAKE, S_out=FAKE, o=FAKE, B=2, H=4,
             dk=128, dv=128, io=1, stream=None)
    a.update(kw)
    return lr.lr_hgrn2_step(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(v=None), -1), (dict(S_out=None), -1), (dict(H=0), -1), (dict(dk=0), -1),
    (dict(B=-1), -1), (dict(io=5), -1),
    (dict(S_in=FAKE + 4), -3),
])
def test_hgrn2_step_validation_codes(lr, kw, code):
    assert call_hg_step(lr, **kw) == code


def test_steps_with_no_elements_launch_nothing(lr):
    # zero batch: nothing to do, no pointer needed, no CUDA call made
    assert call_sel_step(lr, B=0, x=None, y=None, h_out=None) == 0
    assert call_rg_step(lr, D=0, x=None, y=None, h_out=None) == 0
    assert call_hg_step(lr, B=0, q=None, o=None, S_out=None) == 0


def call_mm(lr, **kw):
    a = dict(r=FAKE, s=FAKE, x0=FAKE, y=FAKE, x_final=FAKE, B=2, L=64, D=64, io=1,
             workspace=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lr.lr_minmax_scan_fwd(*a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(r=None), -1), (dict(s=None), -1), (dict(y=None), -1), (dict(B=-1), -1),
    (dict(io=4), -1), (dict(D=12), -2), (dict(D=6, io=0), -2), (dict(L=1 << 40), -2),
    (dict(x0=FAKE + 4), -3), (dict(x_final=FAKE + 8), -3),
])
def test_minmax_validation_codes(lr, kw, code):
    assert call_mm(lr, **kw) == code


@pytest.mark.parametrize("lb", [1.0, -0.1, float("nan")])
def test_hgrn2_preact_rejects_lower_bound_outside_unit_interval(lr, lb):
    a = hg_args()
    a = dict(q=a["q"], k=a["k"], v=a["v"], f=a["g"], lb=lb, S0=a["S0"], o=a["o"],
             S_final=a["S_final"], B=2, L=64, H=4, dk=128, dv=128, chunk=64, io=1,
             workspace=None, ws_bytes=0, stream=None)
    assert lr.lr_hgrn2_preact_fwd(*a.values()) == lr.LR_ERR_INVALID_ARG


def test_rglru_preact_validation_matches_plain(lr):
    a = rg_args(r=None)
    assert lr.lr_rglru_scan_preact_fwd(*a.values()) == lr.LR_ERR_INVALID_ARG
    a = rg_args(D=12)
    assert lr.lr_rglru_scan_preact_fwd(*a.values()) == lr.LR_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,code", [(dict(r=None), -1), (dict(x_out=None), -1), (dict(B=-1), -1),
                                     (dict(x_in=FAKE + 4), -3)])
def test_minmax_step_validation_codes(lr, kw, code):
    a = dict(r=FAKE, s=FAKE, x_in=FAKE, x_out=FAKE, y=FAKE, B=2, D=64, io=1, stream=None)
    a.update(kw)
    assert lr.lr_minmax_scan_step(*a.values()) == code


def test_selective_warmup_knob_round_trips(lr):
    """The warm-up limit is process-wide: negative means automatic (reported
    as -1), 0 turns warm-ups off, larger values are capped at 2^30 steps."""
    prev = lr.lr_set_selective_warmup(5000)
    try:
        assert lr.lr_set_selective_warmup(0) == 5000
        assert lr.lr_set_selective_warmup(-7) == 0
        assert lr.lr_set_selective_warmup(1 << 40) == -1
        assert lr.lr_set_selective_warmup(-1) == 1 << 30
    finally:
        lr.lr_set_selective_warmup(prev)
