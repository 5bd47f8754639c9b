"""Parity of the CUDA selective-SSM and RG-LRU scans with the float64 oracle.

Metric (per output, y and final state separately): max|gpu - ref| / max|ref|,
at most 1e-4 for fp32 I/O and 1e-2 for bf16 I/O.  Oracle-sized cases span
many tiles, ragged tails, odd channel counts and forced time splits (the
decoupled look-back path).  The selective scan has two decay forms: the
workloads' multi-scale A_log sits on the initialisation lattice (the powers
form), and A_log moved off it takes the general one-exp-per-state form; both
are checked, alone and mixed in one launch.  The full-size workloads run in the launch
configuration the benchmark times and are checked on sampled channels, which
the oracle computes independently of one another.
"""
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


WARMUP_DEFAULT = -1   # automatic: 2048 steps for bf16 outputs, look-back for fp32


@pytest.fixture(autouse=True)
def _clean_knobs(lr):
    lr.lr_set_split_override(0)
    lr.lr_test_withhold_split(-1, 1000)
    lr.lr_set_selective_warmup(WARMUP_DEFAULT)
    yield
    lr.lr_set_split_override(0)
    lr.lr_test_withhold_split(-1, 1000)
    lr.lr_set_selective_warmup(WARMUP_DEFAULT)
    assert lr.status() == 0


def cuda(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


# ---------------------------------------------------------------------------
# RG-LRU
# ---------------------------------------------------------------------------
def run_rglru(lr, p):
    g = cuda(p)
    y, hf = lr.rglru_scan(g["x"], g["r"], g["i"], g["a_log"], g["c"], h0=g["h0"])
    torch.cuda.synchronize()
    return y.float().cpu(), hf.cpu()


def check_rglru(lr, p, io):
    y, hf = run_rglru(lr, p)
    yr, hr = oracle.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    assert rel_err(y, yr) <= TOL[io], rel_err(y, yr)
    assert rel_err(hf, hr) <= TOL[io], rel_err(hf, hr)
    return y, hf


def test_rglru_small_f32_page_example(lr):
    """B=2, L=128, D=64, fp32 (the page's (2,128,64) -> (2,128,64) example)."""
    cfg = wl.WORKLOADS["rglru_f32_small"]
    p = wl.make_inputs(cfg)
    y, hf = check_rglru(lr, p, "f32")
    assert y.shape == (2, 128, 64) and hf.shape == (2, 64)


@pytest.mark.parametrize("B,L,D,io,h0", [
    (2, 1000, 256, "bf16", True),    # ragged L (not a multiple of 32)
    (3, 257, 72, "bf16", False),     # D not a multiple of the 64-channel block
    (1, 1, 64, "f32", True),         # single step
    (2, 33, 12, "f32", True),        # tiny ragged everything
    (4, 640, 2560, "bf16", True),    # the RG-LRU workload's channel width
])
def test_rglru_oracle_sized(lr, B, L, D, io, h0):
    p = wl.rglru_inputs(B, L, D, seed=B * 1000 + L, io=io, with_h0=h0)
    check_rglru(lr, p, io)


@pytest.mark.parametrize("splits", [2, 3, 7])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_rglru_forced_time_splits_lookback(lr, splits, io):
    p = wl.rglru_inputs(2, 700, 128, seed=splits, io=io, with_h0=True)
    lr.lr_set_split_override(splits)
    check_rglru(lr, p, io)


def test_rglru_split_resume_matches_one_call(lr):
    """Without time splits the recurrence runs in the same order either way,
    so resuming from the carried state reproduces one call bit for bit."""
    lr.lr_set_split_override(1)
    p = cuda(wl.rglru_inputs(2, 512, 128, seed=5, io="bf16", with_h0=True))
    y, hf = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    h = p["h0"]
    ys = []
    for sl in (slice(0, 96), slice(96, 300), slice(300, 512)):
        yk, h = lr.rglru_scan(p["x"][:, sl], p["r"][:, sl], p["i"][:, sl], p["a_log"],
                              p["c"], h0=h)
        ys.append(yk)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, 1), y)
    assert torch.equal(h, hf)


def test_rglru_zero_length_returns_initial_state(lr):
    p = cuda(wl.rglru_inputs(2, 0, 64, seed=0, io="f32", with_h0=True))
    y, hf = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], 8.0, h0=p["h0"])
    assert y.shape == (2, 0, 64)
    assert torch.equal(hf, p["h0"])


def test_rglru_bf16_B8_L4096_D2560_sampled(lr):
    """B=8, L=4096, D=2560, bf16 I/O, h0 ~ N(0,1): the benchmark's launch."""
    cfg = wl.WORKLOADS["rglru_bf16"]
    p = wl.make_inputs(cfg, device="cuda")
    y, hf = lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    for b in (0, cfg.B - 1):
        ds = np.sort(rng.choice(cfg.D, 48, replace=False))
        ds = torch.from_numpy(np.concatenate([ds, [0, 63, 64, cfg.D - 1]])).cuda()
        sub = {k: p[k][b:b + 1][:, :, ds].cpu() for k in ("x", "r", "i")}
        yr, hr = oracle.rglru_scan(sub["x"], sub["r"], sub["i"], p["a_log"][ds].cpu(),
                                   p["c"], h0=p["h0"][b:b + 1, ds].cpu())
        assert rel_err(y[b:b + 1][:, :, ds].float().cpu(), yr) <= TOL["bf16"]
        assert rel_err(hf[b:b + 1, ds].cpu(), hr) <= TOL["bf16"]


# ---------------------------------------------------------------------------
# Selective SSM
# ---------------------------------------------------------------------------
def run_sel(lr, p, **over):
    g = cuda({**p, **over})
    y, hf = lr.selective_scan(g["x"], g["dt"], g["Bm"], g["Cm"], g["A_log"], z=g["z"],
                              Dskip=g["Dskip"], h0=g["h0"], dt_softplus=g["dt_softplus"])
    torch.cuda.synchronize()
    return y.float().cpu(), hf.cpu()


def check_sel(lr, p, io, **over):
    q = {**p, **over}
    y, hf = run_sel(lr, q)
    yr, hr = oracle.selective_scan(q["x"], q["dt"], q["Bm"], q["Cm"], q["A_log"], z=q["z"],
                                   Dskip=q["Dskip"], h0=q["h0"], dt_softplus=q["dt_softplus"])
    assert rel_err(y, yr) <= TOL[io], rel_err(y, yr)
    assert rel_err(hf, hr) <= TOL[io], rel_err(hf, hr)


def test_selective_f32_B2_L1024_D1536_full(lr):
    """B=2, L=1024, d_inner=1536 (4 scales of 384), N=16, fp32 I/O."""
    p = wl.make_inputs(wl.WORKLOADS["selective_f32"])
    check_sel(lr, p, "f32")


@pytest.mark.parametrize("B,L,D,io,h0", [
    (2, 1000, 256, "bf16", True),
    (3, 97, 40, "bf16", False),      # D not a multiple of the 32-channel block
    (1, 1, 32, "f32", True),
    (2, 45, 8, "f32", True),
    (1, 333, 4096, "bf16", True),    # the selective workload's channel width
])
def test_selective_oracle_sized(lr, B, L, D, io, h0):
    p = wl.selective_inputs(B, L, D, seed=B + L + D, io=io, with_h0=h0)
    check_sel(lr, p, io)


@pytest.mark.parametrize("variant", ["no_gate", "no_skip", "bare", "raw_dt"])
def test_selective_optional_inputs(lr, variant):
    p = wl.selective_inputs(2, 130, 64, seed=9, io="f32", with_h0=True)
    over = {"no_gate": dict(z=None), "no_skip": dict(Dskip=None),
            "bare": dict(z=None, Dskip=None, h0=None),
            "raw_dt": dict(dt=torch.nn.functional.softplus(p["dt"]), dt_softplus=False)}[variant]
    check_sel(lr, p, "f32", **over)


@pytest.mark.parametrize("warmup", [WARMUP_DEFAULT, 2048, 0])
@pytest.mark.parametrize("splits", [2, 3, 5])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selective_forced_time_splits(lr, splits, io, warmup):
    """Pieces that start inside a sequence.  With the warm-up (the default for
    bf16, forced by 2048 for fp32 too) each
    rebuilds its state over the preceding steps -- here all the way from the
    sequence start, since the slowest channels' horizon is longer than the
    sequence; with it disabled the carry comes by decoupled look-back and the
    outputs are corrected."""
    p = wl.selective_inputs(2, 650, 64, seed=20 + splits, io=io, with_h0=True)
    lr.lr_set_split_override(splits)
    lr.lr_set_selective_warmup(warmup)
    check_sel(lr, p, io)


@pytest.mark.parametrize("warmup", [2048, 0])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selective_warmup_stops_at_its_horizon(lr, io, warmup):
    """Pieces of 1500 steps over the four decay scales of a 64-channel
    chain: the warm-up windows end where the carry's contribution has decayed
    below the cut-off (a few hundred to about 1200 steps back), inside the
    preceding pieces, and the result still matches the oracle; the look-back
    path on the same input for comparison."""
    p = wl.selective_inputs(1, 6000, 64, seed=31, io=io, with_h0=True)
    lr.lr_set_split_override(4)
    lr.lr_set_selective_warmup(warmup)
    check_sel(lr, p, io)


@pytest.mark.parametrize("splits", [2, 3])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selective_work_stealing(lr, io, splits):
    """One 64-channel chain of 2048 tiles shared by 2 or 3 warps: the warp
    that starts at the sequence start needs no warm-up and finishes first, so
    it splits off the back half of another warp's unclaimed range (ranges of
    at least 64 tiles are split), warms up to its start and runs it.  Warm-ups
    are on for both dtypes, so the fp32 case runs at its 2^-32 cut-off.  The
    whole output and the final state match the oracle."""
    p = wl.selective_inputs(1, 16384, 64, seed=40 + splits, io=io, with_h0=True)
    # steps about 7x smaller than the workload's: the warm-up horizons (about
    # 280 tiles for bf16, 900 for fp32) make the shares that warm up finish
    # late enough that the first warp finds a remainder worth splitting
    p["dt"] = (p["dt"].float() - 2.0).to(p["dt"].dtype)
    lr.lr_set_split_override(splits)
    lr.lr_set_selective_warmup(1 << 20)   # no share falls back to look-back
    check_sel(lr, p, io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selective_deferred_shares(lr, io):
    """A warm-up limit of 64 steps: most pieces' windows are longer, so their
    shares are left to the second launch, which takes their carries by
    look-back and corrects their outputs, while the few that fit (the fastest
    channels' horizons, or pieces near the sequence start) warm up and can be
    split by idle warps -- both kinds in one call."""
    p = wl.selective_inputs(2, 3000, 128, seed=50, io=io, with_h0=True)
    lr.lr_set_split_override(6)
    lr.lr_set_selective_warmup(64)
    check_sel(lr, p, io)


def off_lattice(A_log, seed, channels=None, scale=0.05):
    """A_log moved off the multi-scale lattice A[n] = (n+1) A[0] (all channels,
    or only `channels`), so the kernel's warps holding them take the general
    one-exp-per-state decays."""
    g = torch.Generator().manual_seed(seed)
    noise = scale * torch.randn(A_log.shape, generator=g)
    if channels is not None:
        mask = torch.zeros(A_log.shape[0], 1)
        mask[channels] = 1.0
        noise = noise * mask
    return (A_log + noise).float()


@pytest.mark.parametrize("B,L,D,io", [
    (2, 1024, 128, "f32"),
    (2, 1000, 256, "bf16"),
    (1, 333, 4096, "bf16"),
])
def test_selective_general_decays_off_lattice(lr, B, L, D, io):
    """Trained-like A_log (off the initialisation lattice): general decays."""
    p = wl.selective_inputs(B, L, D, seed=B + L + D + 1, io=io, with_h0=True)
    check_sel(lr, p, io, A_log=off_lattice(p["A_log"], seed=D))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selective_lattice_and_general_warps_in_one_launch(lr, io):
    """Channel 5 (warp 0 of block 0) and 100 off the lattice, the rest on it:
    both decay forms run side by side and both match the oracle."""
    p = wl.selective_inputs(2, 640, 128, seed=41, io=io, with_h0=True)
    check_sel(lr, p, io, A_log=off_lattice(p["A_log"], seed=5, channels=[5, 100]))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selective_lattice_large_steps(lr, io):
    """Steps of delta ~ 5 (decays down to exp(-640) underflow to zero) on the
    lattice path."""
    p = wl.selective_inputs(2, 256, 64, seed=43, io=io, with_h0=True)
    dt = (p["dt"].float() + 6.5).to(p["dt"].dtype)
    check_sel(lr, p, io, dt=dt)


def test_selective_bf16_B4_L16384_D4096_sampled_and_four_segments(lr):
    """B=4, L=16384, d_inner=4096, N=16, bf16 I/O, h0 ~ N(0,1); also run as 4
    segments of 4096 carried through the final state.  The kernel cuts each
    launch's sequences into pieces of its own (a whole-GPU partition that
    depends on L), so the segmented run rounds differently from the single
    run: the two agree within the bf16 output tolerance, and the carried fp32
    state within the fp32 one."""
    cfg = wl.WORKLOADS["selective_bf16"]
    p = wl.make_inputs(cfg, device="cuda")
    args = (p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"])
    y, hf = lr.selective_scan(*args, z=p["z"], Dskip=p["Dskip"], h0=p["h0"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    for b in (0, cfg.B - 1):
        per = cfg.D // 4
        ds = np.concatenate([rng.choice(np.arange(s * per, (s + 1) * per), 6, replace=False)
                             for s in range(4)] + [np.array([0, cfg.D - 1])])
        ds = torch.from_numpy(np.sort(ds)).cuda()
        sub = {k: p[k][b:b + 1][:, :, ds].cpu() for k in ("x", "dt", "z")}
        yr, hr = oracle.selective_scan(sub["x"], sub["dt"], p["Bm"][b:b + 1].cpu(),
                                       p["Cm"][b:b + 1].cpu(), p["A_log"][ds].cpu(),
                                       z=sub["z"], Dskip=p["Dskip"][ds].cpu(),
                                       h0=p["h0"][b:b + 1, ds].cpu())
        assert rel_err(y[b:b + 1][:, :, ds].float().cpu(), yr) <= TOL["bf16"]
        assert rel_err(hf[b:b + 1, ds].cpu(), hr) <= TOL["bf16"]
    # four segments of 4096 steps, each resumed from the previous final state
    h = p["h0"]
    segs = []
    for k in range(4):
        sl = slice(k * 4096, (k + 1) * 4096)
        yk, h = lr.selective_scan(p["x"][:, sl], p["dt"][:, sl], p["Bm"][:, sl],
                                  p["Cm"][:, sl], p["A_log"], z=p["z"][:, sl],
                                  Dskip=p["Dskip"], h0=h)
        segs.append(yk)
    torch.cuda.synchronize()
    assert rel_err(torch.cat(segs, 1).float().cpu(), y.float().cpu()) <= TOL["bf16"]
    assert rel_err(h.cpu(), hf.cpu()) <= TOL["f32"]


def test_selective_bf16_B4_L16384_D4096_general_decays_sampled(lr):
    """The selective workload with A_log moved off the initialisation
    lattice: the general decays at full size, sampled channels."""
    cfg = wl.WORKLOADS["selective_bf16"]
    p = wl.make_inputs(cfg, device="cuda")
    A_log = off_lattice(p["A_log"].cpu(), seed=11).cuda()
    y, hf = lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], A_log, z=p["z"],
                              Dskip=p["Dskip"], h0=p["h0"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    b = 1
    ds = torch.from_numpy(np.sort(np.concatenate([rng.choice(cfg.D, 20, replace=False),
                                                  [0, cfg.D - 1]]))).cuda()
    sub = {k: p[k][b:b + 1][:, :, ds].cpu() for k in ("x", "dt", "z")}
    yr, hr = oracle.selective_scan(sub["x"], sub["dt"], p["Bm"][b:b + 1].cpu(),
                                   p["Cm"][b:b + 1].cpu(), A_log[ds].cpu(), z=sub["z"],
                                   Dskip=p["Dskip"][ds].cpu(), h0=p["h0"][b:b + 1, ds].cpu())
    assert rel_err(y[b:b + 1][:, :, ds].float().cpu(), yr) <= TOL["bf16"]
    assert rel_err(hf[b:b + 1, ds].cpu(), hr) <= TOL["bf16"]


def test_selective_zero_length_returns_initial_state(lr):
    p = cuda(wl.selective_inputs(1, 0, 32, seed=0, io="bf16", with_h0=True))
    y, hf = lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"], z=p["z"],
                              Dskip=p["Dskip"], h0=p["h0"])
    assert y.shape == (1, 0, 32) and torch.equal(hf, p["h0"])


# ---------------------------------------------------------------------------
# Boundary behaviour with real device tensors
# ---------------------------------------------------------------------------
def test_workspace_too_small_is_rejected(lr):
    p = cuda(wl.rglru_inputs(1, 640, 64, seed=1, io="bf16"))
    lr.lr_set_split_override(4)
    need = lr.lr_rglru_scan_workspace_size(1, 640, 64, 1)
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lr.LrError) as e:
        lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], 8.0, workspace=ws)
    assert e.value.code == lr.LR_ERR_WORKSPACE


def test_bounded_lookback_wait_reports_timeout_and_recovers(lr):
    """A split that never publishes its carry: the successors' waits run out
    after ~50 ms, the kernel finishes, and the status says LR_ERR_TIMEOUT."""
    p = wl.rglru_inputs(1, 512, 64, seed=3, io="f32", with_h0=True)
    lr.lr_set_split_override(4)
    lr.lr_set_selective_warmup(0)   # selective pieces below take their carry by look-back
    lr.lr_test_withhold_split(1, 50)
    run_rglru(lr, p)
    assert lr.status() == lr.LR_ERR_TIMEOUT
    assert lr.status() == 0  # read-and-clear
    lr.lr_test_withhold_split(-1, 1000)
    check_rglru(lr, p, "f32")
    # same for the selective scan
    q = wl.selective_inputs(1, 400, 32, seed=4, io="f32", with_h0=True)
    lr.lr_test_withhold_split(2, 50)
    run_sel(lr, q)
    assert lr.status() == lr.LR_ERR_TIMEOUT
    lr.lr_test_withhold_split(-1, 1000)
    check_sel(lr, q, "f32")
