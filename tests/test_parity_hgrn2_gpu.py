"""Parity of the CUDA HGRN2 chunked tcgen05 kernel with the float64 oracle.

Metric: max|gpu - ref| / max|ref| on o and on the final state separately,
at most 1e-2 (bf16 I/O).  Oracle-sized cases cover several chunks, ragged
sequence ends, a carried initial state and several heads; the full-size
workload (B=4, L=4096, 16 heads of 128) runs in the benchmark's launch and is
checked on sampled heads (the oracle computes heads independently).
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import rel_err
from selective_state_space_chunked_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 1e-2


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


def run(lr, p, S0=None):
    q, k, v, g = (p[n].cuda() for n in ("q", "k", "v", "g"))
    o, Sf = lr.hgrn2(q, k, v, g, H=p["H"], S0=None if S0 is None else S0.cuda())
    torch.cuda.synchronize()
    assert lr.status() == 0
    return o.float().cpu(), Sf.cpu()


def check(lr, p, S0=None):
    o, Sf = run(lr, p, S0)
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], p["H"], S0=S0)
    assert rel_err(o, orf) <= TOL, rel_err(o, orf)
    assert rel_err(Sf, Srf) <= TOL, rel_err(Sf, Srf)


@pytest.mark.parametrize("B,L,H", [(1, 256, 2), (2, 130, 1), (1, 64, 3), (1, 1, 1), (1, 63, 2),
                                   (1, 1000, 2)])
def test_hgrn2_oracle_sized(lr, B, L, H):
    p = wl.hgrn2_inputs(B, L, H, 128, seed=B * 100 + L + H)
    check(lr, p)


def test_hgrn2_initial_state(lr):
    p = wl.hgrn2_inputs(2, 200, 2, 128, seed=7, with_S0=True)
    check(lr, p, S0=0.1 * p["S0"])


def test_hgrn2_slow_and_fast_gates(lr):
    """Gates near 1 (long memory) and near the 0.2 lower bound in one run."""
    p = wl.hgrn2_inputs(1, 320, 2, 128, seed=8)
    g = p["g"].float()
    g[..., :128] = 0.999
    g[..., 128:] = 0.2
    p["g"] = g.to(torch.bfloat16)
    check(lr, p)


def test_hgrn2_split_resume(lr):
    p = {k: (v.cuda() if torch.is_tensor(v) else v)
         for k, v in wl.hgrn2_inputs(1, 512, 2, 128, seed=9).items()}
    o, Sf = lr.hgrn2(p["q"], p["k"], p["v"], p["g"], H=2)
    o1, S1 = lr.hgrn2(p["q"][:, :192], p["k"][:, :192], p["v"][:, :192], p["g"][:, :192], H=2)
    o2, S2 = lr.hgrn2(p["q"][:, 192:], p["k"][:, 192:], p["v"][:, 192:], p["g"][:, 192:], H=2,
                      S0=S1)
    torch.cuda.synchronize()
    assert rel_err(torch.cat([o1, o2], 1).float().cpu(), o.float().cpu()) <= 1e-2
    assert rel_err(S2.cpu(), Sf.cpu()) <= 1e-2


def small_gates(p, kind, seed):
    """Gates whose log2 products over a 64-step chunk fall far below what one
    reference point per chunk can factor (the page's lower bound may be 0):
    the kernel splits such chunks into virtual chunks of 32, 16, .. steps."""
    g = torch.Generator().manual_seed(seed)
    shape = p["g"].shape
    if kind == "const_0.1":            # 64 log2(0.1) = -212 per chunk
        gt = torch.full(shape, 0.1)
    elif kind == "uniform_0_0.2":      # heavy tail towards 0
        gt = 0.2 * torch.rand(shape, generator=g)
    elif kind == "lb0_wide":           # lb = 0, f ~ N(0, 3): sigmoid(f) down to ~1e-5
        gt = torch.sigmoid(3.0 * torch.randn(shape, generator=g))
    elif kind == "mixed":              # per-channel mix of slow, fast and vanishing gates
        gt = torch.sigmoid(torch.randn(shape, generator=g) * 2.0 + 2.0)
        gt[..., 1::3] = 0.02
        gt[..., 2::7] = 0.0            # a reset every step
    else:
        raise ValueError(kind)
    p["g"] = gt.to(torch.bfloat16)
    return p


@pytest.mark.parametrize("kind", ["const_0.1", "uniform_0_0.2", "lb0_wide", "mixed"])
def test_hgrn2_small_gates_match_the_oracle(lr, kind):
    p = small_gates(wl.hgrn2_inputs(1, 448, 2, 128, seed=10, with_S0=True), kind, seed=11)
    check(lr, p, S0=0.1 * p["S0"])


def test_hgrn2_steep_chunk_in_one_block_only(lr):
    """One thread block (batch row 1, head 1, value channels 64..127) meets
    steep gates late in the sequence; the call's second launch redoes that
    block alone and every other block keeps its first-pass results.  The same
    workspace then serves a call with ordinary gates."""
    B, L, H = 2, 640, 3
    p = wl.hgrn2_inputs(B, L, H, 128, seed=14, with_S0=True)
    g = p["g"].float()
    g[1, 400:, 128 + 64:256] = 0.01
    p["g"] = g.to(torch.bfloat16)
    ws = torch.empty(lr.lr_hgrn2_workspace_size(B, L, H, 128, 128, lr.LR_BF16), dtype=torch.uint8,
                     device="cuda")
    assert ws.numel() == 256 + B * H * 2 * 8
    S0 = 0.1 * p["S0"]
    c = {n: p[n].cuda() for n in ("q", "k", "v", "g")}
    o, Sf = lr.hgrn2(c["q"], c["k"], c["v"], c["g"], H=H, S0=S0.cuda(), workspace=ws)
    assert lr.status(ws) == 0
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], H, S0=S0)
    assert rel_err(o.float().cpu(), orf) <= TOL and rel_err(Sf.cpu(), Srf) <= TOL
    q = wl.hgrn2_inputs(B, L, H, 128, seed=15)
    o2, S2 = lr.hgrn2(*(q[n].cuda() for n in ("q", "k", "v", "g")), H=H, workspace=ws)
    assert lr.status(ws) == 0
    orf, Srf = oracle.hgrn2(q["q"], q["k"], q["v"], q["g"], H)
    assert rel_err(o2.float().cpu(), orf) <= TOL and rel_err(S2.cpu(), Srf) <= TOL


@pytest.mark.parametrize("gq,split", [(0.177734375, False), (0.17578125, True)])
def test_hgrn2_gates_at_the_whole_chunk_limit(lr, gq, split):
    """Constant gates (exact in bf16) whose 16-step products sit just inside
    (2^-39.875: the chunk runs whole, its per-step factors span 2^+-79.75 and
    come from running products as small as 2^-39.875) and just outside
    (2^-40.13: the first pass marks every block, the second splits each chunk
    in two) the whole-chunk limit of 2^-40 per quarter, beside ordinary gates
    in the other head."""
    p = wl.hgrn2_inputs(1, 320, 2, 128, seed=16, with_S0=True)
    g = p["g"].float()
    g[..., :128] = gq
    p["g"] = g.to(torch.bfloat16)
    assert (16 * torch.log2(p["g"][..., :128].double()) < -40).all().item() == split
    check(lr, p, S0=0.1 * p["S0"])


def test_hgrn2_small_gates_preact_lower_bound_zero(lr):
    """The page's default configuration: lb = 0 on pre-activation gates."""
    p = wl.hgrn2_inputs(1, 320, 2, 128, seed=12)
    f = (3.0 * torch.randn(p["g"].shape, generator=torch.Generator().manual_seed(13))).to(torch.bfloat16)
    q, k, v = (p[n].cuda() for n in ("q", "k", "v"))
    o, Sf = lr.hgrn2(q, k, v, f.cuda(), H=2, gate_lb=0.0)
    torch.cuda.synchronize()
    assert lr.status() == 0
    gref = torch.sigmoid(f.double())
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], gref, 2)
    assert rel_err(o.float().cpu(), orf) <= TOL and rel_err(Sf.cpu(), Srf) <= TOL


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_hgrn2_gate_not_finite_is_reported(lr, bad):
    """A gate that is not a finite number sets LR_ERR_RANGE."""
    p = wl.hgrn2_inputs(1, 64, 1, 128, seed=10)
    g = p["g"].clone()
    g[0, 17, 5] = bad
    q, k, v = (p[n].cuda() for n in ("q", "k", "v"))
    lr.hgrn2(q, k, v, g.cuda(), H=1)
    assert lr.status() == lr.LR_ERR_RANGE
    assert lr.status() == 0


def test_hgrn2_bf16_B4_L4096_H16_sampled(lr):
    """B=4, L=4096, hidden 2048 = 16 heads x 128, bf16, g = 0.2 + 0.8 sigmoid(f)."""
    cfg = wl.WORKLOADS["hgrn2_bf16"]
    p = wl.make_inputs(cfg, device="cuda")
    o, Sf = lr.hgrn2(p["q"], p["k"], p["v"], p["g"], H=cfg.H)
    torch.cuda.synchronize()
    assert lr.status() == 0
    for b, h in ((0, 0), (3, 15), (1, 7)):
        sl = slice(h * 128, (h + 1) * 128)
        sub = {n: p[n][b:b + 1, :, sl].cpu() for n in ("q", "k", "v", "g")}
        orf, Srf = oracle.hgrn2(sub["q"], sub["k"], sub["v"], sub["g"], 1)
        assert rel_err(o[b:b + 1, :, sl].float().cpu(), orf) <= TOL
        assert rel_err(Sf[b:b + 1, h:h + 1].cpu(), Srf) <= TOL


# ---------------------------------------------------------------- general path
# fp32 I/O, head dims other than 128 x 128 and chunk lengths other than 64 run
# the step-by-step CUDA-core kernel; fp32 I/O meets the 1e-4 bar there.
def general_inputs(B, L, H, dk, dv, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    q, k = (torch.randn(B, L, H * dk, generator=g) / dk ** 0.5 for _ in range(2))
    v = torch.randn(B, L, H * dv, generator=g) / dv ** 0.5
    gate = 0.2 + 0.8 * torch.sigmoid(torch.randn(B, L, H * dv, generator=g) + 2)
    return {"q": q.to(dtype), "k": k.to(dtype), "v": v.to(dtype), "g": gate.to(dtype), "H": H}


@pytest.mark.parametrize("dtype,tol", [(torch.float32, 1e-4), (torch.bfloat16, 1e-2)])
@pytest.mark.parametrize("B,L,H,dk,dv", [(2, 200, 2, 128, 128), (1, 150, 3, 64, 32),
                                         (1, 97, 1, 40, 24), (1, 64, 2, 256, 128),
                                         (1, 33, 1, 300, 16), (1, 77, 2, 33, 7),
                                         (1, 50, 1, 16, 200), (2, 35, 1, 512, 40)])
def test_hgrn2_general_path_matches_oracle(lr, dtype, tol, B, L, H, dk, dv):
    if dtype == torch.bfloat16 and dk == dv == 128:
        pytest.skip("bf16 128 x 128 runs the tensor-core kernel (covered above)")
    p = general_inputs(B, L, H, dk, dv, seed=B + L + dk, dtype=dtype)
    S0 = 0.1 * torch.randn(B, H, dv, dk, generator=torch.Generator().manual_seed(L))
    o, Sf = lr.hgrn2(p["q"].cuda(), p["k"].cuda(), p["v"].cuda(), p["g"].cuda(), H=H, S0=S0.cuda())
    torch.cuda.synchronize()
    assert lr.status() == 0
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], H, S0=S0)
    assert rel_err(o.float().cpu(), orf) <= tol
    assert rel_err(Sf.cpu(), Srf) <= tol


def test_hgrn2_general_path_other_chunk_and_preact(lr):
    """128 x 128 bf16 with chunk != 64 takes the general kernel; with the gate
    given before its activation as well."""
    p = wl.hgrn2_inputs(1, 130, 2, 128, seed=40)
    o, Sf = lr.hgrn2(p["q"].cuda(), p["k"].cuda(), p["v"].cuda(), p["g"].cuda(), H=2, chunk=32)
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], 2)
    assert rel_err(o.float().cpu(), orf) <= TOL and rel_err(Sf.cpu(), Srf) <= TOL
    f = torch.randn(1, 130, 2 * 64, generator=torch.Generator().manual_seed(41)).add(2.0)
    q = torch.randn(1, 130, 2 * 64, generator=torch.Generator().manual_seed(42)) / 8
    k = torch.randn(1, 130, 2 * 64, generator=torch.Generator().manual_seed(43)) / 8
    v = torch.randn(1, 130, 2 * 64, generator=torch.Generator().manual_seed(44)) / 8
    o, Sf = lr.hgrn2(q.cuda(), k.cuda(), v.cuda(), f.cuda(), H=2, gate_lb=0.3)
    gate = 0.3 + 0.7 * torch.sigmoid(f.double())
    orf, Srf = oracle.hgrn2(q, k, v, gate, 2)
    assert rel_err(o.cpu(), orf) <= 1e-4 and rel_err(Sf.cpu(), Srf) <= 1e-4


def test_hgrn2_general_path_fast_decay_has_no_range_limit(lr):
    """Gates of 0.1 (the tensor-core path reports LR_ERR_RANGE) are fine on the
    step-by-step kernel."""
    p = general_inputs(1, 128, 1, 64, 64, seed=45, dtype=torch.float32)
    p["g"] = torch.full_like(p["g"], 0.1)
    o, Sf = lr.hgrn2(p["q"].cuda(), p["k"].cuda(), p["v"].cuda(), p["g"].cuda(), H=1)
    torch.cuda.synchronize()
    assert lr.status() == 0
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], 1)
    assert rel_err(o.cpu(), orf) <= 1e-4 and rel_err(Sf.cpu(), Srf) <= 1e-4



@pytest.mark.parametrize("dtype,tol", [(torch.float32, 1e-4), (torch.bfloat16, 1e-2)])
@pytest.mark.parametrize("B,L,H", [(2, 80, 64), (1, 70, 40)])
def test_hgrn2_general_path_wide_grids(lr, dtype, tol, B, L, H):
    """Enough heads that the general kernel gives each thread 32 key columns
    of two value rows (2 x 64 heads) or of one row (40 heads) instead of 16
    columns of one row."""
    dk = dv = 128
    if dtype == torch.bfloat16:
        dk = dv = 64 * 2 if H == 40 else 128
    p = general_inputs(B, L, H, dk, dv, seed=B * 7 + H, dtype=dtype)
    if dtype == torch.bfloat16:   # 128 x 128 bf16 is the tensor-core kernel's: use chunk 32
        o, Sf = lr.hgrn2(p["q"].cuda(), p["k"].cuda(), p["v"].cuda(), p["g"].cuda(), H=H, chunk=32)
    else:
        o, Sf = lr.hgrn2(p["q"].cuda(), p["k"].cuda(), p["v"].cuda(), p["g"].cuda(), H=H)
    torch.cuda.synchronize()
    assert lr.status() == 0
    orf, Srf = oracle.hgrn2(p["q"], p["k"], p["v"], p["g"], H)
    assert rel_err(o.float().cpu(), orf) <= tol
    assert rel_err(Sf.cpu(), Srf) <= tol
