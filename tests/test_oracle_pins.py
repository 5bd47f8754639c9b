"""Pins for the float64 oracle against facts that do not come from the oracle.

Each test checks one of: a closed form (a == 1 prefix sums, a == 0 identity,
constant-decay geometric series and its steady state), brute force on tiny
inputs (the unrolled product form of the recurrence), a library routine
(torch softplus / silu, numpy power, scipy matrix exponential for the ZOH
decay, dense numpy matmuls for the HGRN2 attention form), the page's example
shape, the page's multi-scale A values, and the split-sequence invariant
(running the sequence in segments that carry the final state equals one run).

These run on the CPU only.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from conftest import read_golden_constants, read_golden_table
from selective_state_space_chunked_gb300 import workloads

RTOL = 1e-11


def close(a, b, rtol=RTOL):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(1.0, float(np.max(np.abs(b))))
    assert np.max(np.abs(a - b)) <= rtol * scale, np.max(np.abs(a - b))


def rng(seed):
    return np.random.default_rng(seed)


def torch_softplus(v):
    return F.softplus(torch.from_numpy(np.asarray(v, np.float64))).numpy()


def torch_silu(v):
    return F.silu(torch.from_numpy(np.asarray(v, np.float64))).numpy()


# ----------------------------------------------------------------------------
# Selective SSM
# ----------------------------------------------------------------------------

def sel_random(seed, B=2, L=9, D=3, N=4):
    g = rng(seed)
    return dict(
        x=g.standard_normal((B, L, D)),
        dt=g.uniform(-4.0, 0.5, (B, L, D)),
        z=g.standard_normal((B, L, D)),
        Bm=g.standard_normal((B, L, N)),
        Cm=g.standard_normal((B, L, N)),
        A_log=g.uniform(-1.0, 2.0, (D, N)),
        Dskip=g.standard_normal(D),
        h0=g.standard_normal((B, D, N)),
    )


def test_selective_a_one_is_prefix_sum():
    """A_log = -inf gives A = 0, a = exp(0) = 1: h is h0 plus a running sum."""
    p = sel_random(1)
    p["A_log"][:] = -np.inf
    y, hf = oracle.selective_scan(**p, dt_softplus=True)
    delta = torch_softplus(p["dt"])                                  # (B,L,D)
    b = delta[..., None] * p["Bm"][:, :, None, :] * p["x"][..., None]  # (B,L,D,N)
    H = p["h0"][:, None] + np.cumsum(b, axis=1)
    yr = np.einsum("bldn,bln->bld", H, p["Cm"]) + p["Dskip"] * p["x"]
    yr = yr * torch_silu(p["z"])
    close(y, yr)
    close(hf, H[:, -1])


def test_selective_a_zero_is_identity():
    """A huge makes a = 0: h_t = delta_t B_t x_t and y_t uses only step t."""
    p = sel_random(2)
    p["A_log"][:] = 60.0
    y, hf = oracle.selective_scan(**p, dt_softplus=True)
    delta = torch_softplus(p["dt"])
    cb = np.einsum("bln,bln->bl", p["Cm"], p["Bm"])[..., None]
    yr = (delta * p["x"] * cb + p["Dskip"] * p["x"]) * torch_silu(p["z"])
    close(y, yr)
    close(hf, delta[:, -1, :, None] * p["Bm"][:, -1, None, :] * p["x"][:, -1, :, None])


def test_selective_constant_decay_geometric_series():
    """Constant delta and constant b: h_t = a^(t+1) h0 + b (1 - a^(t+1)) / (1 - a)."""
    g = rng(3)
    B, L, D, N = 1, 40, 2, 5
    delta = 0.07
    x = np.broadcast_to(g.standard_normal((1, 1, D)), (B, L, D)).copy()
    Bm = np.broadcast_to(g.standard_normal((1, 1, N)), (B, L, N)).copy()
    Cm = g.standard_normal((B, L, N))
    A_log = g.uniform(-1.0, 2.0, (D, N))
    h0 = g.standard_normal((B, D, N))
    y, hf = oracle.selective_scan(x, np.full((B, L, D), delta), Bm, Cm, A_log,
                                  h0=h0, dt_softplus=False)
    a = np.exp(-delta * np.exp(A_log))                                 # (D,N)
    bconst = delta * Bm[0, 0][None, :] * x[0, 0][:, None]              # (D,N)
    t1 = np.arange(1, L + 1)[:, None, None]                            # (L,1,1)
    H = a ** t1 * h0[0] + bconst * (1 - a ** t1) / (1 - a)             # (L,D,N)
    close(hf[0], H[-1])
    close(y[0], np.einsum("ldn,ln->ld", H, Cm[0]))


def test_selective_brute_force_unrolled_with_zoh_expm():
    """h_t = (prod_{u<=t} Abar_u) h0 + sum_s (prod_{s<u<=t} Abar_u) delta_s B_s x_s,
    with Abar_u = expm(delta_u * diag(A)) from scipy (the ZOH transition)."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    p = sel_random(4, B=1, L=7, D=2, N=3)
    y, hf = oracle.selective_scan(**p, dt_softplus=True)
    delta = torch_softplus(p["dt"])[0]                                 # (L,D)
    L, D = delta.shape
    N = p["A_log"].shape[1]
    for d in range(D):
        A = np.diag(-np.exp(p["A_log"][d]))
        Abar = [scipy_linalg.expm(delta[u, d] * A) for u in range(L)]
        for t in range(L):
            P0 = np.eye(N)
            for u in range(t + 1):
                P0 = Abar[u] @ P0
            h = P0 @ p["h0"][0, d]
            for s in range(t + 1):
                Ps = np.eye(N)
                for u in range(s + 1, t + 1):
                    Ps = Abar[u] @ Ps
                h = h + Ps @ (delta[s, d] * p["Bm"][0, s] * p["x"][0, s, d])
            yt = (p["Cm"][0, t] @ h + p["Dskip"][d] * p["x"][0, t, d])
            yt *= torch_silu(p["z"][0, t, d])
            close(y[0, t, d], yt)
            if t == L - 1:
                close(hf[0, d], h)


def test_selective_softplus_matches_torch_including_threshold():
    """With a = 1, h0 = 0, B = C = x = 1 and no gate/skip, y equals delta."""
    dts = np.array([-30.0, -1.0, 0.0, 1.0, 19.9, 20.0, 20.1, 40.0])
    L = dts.size
    ones_l = np.ones((1, L, 1))
    y, _ = oracle.selective_scan(ones_l, dts.reshape(1, L, 1), ones_l, ones_l,
                                 np.full((1, 1), -np.inf), dt_softplus=True)
    # y_t = sum of deltas so far (a == 1): difference to recover each delta
    d = np.diff(np.concatenate([[0.0], y[0, :, 0]]))
    close(d, torch_softplus(dts), rtol=1e-13)


def test_selective_optional_gate_and_skip():
    """z = None drops the silu gate, Dskip = None drops the skip."""
    p = sel_random(5)
    full, _ = oracle.selective_scan(**p)
    nogate, _ = oracle.selective_scan(**{**p, "z": None})
    bare, _ = oracle.selective_scan(**{**p, "z": None, "Dskip": None})
    close(full, nogate * torch_silu(p["z"]))
    close(nogate, bare + p["Dskip"] * p["x"])


def test_selective_zero_length_and_zero_h0():
    p = sel_random(6)
    p0 = {**p, "h0": None}
    y0, hf0 = oracle.selective_scan(**p0)
    yz, hfz = oracle.selective_scan(**{**p, "h0": np.zeros_like(p["h0"])})
    close(y0, yz)
    close(hf0, hfz)
    e = {k: (v[:, :0] if k in ("x", "dt", "z", "Bm", "Cm") else v) for k, v in p.items()}
    y, hf = oracle.selective_scan(**e)
    assert y.shape == (2, 0, 3)
    close(hf, p["h0"])


@pytest.mark.parametrize("segments", [2, 4])
def test_selective_split_resume_equals_full(segments):
    p = sel_random(7, B=2, L=24, D=3, N=4)
    y, hf = oracle.selective_scan(**p)
    ys, h = [], p["h0"]
    for part in np.array_split(np.arange(24), segments):
        sl = slice(part[0], part[-1] + 1)
        seg = {k: (v[:, sl] if k in ("x", "dt", "z", "Bm", "Cm") else v)
               for k, v in p.items()}
        seg["h0"] = h
        yk, h = oracle.selective_scan(**seg)
        ys.append(yk)
    close(np.concatenate(ys, axis=1), y, rtol=1e-13)
    close(h, hf, rtol=1e-13)


def test_multiscale_A_matches_page_values():
    want = np.array(read_golden_table("multiscale_A_d8_n16_s4.txt"))
    A_log = workloads.multiscale_A_log(8, 16, 4)
    np.testing.assert_array_equal(torch.exp(A_log.double()).round().numpy(), want)
    # float32 log of the exact integers, as the page stores the parameter
    np.testing.assert_array_equal(
        A_log.numpy(), torch.log(torch.tensor(want, dtype=torch.float32)).numpy())


def test_selective_workload_distributions():
    k = read_golden_constants()
    p = workloads.selective_inputs(2, 256, 64, seed=1)
    delta = F.softplus(p["dt"].double())
    # dt bias range [0.001, 0.1] before the N(0, 0.1) perturbation
    assert 0.0005 < float(delta.median()) < 0.05
    assert torch.all(p["Dskip"] == k["ssm_D_init"])
    assert p["A_log"].shape == (64, int(k["ssm_state_size"]))


# ----------------------------------------------------------------------------
# RG-LRU
# ----------------------------------------------------------------------------

def rg_random(seed, B=2, L=11, D=3):
    g = rng(seed)
    return dict(
        x=g.standard_normal((B, L, D)),
        r=1 / (1 + np.exp(-g.standard_normal((B, L, D)))),
        i=1 / (1 + np.exp(-g.standard_normal((B, L, D)))),
        a_log=np.log(g.uniform(0.9, 0.999, D)),
        h0=g.standard_normal((B, D)),
    )


def test_rglru_a_one_keeps_state():
    """r = 0 gives a_t = a^0 = 1 and sqrt(1 - 1) = 0: the state never moves."""
    p = rg_random(11)
    p["r"][:] = 0.0
    y, hf = oracle.rglru_scan(**p, c=8.0)
    close(y, np.broadcast_to(p["h0"][:, None, :], y.shape))
    close(hf, p["h0"])


def test_rglru_a_zero_is_gated_input():
    """Base a = 0 (a_log = -inf) with r > 0: a_t = 0, sqrt(1 - 0) = 1, h_t = i_t x_t."""
    p = rg_random(12)
    p["a_log"][:] = -np.inf
    y, hf = oracle.rglru_scan(**p, c=8.0)
    close(y, p["i"] * p["x"])
    close(hf, (p["i"] * p["x"])[:, -1])


def test_rglru_constant_gate_geometric_series_and_steady_state():
    """Constant r and u = i x: h_t = a^(t+1) h0 + sqrt(1-a^2) u (1-a^(t+1))/(1-a);
    it tends to sqrt((1+a)/(1-a)) u, the RG-LRU steady state."""
    g = rng(13)
    B, L, D = 1, 3000, 3
    c = 8.0
    base = g.uniform(0.9, 0.999, D)
    r = np.broadcast_to(g.uniform(0.2, 0.9, (1, 1, D)), (B, L, D)).copy()
    u = g.standard_normal(D)
    x = np.broadcast_to(u, (B, L, D)).copy()
    ig = np.ones((B, L, D))
    h0 = g.standard_normal((B, D))
    y, hf = oracle.rglru_scan(x, r, ig, np.log(base), c=c, h0=h0)
    a = np.power(base, c * r[0, 0])                   # the page's a ** (c r)
    t1 = np.arange(1, L + 1)[:, None]
    H = a ** t1 * h0[0] + np.sqrt(1 - a * a) * u * (1 - a ** t1) / (1 - a)
    close(y[0], H, rtol=1e-10)
    close(hf[0], np.sqrt((1 + a) / (1 - a)) * u, rtol=1e-6)


def test_rglru_brute_force_unrolled_page_form():
    """h_t = (prod a_u) h0 + sum_s (prod_{s<u<=t} a_u) sqrt(1 - a_s^2) i_s x_s with
    a_u = base ** (c r_u) (numpy power) and the page's sqrt(1 - a^2)."""
    p = rg_random(14, B=2, L=9, D=2)
    c = 8.0
    y, hf = oracle.rglru_scan(**p, c=c)
    base = np.exp(p["a_log"])
    a = np.power(base, c * p["r"])
    m = np.sqrt(1 - a * a) * p["i"] * p["x"]
    B, L, D = p["x"].shape
    for b in range(B):
        for d in range(D):
            for t in range(L):
                h = np.prod(a[b, : t + 1, d]) * p["h0"][b, d]
                for s in range(t + 1):
                    h += np.prod(a[b, s + 1: t + 1, d]) * m[b, s, d]
                close(y[b, t, d], h, rtol=1e-12)
    close(hf, y[:, -1])


def test_rglru_page_example_shape():
    k = read_golden_constants()
    B, L, D = int(k["rglru_example_B"]), int(k["rglru_example_L"]), int(k["rglru_example_D"])
    p = workloads.rglru_inputs(B, L, D, seed=0)
    y, hf = oracle.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], c=k["rglru_c"])
    assert y.shape == (B, L, D) and hf.shape == (B, D)
    assert np.all(np.isfinite(y))


def test_rglru_workload_constants():
    k = read_golden_constants()
    p = workloads.rglru_inputs(2, 16, 512, seed=0)
    a = torch.exp(p["a_log"].double())
    assert float(a.min()) >= k["rglru_a_lo"] - 1e-6
    assert float(a.max()) <= k["rglru_a_hi"] + 1e-6
    assert p["c"] == k["rglru_c"]
    assert float(p["r"].min()) > 0 and float(p["r"].max()) < 1


@pytest.mark.parametrize("segments", [2, 5])
def test_rglru_split_resume_equals_full(segments):
    p = rg_random(15, B=2, L=30, D=4)
    y, hf = oracle.rglru_scan(**p)
    ys, h = [], p["h0"]
    for part in np.array_split(np.arange(30), segments):
        sl = slice(part[0], part[-1] + 1)
        yk, h = oracle.rglru_scan(p["x"][:, sl], p["r"][:, sl], p["i"][:, sl],
                                  p["a_log"], h0=h)
        ys.append(yk)
    close(np.concatenate(ys, axis=1), y, rtol=1e-13)
    close(h, hf, rtol=1e-13)


def test_rglru_near_one_decay_has_no_cancellation():
    """a_t within 1e-9 of 1: sqrt(1 - a^2) must keep its leading digits (the
    float64 subtraction 1 - a*a would keep only ~7 of them)."""
    eps = -1e-9
    y, _ = oracle.rglru_scan(np.ones((1, 1, 1)), np.ones((1, 1, 1)),
                             np.ones((1, 1, 1)), np.array([eps]), c=1.0)
    close(y[0, 0, 0], math.sqrt(2e-9) * math.sqrt(1 - 0.5e-9), rtol=1e-12)


def test_bf16_inputs_widen_exactly():
    v = torch.tensor([1 + 2 ** -7, -3.0, 2 ** -20], dtype=torch.bfloat16)
    x = v.reshape(1, 3, 1)
    y, _ = oracle.rglru_scan(x, torch.zeros_like(x) + 1, torch.ones_like(x),
                             np.array([-np.inf]))
    np.testing.assert_array_equal(y[0, :, 0], np.array([1 + 2 ** -7, -3.0, 2 ** -20]))


# ----------------------------------------------------------------------------
# HGRN2
# ----------------------------------------------------------------------------

def hg_random(seed, B=2, L=8, H=2, dk=3, dv=4, S0=True):
    g = rng(seed)
    return dict(
        q=g.standard_normal((B, L, H * dk)),
        k=g.standard_normal((B, L, H * dk)),
        v=g.standard_normal((B, L, H * dv)),
        g=g.uniform(0.2, 1.0, (B, L, H * dv)),
        H=H,
        S0=g.standard_normal((B, H, dv, dk)) if S0 else None,
    )


def heads(a, H):
    B, L, HD = a.shape
    return a.reshape(B, L, H, HD // H).transpose(0, 2, 1, 3)    # (B,H,L,d)


def test_hgrn2_g_one_is_causal_linear_attention():
    p = hg_random(21)
    p["g"][:] = 1.0
    o, Sf = oracle.hgrn2(**p)
    Q, K, V = heads(p["q"], 2), heads(p["k"], 2), heads(p["v"], 2)
    P = np.tril(Q @ K.transpose(0, 1, 3, 2))                    # (B,H,L,L)
    Or = P @ V + Q @ p["S0"].transpose(0, 1, 3, 2)              # + S0 q_t
    close(heads(o, 2), Or)
    close(Sf, p["S0"] + V.transpose(0, 1, 3, 2) @ K)


def test_hgrn2_g_zero_is_single_outer_product():
    p = hg_random(22)
    p["g"][:] = 0.0
    o, Sf = oracle.hgrn2(**p)
    Q, K, V = heads(p["q"], 2), heads(p["k"], 2), heads(p["v"], 2)
    qk = np.sum(Q * K, axis=-1, keepdims=True)
    close(heads(o, 2), V * qk)
    close(Sf, V[:, :, -1, :, None] * K[:, :, -1, None, :])


def test_hgrn2_constant_gate_is_decay_masked_attention():
    """g_t[i] = gamma_i: o_t[i] = gamma_i^(t+1) (S0 q_t)[i]
    + sum_{s<=t} gamma_i^(t-s) (q_t . k_s) v_s[i]  (decay on the value row)."""
    g = rng(23)
    p = hg_random(23, B=1, L=10, H=1, dk=3, dv=4)
    gamma = g.uniform(0.3, 0.95, 4)
    p["g"] = np.broadcast_to(gamma, p["g"].shape).copy()
    o, Sf = oracle.hgrn2(**p)
    Q, K, V = p["q"][0], p["k"][0], p["v"][0]
    L = Q.shape[0]
    tt, ss = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
    P = np.tril(Q @ K.T)
    S0 = p["S0"][0, 0]
    for i in range(4):
        G = np.where(tt >= ss, gamma[i] ** np.maximum(tt - ss, 0), 0.0)
        oi = (P * G) @ V[:, i] + gamma[i] ** (np.arange(L) + 1) * (Q @ S0[i])
        close(o[0, :, i], oi)
    close(Sf[0, 0], (gamma[:, None] ** L) * S0
          + ((gamma[:, None] ** (L - 1 - np.arange(L))[None, :]) * V.T) @ K)


def test_hgrn2_brute_force_unrolled():
    p = hg_random(24, B=1, L=6, H=2, dk=2, dv=3)
    o, Sf = oracle.hgrn2(**p)
    B, L, _ = p["q"].shape
    for h in range(2):
        Q = p["q"][0, :, h * 2:(h + 1) * 2]
        K = p["k"][0, :, h * 2:(h + 1) * 2]
        V = p["v"][0, :, h * 3:(h + 1) * 3]
        G = p["g"][0, :, h * 3:(h + 1) * 3]
        for t in range(L):
            S = np.diag(np.prod(G[: t + 1], axis=0)) @ p["S0"][0, h]
            for s in range(t + 1):
                S += np.diag(np.prod(G[s + 1: t + 1], axis=0)) @ np.outer(V[s], K[s])
            close(o[0, t, h * 3:(h + 1) * 3], S @ Q[t])
            if t == L - 1:
                close(Sf[0, h], S)


@pytest.mark.parametrize("segments", [2, 3])
def test_hgrn2_split_resume_equals_full(segments):
    p = hg_random(25, B=2, L=12, H=2, dk=3, dv=3)
    o, Sf = oracle.hgrn2(**p)
    os_, S = [], p["S0"]
    for part in np.array_split(np.arange(12), segments):
        sl = slice(part[0], part[-1] + 1)
        ok, S = oracle.hgrn2(p["q"][:, sl], p["k"][:, sl], p["v"][:, sl],
                             p["g"][:, sl], 2, S0=S)
        os_.append(ok)
    close(np.concatenate(os_, axis=1), o, rtol=1e-13)
    close(S, Sf, rtol=1e-13)


def test_hgrn2_workload_gate_bounds():
    p = workloads.hgrn2_inputs(1, 64, 2, 128, seed=4)
    gv = p["g"].float()
    assert float(gv.min()) >= 0.2 - 1e-3 and float(gv.max()) <= 1.0
    assert p["q"].dtype == torch.bfloat16


# ------------------------------------------------------------------ MinMax
# [MINMAX] minmaxrnc minmax_neuron.py (MinMaxNeuron: x_{t+1} = max(min(r_t,
# x_t), s_t), forward returns every state) and minmax_operator.py (apply,
# compose).
def minmax_inputs(B, L, D, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    r = torch.randn(B, L, D, generator=g).to(dtype)
    s = torch.randn(B, L, D, generator=g).to(dtype) - 1.0
    x0 = torch.randn(B, D, generator=g).to(dtype).float()
    return r, s, x0


def test_minmax_identity_operators_keep_the_state():
    """a = +inf, b = -inf is the identity operator of minmax_operator.apply."""
    B, L, D = 2, 9, 5
    _, _, x0 = minmax_inputs(B, L, D, 1)
    r = np.full((B, L, D), np.inf)
    s = np.full((B, L, D), -np.inf)
    y, xf = oracle.minmax_scan(r, s, x0)
    assert np.array_equal(y, np.broadcast_to(x0.numpy()[:, None, :], (B, L, D)))
    assert np.array_equal(xf, x0.numpy())


def test_minmax_without_upper_bound_is_a_running_max():
    """r = +inf: x_t = max(x_{t-1}, s_t), numpy's running maximum."""
    B, L, D = 3, 40, 7
    _, s, x0 = minmax_inputs(B, L, D, 2)
    y, xf = oracle.minmax_scan(np.full((B, L, D), np.inf), s, x0)
    seq = np.concatenate([x0.numpy()[:, None, :], s.numpy().astype(np.float64)], axis=1)
    ref = np.maximum.accumulate(seq, axis=1)[:, 1:, :]
    assert np.array_equal(y, ref) and np.array_equal(xf, ref[:, -1])


def test_minmax_without_lower_bound_is_a_running_min():
    """s = -inf: x_t = min(r_t, x_{t-1}), numpy's running minimum."""
    B, L, D = 3, 40, 7
    r, _, x0 = minmax_inputs(B, L, D, 3)
    y, _ = oracle.minmax_scan(r, np.full((B, L, D), -np.inf), x0)
    seq = np.concatenate([x0.numpy()[:, None, :], r.numpy().astype(np.float64)], axis=1)
    assert np.array_equal(y, np.minimum.accumulate(seq, axis=1)[:, 1:, :])


def _compose(a2, b2, a1, b1):
    # minmax_operator.compose: f2(f1(x)) = max(min(min(a2, a1), x), max(min(a2, b1), b2))
    return np.minimum(a2, a1), np.maximum(np.minimum(a2, b1), b2)


def test_minmax_states_equal_the_composed_operator_applied_to_x0():
    """Every state equals the page's closed-form composition of the first t
    operators applied once to x0 (a different computation from the loop)."""
    B, L, D = 2, 33, 6
    r, s, x0 = minmax_inputs(B, L, D, 4)
    r64, s64, x64 = r.numpy().astype(np.float64), s.numpy().astype(np.float64), x0.numpy()
    y, _ = oracle.minmax_scan(r, s, x0)
    a = np.full((B, D), np.inf)
    b = np.full((B, D), -np.inf)
    for t in range(L):
        a, b = _compose(r64[:, t], s64[:, t], a, b)
        assert np.array_equal(y[:, t], np.maximum(np.minimum(a, x64), b))


def test_minmax_outputs_are_inputs_and_respect_the_bounds():
    B, L, D = 2, 50, 8
    r, s, x0 = minmax_inputs(B, L, D, 5, torch.bfloat16)
    y, _ = oracle.minmax_scan(r, s, x0)
    r64, s64 = r.double().numpy(), s.double().numpy()
    assert np.all(y >= s64) and np.all(y <= np.maximum(r64, s64))
    pool = np.concatenate([x0.double().numpy()[:, None, :], r64, s64], axis=1)
    for b_ in range(B):
        for d in range(D):
            assert set(y[b_, :, d]).issubset(set(pool[b_, :, d]))


@pytest.mark.parametrize("segments", [2, 5])
def test_minmax_split_resume_equals_full(segments):
    B, L, D = 2, 60, 4
    r, s, x0 = minmax_inputs(B, L, D, 6)
    y, xf = oracle.minmax_scan(r, s, x0)
    x = x0
    ys = []
    for seg in np.array_split(np.arange(L), segments):
        yy, x = oracle.minmax_scan(r[:, seg], s[:, seg], x)
        ys.append(yy)
    assert np.array_equal(np.concatenate(ys, 1), y) and np.array_equal(x, xf)


def test_minmax_zero_length_and_default_state():
    r, s, _ = minmax_inputs(1, 0, 3, 7)
    y, xf = oracle.minmax_scan(r, s)
    assert y.shape == (1, 0, 3) and np.array_equal(xf, np.zeros((1, 3)))


def test_minmax_nan_propagates_like_the_page_operator():
    """minmax_operator.apply uses torch.minimum / torch.maximum, which return
    NaN when either argument is NaN: a NaN input poisons every later state."""
    B, L, D = 1, 12, 4
    r, s, x0 = minmax_inputs(B, L, D, 8)
    r[0, 3, 1] = float("nan")
    s[0, 7, 2] = float("nan")
    y, xf = oracle.minmax_scan(r, s, x0)
    x = x0.double()
    ref = []
    for t in range(L):
        x = torch.maximum(torch.minimum(r[:, t].double(), x), s[:, t].double())
        ref.append(x)
    ref = torch.stack(ref, 1).numpy()
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    assert np.array_equal(y[~np.isnan(y)], ref[~np.isnan(ref)])
    assert np.isnan(y[0, 3:, 1]).all() and np.isnan(y[0, 7:, 2]).all()
