"""Host-side check of the selective kernel's decay-form condition.

The selective kernel takes the powers form of the decays only where every
state of every channel of a warp satisfies |A[n] - (n+1) A[0]| <= 2^-20 |A[n]|
with A = -exp(A_log) log2(e) in fp32 (the multi-scale initialisation of
cortexnet MultiScaleSSM.__init__ puts A_log there).  These tests evaluate the
same condition in numpy float32 on the workloads' A_log: it must hold with a
wide margin (so the benchmark's launch takes the form it reports, even when
the device's exp differs from numpy's by an ulp or two), and A_log moved off
the lattice as the GPU tests move it must fail it.
"""
import numpy as np
import pytest
import torch

from selective_state_space_chunked_gb300 import workloads as wl

TOL = 2.0 ** -20


def lattice_deviation(A_log: torch.Tensor) -> np.ndarray:
    """Per channel, max over n of |A2[n] - (n+1) A2[0]| / |A2[n]| in float32."""
    a = A_log.numpy().astype(np.float32)
    A2 = (-np.exp(a.astype(np.float64)).astype(np.float32)) * np.float32(np.log2(np.e))
    k = np.arange(1, a.shape[1] + 1, dtype=np.float32)
    return (np.abs(A2 - k * A2[:, :1]) / np.abs(A2)).max(axis=1)


@pytest.mark.parametrize("name", ["selective_f32", "selective_bf16"])
def test_workload_A_log_is_on_the_lattice_with_margin(name):
    cfg = wl.WORKLOADS[name]
    dev = lattice_deviation(wl.multiscale_A_log(cfg.D, cfg.N, cfg.n_scales))
    assert dev.max() <= 0.4 * TOL, dev.max() / TOL


def test_perturbed_A_log_is_off_the_lattice():
    A_log = wl.multiscale_A_log(256, 16)
    g = torch.Generator().manual_seed(3)
    moved = A_log + 0.05 * torch.randn(A_log.shape, generator=g)
    assert (lattice_deviation(moved) > 100 * TOL).all()
