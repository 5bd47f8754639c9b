"""Host-side logic of bench.py's N > 1 path on CPU: two gloo ranks, the
max-over-ranks timing, the barrier and the whole-job (weak scaling) rate;
the reference arm prints on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    # rank r "took" 10 + 5 r ms; every rank must see the slowest
    slowest = bench.max_over_ranks(10.0 + 5.0 * r, w, torch.device("cpu"))
    rate = bench.job_throughput(w, units_per_rank_step=1000, steps=4, max_ms=slowest)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"slowest": slowest, "rate": rate}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for d in res:
        assert d["slowest"] == 15.0
        # 2 ranks x 1000 units x 4 steps in 15 ms
        assert d["rate"] == pytest.approx(2 * 1000 * 4 / 15e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    bench.barrier(1)
    assert bench.job_throughput(1, 10, 2, 1.0) == pytest.approx(20 / 1e-3)


def test_reference_arm_prints_on_rank0_only():
    """Under torchrun with two ranks the reference arm prints one JSON line
    (rank 0) and the other rank exits 0 without work (HGRN2 sample only, one
    step, to keep the run short)."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--only", "hgrn2", "--seq-len", "64"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # ms_per_step is the measured time of the sampled step; the whole
    # workload's time is labelled as extrapolated
    assert d["ms_per_step"] == pytest.approx(d["cpu_baseline"]["sample_ms"], rel=1.0)
    assert d["ms_per_step_kind"].startswith("measured")
    assert d["full_workload_ms_per_step_extrapolated"] >= d["ms_per_step"]


def test_roofline_entries_lead_with_hbm():
    """Every scan's roofline entry is its HBM fraction; the selective scan's
    also carries the ALU fraction against a peak derived from the SM count
    and clock it is given, HGRN2's the tensor fraction."""
    sys.path.insert(0, ROOT)
    import bench
    from selective_state_space_chunked_gb300 import workloads as wl
    peaks = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0,
             "source": "test"}
    alu = bench.alu_peak(100, 2000.0)
    assert alu[0] == pytest.approx(100 * 2000e6 * 32 / 1e9)
    assert "100 SMs" in alu[1]
    assert bench.alu_peak(152, None)[0] == pytest.approx(152 * 2070e6 * 32 / 1e9)
    sel = wl.WORKLOADS["selective_bf16"]
    a = bench.algorithmic(sel)
    e = bench.kernel_roofline(sel, a, 1.0, peaks, alu)
    assert e["bound"] == "hbm" and e["frac"] == pytest.approx(a["bytes"] / 1e-3 / 1e9 / 8000.0)
    assert e["alu"]["frac"] == pytest.approx(a["units"] * sel.N / 1e-3 / 1e9 / alu[0])
    hg = wl.WORKLOADS["hgrn2_bf16"]
    e = bench.kernel_roofline(hg, bench.algorithmic(hg), 0.1, peaks, alu)
    assert e["bound"] == "hbm" and "alu" not in e
    assert e["tensor"]["frac"] == pytest.approx(bench.algorithmic(hg)["flops"] / 1e-4 / 1e12 / 1600.0)
