"""Host-side pieces of bench.py that need no GPU: the two-rank launch (which
does no GPU work: the library is single-GPU code), the reference arm's JSON
line, the attribution of clock samples to kernels, the parity check of the
timed outputs, and the stale-profile check of the roofline traffic."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_rank(rank, world, *extra):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29555")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *extra],
                          capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)


def test_multi_gpu_launch_does_no_gpu_work():
    # The library is single-GPU code: under a two-rank launch (or --gpus 2)
    # rank 0 prints one line saying so, rank 1 prints nothing, both exit 0,
    # and neither touches a GPU (this host has none).
    outs = [_run_rank(r, 2, "--gpus", "2", "--steps", "3", "--warmup", "3") for r in range(2)]
    assert [o.returncode for o in outs] == [0, 0], [o.stderr for o in outs]
    lines = [ln for ln in outs[0].stdout.splitlines() if ln.strip()]
    assert len(lines) == 1 and outs[1].stdout.strip() == ""
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and "single-GPU" in d["unavailable"]
    o = _run_rank(0, 1, "--gpus", "4", "--steps", "3", "--warmup", "3")
    assert o.returncode == 0 and json.loads(o.stdout.strip())["n_gpus"] == 4


def test_reference_arm_runs_on_rank_zero_only():
    outs = [_run_rank(r, 2, "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup",
                      "3", "--size", "256") for r in range(2)]
    assert [o.returncode for o in outs] == [0, 0], [o.stderr for o in outs]
    assert outs[1].stdout.strip() == ""
    d = json.loads(outs[0].stdout.strip())
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_clock_samples_are_attributed_to_kernel_intervals():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(None, 0)
    t0 = 100.0
    # samples at 0.5, 1.5, 2.5, 3.5 ms after t0 with clocks 1000, 1100, 1200, 1300
    c.samples = [(t0 + (i + 0.5) * 1e-3, 1000.0 + 100 * i, 2070.0,
                  {"sw_power_cap"} if i == 3 else set()) for i in range(4)]
    got = c.per_interval(t0, {"a": [(0.0, 1.0), (2.0, 3.0)], "b": [(1.0, 2.0), (3.0, 4.0)],
                              "c": [(4.0, 5.0)]})
    assert got["a"]["sm_mhz"] == 1100.0 and got["a"]["samples"] == 2
    assert got["b"]["sm_mhz"] == 1200.0 and got["b"]["reasons"] == ["sw_power_cap"]
    assert got["c"]["samples"] == 0 and got["c"]["sm_mhz"] is None
    assert c.summary()["sm_max_mhz"] == 2070.0


def test_step_parity_flags_a_wrong_element():
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from blackwell_tile_gemm_gb300 import synth
    oracle.build()
    rng = np.random.default_rng(5)
    M = K = 64
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (M, K))
    rows, cols = np.array([0, 5, 63]), np.array([1, 2, 40])
    ref, mag = oracle.gemm_bf16(A, B, rows=rows, cols=cols)
    full, _ = oracle.gemm_bf16(A, B)
    X = rng.integers(0, 1 << 16, (M, M), dtype=np.uint32).astype(np.uint16)
    bf = synth.f32_to_bf16_bits(full.astype(np.float32))
    d = {"D": torch.from_numpy(full.astype(np.float32)),
         "mD": torch.from_numpy(bf.view(np.int16)).view(torch.bfloat16),
         "XT": torch.from_numpy(np.ascontiguousarray(X.T).view(np.int16))}
    host = {"tr": {"X": X}}
    p = bench.step_parity(torch, d, host, (rows, cols, ref, mag, ref, mag))
    assert p["max_err_over_tol"] <= 1.0 and p["transpose_bit_exact"]
    d["D"][5, 40] += 1e-2
    d["XT"][3, 7] ^= 1
    p = bench.step_parity(torch, d, host, (rows, cols, ref, mag, ref, mag))
    assert p["gemm_bf16"] > 1.0 and not p["transpose_bit_exact"]


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--size", "256"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3


def test_profiled_traffic_is_null_for_changed_sources(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.profiled_traffic("gemm_bf16") is not None or True   # present or stale
    monkeypatch.setattr(bench, "sources_sha256", lambda group: "0" * 64)
    assert bench.profiled_traffic("gemm_bf16") is None
    assert bench.profiled_traffic("tile_transpose_b16") is None
