"""Host-side logic of bench.py (no GPU): the roofline objects, the choice of
peak, the DRAM-traffic lookup keyed by the CUDA sources' hash, the sizing of
the bounded oracle sample, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

import bench

PK = {"hbm": 6000.0, "bf16": 1500.0, "bf16_sus": 1000.0, "src": "measured"}


def test_tensor_roofline_burst_and_sustained():
    r = bench.tensor_roofline("gemm_kernel<x>", 1.5e12, 1.0, PK, "no_such_workload")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1500.0)
    assert r["peak"] == pytest.approx(3000.0) and r["peak_kind"] == "burst"
    assert r["frac"] == pytest.approx(0.5)
    s = bench.tensor_roofline("gemm_kernel<x>", 1.5e12, 1.0, PK, "no_such_workload", sustained=True)
    assert s["peak"] == pytest.approx(2000.0) and s["peak_kind"] == "sustained"
    assert s["frac"] == pytest.approx(0.75)
    assert s["frac_vs_burst"] == pytest.approx(0.5) and s["frac_vs_sustained"] == pytest.approx(0.75)
    assert r["traffic"] is None  # no capture recorded for this workload


def test_hbm_roofline():
    r = bench.hbm_roofline("quant_rc_kernel<x>", 3.0e9, 1.0, PK, "no_such_workload")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(3000.0) and r["peak"] == 6000.0 and r["frac"] == pytest.approx(0.5)


def test_recorded_traffic_follows_the_sources_hash():
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    sha = bench.kernel_sha()
    entries = []
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(t.split("=", 1) for t in line.split())
        entries.append(kv)
    assert entries, "profiles/traffic.txt lists no capture"
    for kv in entries:
        got = bench.recorded_traffic(kv["kernel"], kv["workload"])
        if kv["sources"] == sha:
            assert got == float(kv["dram_bytes_per_launch"])
        else:
            assert got is None
    assert bench.recorded_traffic("no_such_kernel", "fprop_4096x18432x7168") is None


def test_oracle_sample_scaling_stays_in_bounds():
    M, N = bench.FPROP["M"], bench.FPROP["N"]
    for R, C, f in [(128, 128, 4.0), (128, 128, 1000.0), (M, 128, 3.0), (M, 1024, 0.25), (1, 128, 0.01),
                    (M, N, 50.0)]:
        R2, C2 = bench._scale_sample(R, C, f)
        assert 1 <= R2 <= M and 128 <= C2 <= N and C2 % 128 == 0
        if R2 < M:
            assert C2 == 128 or C2 == C  # rows grow first
    # the work scales by about the factor when nothing saturates
    R2, C2 = bench._scale_sample(128, 128, 8.0)
    assert R2 * C2 == pytest.approx(128 * 128 * 8.0, rel=0.02)


def test_replica_value():
    assert bench.replica_value(2, 1.0e12, 10, 10.0) == pytest.approx(2000.0)


def test_reference_arm_prints_the_contract_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                          "--ref-budget", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "config", "cpu_baseline", "e2e"):
        assert key in d
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith(bench.FPROP_WORKLOAD)
    # the same workload dict as the GPU arm's line
    assert d["config"] == bench.fprop_config(1)


def test_summary_is_compact_and_last():
    r = bench.tensor_roofline("gemm_kernel<x>", 1.5e12, 1.0, PK, "no_such_workload")
    q = bench.hbm_roofline("quant_rc_kernel<x>", 3.0e9, 1.0, PK, "no_such_workload")
    out = {"value": 1.0, "roofline": r, "step_kernels": {"quant_x_rows_4096x7168": q},
           "breakdown": {"act_quant_16384x7168": {"roofline": q},
                         "wgrad_2048x7168x8192": {"roofline": r, "quant_cols_dY_8192x2048": q,
                                                  "quant_cols_X_8192x7168": q}},
           "clocks": {"sm_mhz": 2032.0}}
    out["summary"] = bench.summary(out)
    line = json.dumps(out)
    tail = line[-1500:]
    # every kernel's fraction sits inside the last 1500 characters
    for key in ("fprop_gemm", "quant_x_rows_4096x7168", "quant_act_rows_cols_16384x7168", "wgrad_gemm",
                "quant_cols_dY", "quant_cols_X"):
        assert '"%s"' % key in tail
    assert list(out)[-1] == "summary"


def test_kernel_hash_ignores_comments_only():
    import bench
    a = bench._strip_comments('int a = 1;  // note\n/* block\n comment */\nconst char* s = "x // y";\n')
    b = bench._strip_comments('int a = 1;\nconst char* s = "x // y";  /* other */\n')
    c = bench._strip_comments('int a = 2;\nconst char* s = "x // y";\n')
    assert a == b
    assert a != c
    assert '"x // y"' in a
