"""The benchmark's reference arm runs on the CPU and prints the contract's
JSON line: the same metric, unit and config as the GPU arm, its own
cpu_baseline and e2e objects, and nothing else on stdout."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == bench.DEFAULT_WORKLOAD
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_kernel_table_counts_the_backward_as_five_gemms_and_prefers_the_phase_time():
    import bench
    w = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    n_exec = 2080
    gemm = n_exec * w.B * w.Hq * 2 * 128 * 128 * w.D  # one 128x128xD GEMM per executed block and q head
    pk = {"bf16_tflops": 1000.0}
    ms = {"fwd": 0.4, "rowsum": 0.02, "dkv": 0.7, "dq": 0.5, "bwd_phase": 1.2}
    t = bench.kernel_table(w, n_exec, ms, pk, 2000.0, 152)
    # forward: 2 GEMMs; dK/dV and dQ credited 5/7 of the 4 and 3 they execute
    assert abs(t["fwd"]["tflops_alg"] - round(2 * gemm / 0.4e-3 / 1e12, 1)) < 0.11
    assert abs(t["dkv"]["tflops_alg"] - round(4 * gemm * 5 / 7 / 0.7e-3 / 1e12, 1)) < 0.11
    assert abs(t["dkv"]["tflops_executed"] - round(4 * gemm / 0.7e-3 / 1e12, 1)) < 0.11
    assert abs(t["dq"]["tflops_alg"] - round(3 * gemm * 5 / 7 / 0.5e-3 / 1e12, 1)) < 0.11
    # the backward: 5 GEMMs over the phase time, the sum of kernels beside it
    assert t["bwd"]["ms"] == 1.2 and abs(t["bwd"]["tflops_alg"] - round(5 * gemm / 1.2e-3 / 1e12, 1)) < 0.11
    assert t["bwd"]["sum_of_kernels_ms"] == 1.22
    assert abs(t["bwd"]["frac_alg"] - 5 * gemm / 1.2e-3 / 1e12 / 1000.0) < 1e-4
    # cycles per block at the given clock, tensor cycles per block for D = 128
    assert t["fwd"]["tensor_cycles_per_block"] == 1024 and t["dkv"]["tensor_cycles_per_block"] == 2048
    assert abs(t["fwd"]["sm_cycles_per_block"] - 0.4e-3 * 2000e6 * 152 / (n_exec * w.B * w.Hq)) < 0.11
    # without the phase time the backward falls back to the sum of kernels
    del ms["bwd_phase"]
    assert bench.kernel_table(w, n_exec, ms, pk, 2000.0, 152)["bwd"]["ms"] == 1.22
