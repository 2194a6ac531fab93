"""bench.py's JSON line contract, checked through the reference arm (the CPU oracle), which
runs without a GPU: one line on stdout with the keys the driver reads."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600, check=True).stdout
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1, out
    return json.loads(lines[0])


def test_reference_line_has_the_contract_keys():
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_workload_accounting():
    import bench
    assert bench.gemm_flops("mla") == 2.0 * 4096 * 2112 * 7168
    assert bench.gemm_flops("moe_chain") == 2.0 * 32768 * (4096 * 7168 + 7168 * 2048)
    assert abs(bench.quant_bytes("ffn") - (16384 * 7168 * (3 + 4 / 128) + 18432 * 7168 * (3 + 4 / 16384))) < 1
    assert bench.job_throughput(10.0, 2.0, 4) == 20.0
