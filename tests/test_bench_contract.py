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


def test_profile_links():
    """Every ncu summary bench.py links for a roofline's traffic exists and gives
    the source hash and a per-launch byte count in the form bench.py parses (a
    hash that no longer matches the source makes bench.py print null)."""
    sys.path.insert(0, ROOT)
    import bench
    for workload, (name, sources) in bench.GEMM_PROFILE.items():
        text = open(os.path.join(ROOT, "profiles", name)).read()
        fields = dict(l.split(":", 1) for l in text.splitlines()
                      if l.startswith(("kernel_source_sha256_16:", "traffic_bytes_per_launch:")))
        assert set(fields) == {"kernel_source_sha256_16", "traffic_bytes_per_launch"}, name
        assert int(fields["traffic_bytes_per_launch"].split()[0]) > 0
        assert "ncu " in text and "--clock-control none" in text, name
        assert len(fields["kernel_source_sha256_16"].split()[0]) == 16, name


def test_every_profile_gives_its_command():
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        text = open(os.path.join(ROOT, "profiles", name)).read()
        assert "python bench.py" in text and "ncu " in text and "--clock-control none" in text, name
