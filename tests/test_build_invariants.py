"""Build-time invariants of the GEMM kernels, checked from the ptxas report
(CPU only).  Warpgroup 0 lowers its register limit and the promotion
warpgroups raise theirs (setmaxnreg); the raised limits are drawn from the
registers the CTA was launched with, so every instance must be compiled with
exactly the per-thread count the split assumes: 168 at 384 threads, 128 at
512 threads.  A smaller count would leave setmaxnreg.inc waiting forever."""
import re
import subprocess

from fp8_fine_grained_27_b300 import build

PAT = re.compile(r"Function properties for (_ZN5fp8bs4gemm11gemm_kernelILi(\d+)ELi(\d)ELb(\d)ELb(\d)E\S*)\n"
                 r"\s+\d+ bytes stack frame, \d+ bytes spill stores, \d+ bytes spill loads\n"
                 r"ptxas info\s+: Used (\d+) registers")


def test_gemm_launch_register_counts_match_setmaxnreg_split(tmp_path):
    out = tmp_path / "lib.so"
    r = subprocess.run([build.NVCC, *build.FLAGS, "-Xptxas=-v", "-o", str(out), build.SRC],
                       capture_output=True, text=True, check=True)
    found = PAT.findall(r.stderr + r.stdout)
    assert len(found) >= 10, "GEMM instances missing from the ptxas report"
    for name, bn, bmode, f32, grouped, regs in found:
        threads = 512 if int(bn) == 192 else 384
        expect = 128 if threads == 512 else 168
        assert int(regs) == expect, (name, regs, expect)
