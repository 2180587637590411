"""The 8-bit cache write's division method, checked exhaustively on the CPU.

The quantiser divides each value x by its group's fp16 scale d as IEEE fp32
division rounds (the rule of the 8-bit cache: code = clamp(rint(x / d))), but
the kernel forms the quotient from one correctly rounded reciprocal per group
and a fused residual step instead of a division per value.  The C program
beside this test (``csrc/q8_division_check.c``) restates that method with
C's fmaf and compares it with IEEE division for every finite bf16 and fp16 x
and every fp16 d a group can produce with it; the codes, the quotients (above
2^-100) and the scale's own division must all agree.  CPU only: the GPU
tests compare the kernel itself with the oracle on every input bit pattern.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_reciprocal_and_residual_give_ieee_codes():
    if shutil.which("gcc") is None:
        pytest.skip("needs gcc")
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "q8_division_check")
    src = os.path.join(HERE, "csrc", "q8_division_check.c")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-o", exe, src, "-lm"],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    counts = dict(zip(*[iter(r.stdout.split())] * 2))           # "name value" pairs
    assert int(counts["pairs"]) > 2_500_000_000          # every reachable (x, d) pair
    assert counts["code_differences"] == "0", r.stdout
    assert counts["quotient_differences"] == "0", r.stdout
    assert counts["scale_differences"] == "0", r.stdout
    assert r.returncode == 0
