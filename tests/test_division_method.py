"""The quantiser kernels divide by the group scale with a reciprocal and one
Markstein correction step; this checks, on the CPU and exhaustively over
every fp16 scale, that the method gives the IEEE single-precision quotient
(r - z) / s that the quantiser is defined with (Quant VideoGen explainer,
Sommario tecnico sec. 2B: each stage quantises the residual with the group's
scale and zero-point)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def test_markstein_division_equals_ieee_division(tmp_path):
    exe = tmp_path / "division_check"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-o", str(exe),
                           os.path.join(HERE, "division_check.c"), "-lm"])
    out = subprocess.check_output([str(exe), "64", "200"], text=True).split()
    checked, mismatches = int(out[1]), int(out[3])
    assert checked > 70_000_000
    assert mismatches == 0
