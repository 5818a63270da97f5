"""The SwiGLU exp of the GPU kernels runs its steps on x clamped to [-104, 89] (NaN propagated) and
selects nothing afterwards.  The specification selects +inf above 89, +0 below -104 and NaN for NaN.  The
clamp alone gives the same bits because the steps overflow to +inf at x = 89 and round to +0 at x = -104.
This test compiles a plain C sweep on the host, every binary32 value in [-112, -100] and [84, 96] plus the
infinities, with the same binary32 steps, and checks the two forms agree everywhere.  (A NaN input gives
a NaN either way; the kernels' NaN comes out of the arithmetic.)  (No GPU.)"""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_clamp_alone_gives_the_specified_exp_outside_the_range():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "sweep")
        subprocess.run([cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                        os.path.join(HERE, "native", "exp_clamp_sweep.c"), "-lm"], check=True)
        n, differ, at89, at_m104 = subprocess.run([exe], check=True, capture_output=True, text=True,
                                                  timeout=300).stdout.split()
    assert int(n) > 3_000_000
    assert int(differ) == 0
    assert at89 == "7f800000"   # e^89 > FLT_MAX: +inf
    assert at_m104 == "00000000"  # e^-104 < 2^-150: +0
