"""The dynamic quantiser computes each code without a division: y0 = x * (1/s), one correction
y = y0 + (x - y0 s) / s with fused multiply-adds, then rint.  It relies on this: over every (absmax, x)
pair it can meet whose scale s = amax / 127 is at least 2^-120, rint(y) equals rint of the correctly
rounded quotient x / s.  This test compiles a plain C sweep of all 531 million such pairs and runs it on
the host: every step is an IEEE binary32 operation rounded to nearest, as on the GPU.  The plain product
y0 must miss some codes (the check has teeth); the corrected quotient must miss none.  (No GPU.)"""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_corrected_quotient_gives_every_code_over_the_whole_domain():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "sweep")
        src = os.path.join(HERE, "native", "quant_method_sweep.c")
        subprocess.run([cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-o", exe, src, "-lm"],
                       check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=600).stdout.split()
    pairs, miss_plain, miss_corrected = (int(v) for v in out)
    assert pairs == 531098175
    assert miss_plain > 0
    assert miss_corrected == 0
