"""Host-side check of the library's table-driven fp32 exp (csrc/ffexp.cuh),
which the draft-row log-sum-exp uses: relative error below 1e-11 against
long-double expl over [-72, 0], exact two-step argument reduction, and an
error-free two_sum.  Compiled with g++ (no GPU needed)."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not available")
def test_ffexp_host_accuracy():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "ffexp_check")
        subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-o", exe,
                        os.path.join(HERE, "native", "ffexp_host_check.cpp")], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
        assert r.returncode == 0, r.stdout + r.stderr
