"""Exhaustive host checks of the arithmetic shortcuts of the CUDA
quantisers (see tests/kernel_identities.c): the division-free RN(x / 6) of
the block scale, and the integer form of the E2M1 stochastic-rounding
decision, each against the definition it replaces, over every finite FP32
input.  The GPU parity tests check the compiled kernels against the oracle;
these pin the two identities the kernels rely on for inputs no test tensor
reaches."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_div6_and_sr_integer_form_exhaustive(tmp_path):
    exe = tmp_path / "kernel_identities"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-o", str(exe),
                           os.path.join(HERE, "kernel_identities.c"), "-lm"])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=900, check=True).stdout
    res = dict(line.split() for line in out.strip().splitlines())
    assert res == {"div6": "0", "sr": "0"}, out
