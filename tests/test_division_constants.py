"""The kernels compute amax / 127 (the quantization scale) and A / 255 (the
UINT8 probability scale) as a product with RN(1/b) and one Markstein step
instead of a division.  This checks, on the CPU, that the method returns the
IEEE quotient for every float of the binades that determine it (see
tests/native/markstein_const.c for why those binades suffice)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_constant_divisor_quotients_are_correctly_rounded(tmp_path):
    exe = tmp_path / "markstein_const"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe),
                    os.path.join(HERE, "native", "markstein_const.c"), "-lm"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "divisor 127: 0 mismatches" in r.stdout and "divisor 255: 0 mismatches" in r.stdout
