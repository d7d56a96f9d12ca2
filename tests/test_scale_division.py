"""The CUDA NVFP4 quantizers divide with Markstein's FMA-corrected quotient
instead of an IEEE division.  This CPU test runs an exhaustive check that the
method gives the IEEE quotient bit for bit on every input the kernels can see
(every bf16 block maximum over 6; every S_enc from a bf16 amax over every
positive E4M3 block scale).  The check is plain C compiled here; it shares no
code with the oracle or the kernels."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_markstein_quotients_match_ieee_division(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    exe = str(tmp_path / "scale_division_check")
    subprocess.check_call([gcc, "-O2", "-ffp-contract=off", "-o", exe,
                           os.path.join(HERE, "csrc", "scale_division_check.c"), "-lm"])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "0 mismatches; S_enc/sb" in out.stdout and out.stdout.rstrip().endswith("0 mismatches")
