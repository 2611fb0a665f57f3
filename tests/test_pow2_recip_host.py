"""The kernels' Newton-Raphson reciprocal, built for the host from the same
device header and compared with the exact quotient it defines: the per-row
quantisation multiplier floor(127 2^(e+16) / a) of the per-token ActQuant and
NormQuant (DetLLM blog, section "DetLLM": one integer multiply and one shift
per element, one division per row) and the softmax row-sum reciprocal
floor(2^(e+23) / sum)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def test_pow2_recip_matches_floor_division(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "pow2_recip")
    r = subprocess.run([nvcc, "-O2", "-x", "cu", os.path.join(HERE, "host_pow2_recip.cu"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe, "127", "20000"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    cases, bad = r.stdout.split()[1], r.stdout.split()[3]
    assert int(bad) == 0 and int(cases) > 30_000_000, r.stdout
