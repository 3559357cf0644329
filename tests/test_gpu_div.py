"""The quantize kernels divide by a scale through its correctly rounded
reciprocal and one Markstein correction step instead of an IEEE division per
element. The codes must still equal the formula's IEEE fp32 quotient, so the
quotient itself is checked against __fdiv_rn over about 1.6e9 operand pairs:
every fp16 scale against every fp16 numerator, random fp32 differences of fp16
values with the half-integer quotients where rounding decides a code, and every
fp16 pattern (zeros, infinities and NaNs included) against fp32 scales from
2^-96 to 2^96 (the FP8 path)."""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "quantized_kv_cache_quant_gb300", "csrc")


def test_reciprocal_quotient_is_the_ieee_quotient():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "div_check")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-I", CSRC,
                        os.path.join(HERE, "div_check.cu"), "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    m = re.search(r"A=(\d+) B=(\d+) C=(\d+) checked_A=(\d+) checked_B=(\d+) checked_C=(\d+) err=(.*)", out)
    assert m, out
    a, b, c, na, nb, nc, err = m.groups()
    assert err.strip() == "no error"
    assert int(na) > 9e8 and int(nb) > 1e9 and int(nc) > 5e8
    assert (int(a), int(b), int(c)) == (0, 0, 0), out
