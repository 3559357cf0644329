"""Failure detection on the GPU without a fault: every device wait of the
decode kernels is bounded (1 s) and reports bit 0 of a status word instead of
hanging. This test builds a kernel around the same bounded-wait helper the
kernels use, waits on an mbarrier that nothing ever completes, and checks that
the wait gives up, the status bit is set and the context keeps working."""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "quantized_kv_cache_quant_gb300", "csrc")


def test_bounded_wait_reports_timeout():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "wait_timeout_check")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-I", CSRC,
                        os.path.join(HERE, "wait_timeout_check.cu"), "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120).stdout
    m = re.search(r"status=(\d+) completed=(-?\d+) ms=([\d.]+) err=(.*) after=(-?\d+) err2=(.*)", out)
    assert m, out
    status, completed, ms, err, after, err2 = m.groups()
    assert int(status) == 1 and int(completed) == 0
    assert 900 <= float(ms) <= 5000          # gave up after about its 1 s limit
    assert err.strip() == "no error" and err2.strip() == "no error" and int(after) == 1


def test_decode_status_stays_clear_after_normal_calls():
    import numpy as np
    import torch
    from quantized_kv_cache_quant_gb300 import kvq, workloads
    x = workloads.make_inputs(2, 2, 8, 128, 500, 1, 3)
    c = kvq.KiviCache(2, 2, 8, 128, 2, 2, 128, 600)
    c.prefill(torch.from_numpy(x.k).cuda(), torch.from_numpy(x.v).cuda())
    for _ in range(3):
        c.decode(torch.from_numpy(np.ascontiguousarray(x.q[0])).cuda())
    assert c.status() == 0
