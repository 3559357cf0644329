"""The bench contract on the host: the reference arm's JSON line, the warm-up
rule, and the algorithmic byte counts the GB/s figures divide by."""
import json
import os
import subprocess
import sys

import pytest

from oracle import sizes
from quantized_kv_cache_quant_gb300 import metrics, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_prints_one_json_line():
    r = _bench("--impl", "reference", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == workloads.STREAM_128K.name
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_refused():
    r = _bench("--steps", "2", "--warmup", "2", timeout=120)
    assert r.returncode != 0
    assert "--warmup must be >= 3" in r.stderr


@pytest.mark.parametrize("d,kb,vb,per_token", [(128, 2, 2, 84.0), (128, 4, 4, 148.0), (64, 2, 2, 44.0)])
def test_grouped_bytes_per_token_follow_the_layout(d, kb, vb, per_token):
    """84 B per grouped token and kv head at D = 128 and 2 bits (2688-byte group records), 148 B at 4
    bits, 44 B at D = 64 (the value meta stays 128 bytes), in agreement with the oracle's record sizes."""
    assert metrics.grouped_bytes_per_token(d, kb, vb) == per_token
    assert sum(sizes.kivi_group_bytes(d, kb, vb).values()) == 32 * per_token


def test_decode_bytes_of_the_128k_workload():
    """One decode call at the start of the 128K run: 130944 grouped + 128 window tokens over 32
    (b, kv head) pairs, plus q (fp16) and out (fp32)."""
    w = workloads.STREAM_128K
    got = metrics.kivi_decode_bytes(w.batch, w.kv_heads, w.q_heads, w.head_dim, 2, 2, 130944, 128)
    grouped = 130944 * 84 * 32
    window = 128 * 128 * 2 * 2 * 32
    assert got == grouped + window + 4 * 64 * 128 * 2 + 4 * 64 * 128 * 4


def test_paged_decode_bytes_are_the_sequences_sum():
    ng, nr = [0, 32 * 5, 32 * 100], [7, 128, 97]
    total = metrics.kivi_paged_decode_bytes(8, 32, 128, 2, 2, ng, nr)
    want = sum(metrics.kivi_decode_bytes(1, 8, 32, 128, 2, 2, g, r) + 4 * (g // 32) for g, r in zip(ng, nr))
    assert total == want


def test_gpus_that_disagree_with_the_launcher_are_refused():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode != 0
    assert "--gpus 2 but WORLD_SIZE=1" in r.stderr


def test_gpus_without_a_launcher_runs_one_rank_per_gpu():
    sys.path.insert(0, ROOT)
    import bench
    cmd = bench.launcher_cmd(4, ["--gpus", "4", "--steps", "7"], 29511)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--nnodes=1" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1" and cmd[cmd.index("--master-port") + 1] == "29511"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "7"] and cmd[-5].endswith("bench.py")


@pytest.mark.parametrize("warmup,steps", [(3, 128), (5, 20), (3, 3), (200, 10), (3, 300)])
def test_timed_steps_cover_a_residual_flush(warmup, steps):
    sys.path.insert(0, ROOT)
    import bench
    w = workloads.STREAM_128K
    first = bench.timed_window_start(w, warmup, steps)
    assert first >= warmup and first + steps <= w.decode_steps
    assert any(first <= f < first + steps for f in range(w.residual, w.decode_steps, w.residual))
