"""Benchmark of the quantized-KV decode hot path on GB300.

Workload (default): the 128K streaming KIVI 2-bit cache — batch 4, 8 kv heads,
64 query heads (GQA 8), head_dim 128, prefill-quantize 131072 tokens, then
decode steps that each append one fp16 K/V token (flushing the 128-token fp16
window into 4 new groups every 128 steps) and run split-K decode attention
over 130944+ grouped tokens plus the window.

One timed step = kv_append_token (+ the flush when due) + kv_decode_attention.
``value`` = algorithmic bytes of the timed steps / device time (GB/s), inputs
resident in HBM. ``e2e`` repeats the steps through the same C-ABI calls with
the step inputs (q, k_new, v_new) copied from pinned host memory and the
output copied back inside the timed region. The prefill is timed separately
(quantize tokens/s). ``roofline`` reports the decode kernel alone (CUDA events
around each kv_decode_attention launch) against the measured HBM copy
bandwidth. ``cpu_baseline`` / ``--impl reference`` time the CPU oracle on a
bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# the CPU-baseline leg is timed single-threaded: pin BLAS/OpenMP before numpy loads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_kv_cache_quant_gb300 import metrics, workloads  # noqa: E402

METRIC = "decode-attn KV bytes GB/s (% of GB300 HBM peak); quantize tokens/s"
# ncu summary of the decode kernel on the default workload; its "traffic-record:"
# line holds DRAM bytes of one captured launch and a hash of the sources it ran
DECODE_PROFILE = os.path.join(ROOT, "profiles", "kivi_decode_kernel_128k_stream.md")
DECODE_SOURCES = ("kivi_kernels.cu", "kvq_device.cuh")  # the decode kernel and its device helpers
FALLBACK_HBM_GBS = 6800.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling: one independent cache per GPU)
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(x: float, world: int, op_name: str) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=getattr(dist.ReduceOp, op_name))
    return float(t.item())


def max_over_ranks(x: float, world: int) -> float:
    return _reduce(x, world, "MAX")


def sum_over_ranks(x: float, world: int) -> float:
    return _reduce(x, world, "SUM")


def aggregate(bytes_local: float, seconds_local: float, world: int):
    """Whole-job throughput under weak scaling: the bytes every rank moved over
    the slowest rank's time. Returns (GB/s, max seconds)."""
    t = max_over_ranks(seconds_local, world)
    return sum_over_ranks(float(bytes_local), world) / t / 1e9, t


def timed_window_start(w, warmup: int, steps: int) -> int:
    """First timed step: after at least `warmup` untimed steps, and early enough
    that the timed steps cover a residual flush (the appends that find a full
    window: steps residual, 2 * residual, ... after a prefill that fills it)."""
    if w.residual <= 0:
        return warmup
    flush_steps = range(w.residual, w.decode_steps, w.residual)
    if any(warmup <= f < warmup + steps for f in flush_steps):
        return warmup
    for f in flush_steps:
        start = max(warmup, f - steps // 2)
        if start <= f < start + steps and start + steps <= w.decode_steps:
            return start
    return warmup


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import torch
    from quantized_kv_cache_quant_gb300 import kvq

    torch.cuda.set_device(local)
    w = workloads.WORKLOADS[args.workload]
    assert isinstance(w, workloads.KiviWorkload), "bench.py times the KIVI streaming workloads"
    first = timed_window_start(w, args.warmup, args.steps)
    if first + args.steps > w.decode_steps:
        raise SystemExit(f"--warmup + --steps must be <= {w.decode_steps} for {w.name}")
    x = workloads.kivi_inputs(w)   # same seeded data on every rank (weak scaling replicas)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    k_d, v_d = dev(x.k), dev(x.v)
    q_d = [dev(x.q[s]) for s in range(w.decode_steps)]
    kn_d = [dev(x.k_new[s]) for s in range(w.decode_steps)]
    vn_d = [dev(x.v_new[s]) for s in range(w.decode_steps)]
    cache = kvq.KiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual,
                          w.max_tokens)
    stream = torch.cuda.current_stream()
    out = torch.empty((w.batch, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")

    # --- prefill (quantize tokens/s): warm-up then timed repetitions ---
    for _ in range(2):
        cache.prefill(k_d, v_d)
    reps = 5
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        cache.prefill(k_d, v_d)
    e1.record(stream)
    torch.cuda.synchronize()
    prefill_s = e0.elapsed_time(e1) / 1e3 / reps
    prefill_tokens = w.batch * w.prefill
    prefill_bytes = metrics.kivi_prefill_bytes(w.batch, w.kv_heads, w.head_dim, w.k_bits, w.v_bits,
                                               cache.n_grouped, cache.n_resid)

    def step_bytes(before_grouped, after_grouped, n_resid):
        b = metrics.kivi_append_bytes(w.batch, w.kv_heads, w.head_dim)
        if after_grouped != before_grouped:
            b += metrics.kivi_flush_bytes(w.batch, w.kv_heads, w.head_dim, w.k_bits, w.v_bits,
                                          after_grouped - before_grouped)
        return b + metrics.kivi_decode_bytes(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits,
                                             after_grouped, n_resid)

    def run_steps(first, count, timed_events=None):
        """Enqueue `count` device-resident steps; returns (bytes, launches, decode bytes list)."""
        nbytes, launches, dec_bytes = 0, 0, []
        for i in range(count):
            s = first + i
            g0 = cache.n_grouped
            cache.append(kn_d[s], vn_d[s])
            launches += 1 + (1 if cache.n_grouped != g0 else 0)
            if timed_events is not None:
                timed_events[i][0].record(stream)
            cache.decode(q_d[s], out=out)
            if timed_events is not None:
                timed_events[i][1].record(stream)
            launches += 1
            nbytes += step_bytes(g0, cache.n_grouped, cache.n_resid)
            dec_bytes.append(metrics.kivi_decode_bytes(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits,
                                                       w.v_bits, cache.n_grouped, cache.n_resid))
        return nbytes, launches, dec_bytes

    # --- the decode kernel alone: events around each decode of the same steps ---
    cache.prefill(k_d, v_d)
    run_steps(0, first)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    _, _, dec_bytes = run_steps(first, args.steps, ev)
    torch.cuda.synchronize()
    dec_times = [a.elapsed_time(b) / 1e3 for a, b in ev]
    achieved = statistics.mean(db / dt for db, dt in zip(dec_bytes, dec_times)) / 1e9

    # --- device-resident timed steps (nothing between the kernels of a step, as a
    # caller runs them: the decode may start while the append's copy finishes) ---
    cache.prefill(k_d, v_d)
    run_steps(0, first)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    start.record(stream)
    g_before = cache.n_grouped
    nbytes, launches, _ = run_steps(first, args.steps)
    end.record(stream)
    timed_flushes = (cache.n_grouped - g_before) // w.residual
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    barrier(world)
    value, t = aggregate(nbytes, start.elapsed_time(end) / 1e3, world)
    status = cache.status()

    # --- end to end: host buffers, copies inside the timed region ---
    # One pinned host block per step holds [q | k_new | v_new] back to back, so a
    # step's inputs cross in one copy (device tensors are views of one buffer,
    # offsets multiples of 256 bytes as the calls require). The copies run on
    # their own streams, as a serving loop runs them: step i + 1's inputs go up
    # while step i computes, step i's output comes down while step i + 1
    # computes; two input and two output buffers alternate, and events order
    # every reuse. The timed region ends after the last output has landed.
    nq, nk = x.q[0].size, x.k_new[0].size
    assert (2 * nq) % 256 == 0 and (2 * nk) % 256 == 0
    step_h = [torch.from_numpy(np.concatenate([x.q[s].ravel(), x.k_new[s].ravel(), x.v_new[s].ravel()])).pin_memory()
              for s in range(w.decode_steps)]
    bufs = [torch.empty_like(step_h[0], device="cuda") for _ in range(2)]
    views = [(b[:nq].view(x.q[0].shape), b[nq:nq + nk].view(x.k_new[0].shape), b[nq + nk:].view(x.v_new[0].shape))
             for b in bufs]
    outs = [torch.empty_like(out) for _ in range(2)]
    outs_h = [torch.empty(out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done, used, d2h_done = ([ev() for _ in range(args.steps)] for _ in range(3))
    cache.prefill(k_d, v_d)
    run_steps(0, first)
    barrier(world)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    up.wait_event(e_start)
    down.wait_event(e_start)

    def upload(i):
        if i >= 2:
            up.wait_event(used[i - 2])  # step i - 2 is done with this buffer
        with torch.cuda.stream(up):
            bufs[i % 2].copy_(step_h[first + i], non_blocking=True)
        h2d_done[i].record(up)

    e2e_bytes = 0
    upload(0)
    for i in range(args.steps):
        if i + 1 < args.steps:
            upload(i + 1)
        stream.wait_event(h2d_done[i])
        if i >= 2:
            stream.wait_event(d2h_done[i - 2])  # step i - 2's output has left this buffer
        qb, kb, vb = views[i % 2]
        g0 = cache.n_grouped
        cache.append(kb, vb)
        cache.decode(qb, out=outs[i % 2])
        used[i].record(stream)
        down.wait_event(used[i])
        with torch.cuda.stream(down):
            outs_h[i % 2].copy_(outs[i % 2], non_blocking=True)
        d2h_done[i].record(down)
        e2e_bytes += step_bytes(g0, cache.n_grouped, cache.n_resid)
    stream.wait_event(d2h_done[args.steps - 1])
    e_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_value, _ = aggregate(e2e_bytes, e_start.elapsed_time(e_end) / 1e3, world)
    h2d = step_h[0].numel() * 2
    d2h = outs_h[0].numel() * 4

    hbm, peak_kind = peaks()
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16",
        "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.batch, "kv_heads": w.kv_heads, "q_heads": w.q_heads,
            "head_dim": w.head_dim, "k_bits": w.k_bits, "v_bits": w.v_bits, "group": 32, "residual": w.residual,
            "context_start": w.prefill, "steps_from": first, "timed_flushes": timed_flushes,
            "dtypes": {"cache": f"int{w.k_bits}/int{w.v_bits} codes, fp16 scales, zero points and window",
                       "q": "fp16", "tensor_core_operands": "fp16", "accumulate": "fp32", "out": "fp32"},
            "operands": "2-bit codes as fp16 tensor-core operands, fp32 accumulation",
            "l2": "inputs larger than L2: each step reads ~355 MB of cache against a 129 MB L2",
        },
        "pct_of_hbm_peak": round(100 * value / hbm, 2),
        "quantize_tokens_per_s": round(prefill_tokens / prefill_s, 1),
        "quantize_gb_s": round(prefill_bytes / prefill_s / 1e9, 2),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": measured_traffic(w.name, statistics.mean(dec_bytes)),
                     "traffic_unit": "DRAM bytes per launch (ncu capture, scaled to the mean launch)",
                     "kernel": "kivi_decode_kernel<128,2,2,4,NoSeqs>", "peak_source": f"{peak_kind} hbm_gbs",
                     "decode_us": round(statistics.mean(dec_times) * 1e6, 2)},
        "device_status": status,
    }
    if clk:
        res["clocks"] = clk
    return res


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
def decode_sources_sha256():
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "quantized_kv_cache_quant_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload, mean_alg_bytes):
    """DRAM read + write bytes per decode launch from the committed ncu capture,
    scaled from the captured launch's algorithmic bytes to this run's mean. None
    when the capture is of another workload or of decode sources that have
    changed since it was taken."""
    try:
        with open(DECODE_PROFILE) as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    for line in lines:
        if line.startswith("traffic-record:"):
            rec = json.loads(line.split(":", 1)[1])
            if rec.get("workload") != workload or rec.get("sources_sha256") != decode_sources_sha256():
                return None
            return int(round(rec["dram_bytes"] * mean_alg_bytes / rec["algorithmic_bytes"]))
    return None


def oracle_sample_setup(w):
    """One (batch row 0, kv head 0) of the workload, as a 1 x 1 oracle cache."""
    from oracle import kivi
    x = workloads.kivi_inputs(w)
    gq = w.q_heads // w.kv_heads
    c = kivi.KiviCache(1, 1, w.head_dim, w.k_bits, w.v_bits, w.residual, w.max_tokens)
    c.prefill(x.k[:1, :1], x.v[:1, :1])
    return x, c, gq


def oracle_step(w, x, c, gq, s):
    from oracle import attention
    c.append(x.k_new[s, :1, :1], x.v_new[s, :1, :1])
    kh, vh = c.keys_hat(0, 0), c.values_hat(0, 0)
    scale = attention.default_scale(w.head_dim)
    for r in range(gq):
        attention.softmax_attend(x.q[s, 0, r], kh, vh, scale)
    return metrics.kivi_decode_bytes(1, 1, gq, w.head_dim, w.k_bits, w.v_bits, c.n_grouped, c.n_resid)


def _oracle_worker(conn, w, pair, k, v, q, k_new, v_new):
    """One host process: the oracle cache of one (batch row, kv head) pair of the
    workload; runs decode steps on request and answers with their bytes."""
    from oracle import attention, kivi
    gq = w.q_heads // w.kv_heads
    c = kivi.KiviCache(1, 1, w.head_dim, w.k_bits, w.v_bits, w.residual, w.max_tokens)
    c.prefill(k, v)
    scale = attention.default_scale(w.head_dim)
    conn.send("ready")
    while True:
        s = conn.recv()
        if s is None:
            break
        if isinstance(s, tuple):  # ("advance", step): the cache state only, no attention (untimed steps)
            c.append(k_new[s[1]], v_new[s[1]])
            conn.send(0)
            continue
        c.append(k_new[s], v_new[s])
        kh, vh = c.keys_hat(0, 0), c.values_hat(0, 0)
        for r in range(gq):
            attention.softmax_attend(q[s, r], kh, vh, scale)
        conn.send(metrics.kivi_decode_bytes(1, 1, gq, w.head_dim, w.k_bits, w.v_bits, c.n_grouped, c.n_resid))


class OraclePool:
    """One spawned process per host core (at most one per (batch row, kv head)
    pair), each holding the oracle cache of its own pair; a step runs the same
    decode step on every pair at once. Spawned, not forked: the parent may hold
    a CUDA context."""

    def __init__(self, w, n_proc):
        import multiprocessing as mp
        x = workloads.kivi_inputs(w)
        pairs = [(b, h) for b in range(w.batch) for h in range(w.kv_heads)][:max(1, n_proc)]
        gq = w.q_heads // w.kv_heads
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for b, h in pairs:
            a, bconn = ctx.Pipe()
            args = (bconn, w, (b, h), x.k[b:b + 1, h:h + 1].copy(), x.v[b:b + 1, h:h + 1].copy(),
                    x.q[:, b, h * gq:(h + 1) * gq].copy(), x.k_new[:, b:b + 1, h:h + 1].copy(),
                    x.v_new[:, b:b + 1, h:h + 1].copy())
            p = ctx.Process(target=_oracle_worker, args=args, daemon=True)
            p.start()
            self.conns.append(a)
            self.procs.append(p)
        for cn in self.conns:
            assert cn.recv() == "ready"
        self.n = len(self.conns)
        self.gq = gq

    def step(self, s) -> int:
        for cn in self.conns:
            cn.send(s)
        return sum(cn.recv() for cn in self.conns)

    def advance(self, s) -> None:
        """Append step s's token on every pair without the attention (untimed steps)."""
        for cn in self.conns:
            cn.send(("advance", s))
        for cn in self.conns:
            cn.recv()

    def close(self):
        for cn in self.conns:
            cn.send(None)
        for p in self.procs:
            p.join(timeout=10)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(w, budget_s=12.0):
    """The oracle on the host cores: single-threaded on one (batch row, kv head)
    pair, and one process per core over as many pairs, each for about budget_s."""
    x, c, gq = oracle_sample_setup(w)
    t0 = time.perf_counter()
    nbytes, steps = 0, 0
    while time.perf_counter() - t0 < budget_s and steps < w.decode_steps:
        nbytes += oracle_step(w, x, c, gq, steps)
        steps += 1
    single = nbytes / (time.perf_counter() - t0) / 1e9
    del x, c
    cores = min(host_cores(), w.batch * w.kv_heads)
    pool = OraclePool(w, cores)
    t0 = time.perf_counter()
    nbytes, asteps = 0, 0
    while time.perf_counter() - t0 < budget_s and asteps < w.decode_steps:
        nbytes += pool.step(asteps)
        asteps += 1
    dt = time.perf_counter() - t0
    pool.close()
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": pool.n, "kind": "oracle",
            "sample": f"{asteps} decode steps of {pool.n} (batch row, kv head) pairs of {w.name}, one process per "
                      f"core: append + flush + float64 dequantize + attention for each pair's {gq} query heads",
            "single_core": {"value": round(single, 4), "cores": 1,
                            "sample": f"{steps} decode steps of one pair, single-threaded"}}


def run_reference(args, world, rank):
    w = workloads.WORKLOADS[args.workload]
    cores = min(host_cores(), w.batch * w.kv_heads)
    pool = OraclePool(w, cores)
    first = timed_window_start(w, args.warmup, args.steps)
    for s in range(first - args.warmup):
        pool.advance(s)            # the cache state of the steps before the warm-up window
    for s in range(first - args.warmup, first):
        pool.step(s)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += pool.step(first + i)
    dt = time.perf_counter() - t0
    pool.close()
    value = nbytes / dt / 1e9
    sample = (f"per step: {pool.n} (batch row, kv head) pairs of {w.name}, one process per core — append + flush + "
              f"float64 dequantize + attention for each pair's {pool.gq} query heads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": pool.n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# --table: every workload's decode call (and quantize) timed alone
# ---------------------------------------------------------------------------
TABLE_ALL = (workloads.MHA_4K.name, workloads.GQA_8K_2BIT.name, workloads.GQA_8K_4BIT.name,
             workloads.STREAM_128K.name, workloads.FP8_32K.name, workloads.FP8_32K_E5M2_PH.name,
             workloads.FP8_32K_QFP8.name, workloads.NVFP4_32K.name, workloads.PAGED_GQA_8K.name,
             workloads.PAGED_VAR_16K.name, workloads.PAGED_GQA4_VAR_16K.name)


def table_rows(names):
    """One dict per workload: trimmed mean time of the decode-attention call over
    the prefilled cache, its algorithmic GB/s and fraction of the HBM peak, and
    the quantize rate. Before each repetition L2 is flushed by writing 512 MB
    and reading them back: the timed call finds none of its data in L2 and no
    dirty lines of the flush to write back (after the write alone, the 129 MB
    of dirty lines cost a 128K prefill ~20 us of write-back)."""
    import torch
    from quantized_kv_cache_quant_gb300 import kvq

    hbm, _ = peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def timed(fn, reps=40, warm=3):
        # The event clock ticks in steps of about 2 us here; its phase against
        # the kernel start is random, so the mean of many calls (the fastest and
        # slowest tenth dropped) resolves below one step where a median cannot.
        ts = []
        for r in range(reps + warm):
            flush.zero_()
            flush_sum = torch.sum(flush, dtype=torch.int64)  # reads the 512 MB back: L2 clean
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            if r >= warm:
                ts.append(a.elapsed_time(b) / 1e3)
        del flush_sum
        ts.sort()
        cut = len(ts) // 10
        return statistics.mean(ts[cut:len(ts) - cut])

    def row(w, call, t_dec, nbytes, **extra):
        line = {"workload": w.name, "call": call, "us": round(t_dec * 1e6, 2), "bytes": nbytes,
                "GB_s": round(nbytes / t_dec / 1e9, 1), "frac": round(nbytes / t_dec / 1e9 / hbm, 4)}
        line.update(extra)
        return line

    rows = []
    for name in names:
        w = workloads.WORKLOADS[name]
        if isinstance(w, workloads.PagedKiviWorkload):
            x, lens, table = workloads.paged_inputs(w, steps=1)
            cache = kvq.PagedKiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual,
                                       w.max_tokens, w.num_blocks)
            cache.table.copy_(dev(table))
            k_d, v_d, q_d = dev(x.k), dev(x.v), dev(x.q[0])
            t_pre = timed(lambda: cache.prefill(k_d, v_d, lens.tolist()), reps=20)
            out = torch.empty((w.batch, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
            t_dec = timed(lambda: cache.decode(q_d, out=out))
            ng = [cache.n_grouped(b) for b in range(w.batch)]
            nr = [cache.n_resid(b) for b in range(w.batch)]
            nbytes = metrics.kivi_paged_decode_bytes(w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, ng, nr)
            rows.append(row(w, "kv_paged_decode_attention", t_dec, nbytes, tokens=int(lens.sum()),
                            prefill_us=round(t_pre * 1e6, 1),
                            quantize_tokens_per_s=round(float(lens.sum()) / t_pre, 1), status=cache.status()))
            del k_d, v_d, cache
        elif isinstance(w, workloads.KiviWorkload):
            x = workloads.kivi_inputs(w, steps=1)
            cache = kvq.KiviCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits, w.residual,
                                  w.max_tokens)
            k_d, v_d, q_d = dev(x.k), dev(x.v), dev(x.q[0])
            t_pre = timed(lambda: cache.prefill(k_d, v_d), reps=20)
            out = torch.empty((w.batch, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
            t_dec = timed(lambda: cache.decode(q_d, out=out))
            nbytes = metrics.kivi_decode_bytes(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.k_bits, w.v_bits,
                                               cache.n_grouped, cache.n_resid)
            pre_bytes = metrics.kivi_prefill_bytes(w.batch, w.kv_heads, w.head_dim, w.k_bits, w.v_bits,
                                                   cache.n_grouped, cache.n_resid)
            rows.append(row(w, "kv_decode_attention", t_dec, nbytes, prefill_us=round(t_pre * 1e6, 1),
                            prefill_GB_s=round(pre_bytes / t_pre / 1e9, 1),
                            prefill_frac=round(pre_bytes / t_pre / 1e9 / hbm, 4),
                            quantize_tokens_per_s=round(w.batch * w.prefill / t_pre, 1), status=cache.status()))
            del k_d, v_d, cache
        elif isinstance(w, workloads.Nvfp4Workload):
            k, v, q, table = workloads.fp8_inputs(w)
            nb = w.blocks_per_seq
            tbl = dev(table)
            pools, t_q = [], []
            for x16, role in ((k, kvq.ROLE_KEY), (v, kvq.ROLE_VALUE)):
                xd = dev(x16)
                p = kvq.Nvfp4Pool(role, w.batch * nb, w.kv_heads, w.head_dim)
                t_q.append(timed(lambda: p.quantize(xd, tbl, nb), reps=10))
                pools.append(p)
                del xd
            out = torch.empty((w.batch, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
            wsd = kvq.nvfp4_decode_workspace_bytes(w.batch, w.q_heads, w.head_dim)
            ws = torch.zeros(wsd, dtype=torch.uint8, device="cuda")
            lens = dev(np.full(w.batch, w.context, np.int32))
            q_d = dev(q)
            t_dec = timed(lambda: kvq.nvfp4_decode_attention(q_d, pools[0].desc, pools[1].desc, tbl, lens, w.batch,
                                                             w.q_heads, nb, w.context, out, True, 0.0, ws, wsd))
            nbytes = metrics.nvfp4_decode_bytes(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.context, nb)
            qbytes = metrics.nvfp4_quantize_bytes(w.batch, w.kv_heads, w.context, w.head_dim, True)
            rows.append(row(w, "nvfp4_decode_attention", t_dec, nbytes,
                            quantize_us_k_v=[round(t * 1e6, 1) for t in t_q],
                            quantize_GB_s=round(qbytes / statistics.mean(t_q) / 1e9, 1),
                            quantize_tokens_per_s=round(w.batch * w.context / statistics.mean(t_q), 1),
                            status=int(ws[:4].view(torch.int32).item())))
            del pools
        else:
            k, v, q, table = workloads.fp8_inputs(w)
            nb = w.blocks_per_seq
            tbl = dev(table)
            pools, t_q = [], []
            for x16, role in ((k, kvq.ROLE_KEY), (v, kvq.ROLE_VALUE)):
                xd = dev(x16)
                p = kvq.Fp8Pool(role, w.batch * nb, w.kv_heads, w.head_dim, fp8_format=kvq.FP8_FORMATS[w.fmt],
                                per_head=w.per_head)
                t_q.append(timed(lambda: p.quantize(xd, tbl, nb), reps=10))
                pools.append(p)
                del xd
            out = torch.empty((w.batch, w.q_heads, w.head_dim), dtype=torch.float32, device="cuda")
            wsd = kvq.fp8_decode_workspace_bytes(w.batch, w.q_heads, w.head_dim)
            ws = torch.zeros(wsd, dtype=torch.uint8, device="cuda")
            lens = dev(np.full(w.batch, w.context, np.int32))
            q_d = dev(q)
            t_dec = timed(lambda: kvq.fp8_decode_attention(q_d, pools[0].desc, pools[1].desc, tbl, lens, w.batch,
                                                           w.q_heads, nb, w.context, out, True, 0.0, ws, wsd,
                                                           q_fp8=w.q_fp8))
            nbytes = metrics.fp8_decode_bytes(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.context, nb)
            qbytes = metrics.fp8_quantize_bytes(w.batch, w.kv_heads, w.context, w.head_dim, True)
            rows.append(row(w, "fp8_decode_attention", t_dec, nbytes,
                            quantize_us_k_v=[round(t * 1e6, 1) for t in t_q],
                            quantize_GB_s=round(qbytes / statistics.mean(t_q) / 1e9, 1),
                            quantize_tokens_per_s=round(w.batch * w.context / statistics.mean(t_q), 1),
                            status=int(ws[:4].view(torch.int32).item())))
            del pools
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return rows


def run_table(args):
    names = TABLE_ALL if args.table == "all" else args.table.split(",")
    for r in table_rows(names):
        print(json.dumps(r), flush=True)


def launcher_cmd(n_gpus: int, argv, port: int):
    """The command that runs this script as n_gpus ranks on one node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.STREAM_128K.name, choices=sorted(
        n for n, w in workloads.WORKLOADS.items() if isinstance(w, workloads.KiviWorkload)))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-table", action="store_true", help="leave the per-workload decode table out of the line")
    ap.add_argument("--table", default=None,
                    help="'all' or comma-separated workload names: time each decode call alone instead")
    args = ap.parse_args(argv)
    if args.table:
        run_table(args)
        return 0
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # started without a launcher: run the N ranks under torch.distributed.run
        return subprocess.call(launcher_cmd(args.gpus, sys.argv[1:] if argv is None else argv, free_port()))
    world, rank, local = dist_setup()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU")
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    res = run_ours(args, world, rank, local)
    if rank == 0 and world == 1 and not args.no_table:
        res["table"] = {r.pop("workload"): r for r in table_rows(TABLE_ALL)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(workloads.WORKLOADS[args.workload])
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
