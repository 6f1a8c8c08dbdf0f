#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one attn_fwd call (the whole path: tensor maps, the prefill
kernel, or the split-KV decode kernel plus its combine kernel) over one batch
of synthetic bf16 inputs already resident in HBM.  L2 is flushed (a 256 MB
write) before every step, outside the per-step CUDA events; the timed value is
the sum of the per-step event durations on the launching stream, between a
barrier + synchronize on both sides.  Multi-GPU runs (torchrun) are
independent replicas of the same problem on each GPU ("weak" scaling): the
path has no exchange step, so there is no collective on the data path.

Rank 0 prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle
(the only reference this path has) on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from blackwell_programming_gb300 import synthetic as syn  # noqa: E402

METRIC = "attention fwd TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "gqa_causal_d128"
L2_FLUSH_BYTES = 256 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {"gemm": "blackwell_programming_gb300/csrc/gemm_sm103.cu",
                  "prefill": "blackwell_programming_gb300/csrc/prefill_sm103.cu",
                  "decode": "blackwell_programming_gb300/csrc/decode_pair_sm103.cu",
                  "latent_prefill": "blackwell_programming_gb300/csrc/decode_pair_sm103.cu"}


# ----------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int) -> float:
    """Maximum of a float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    return units_per_rank * world / seconds_max


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_hash(kind: str) -> str:
    with open(os.path.join(ROOT, KERNEL_SOURCES[kind]), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def committed_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel") != kind or e.get("source_sha256_16") != kernel_hash(kind):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ------------------------------------------------------------ CPU oracle

def oracle_sample(wl, budget_s: float = 12.0):
    """Time the fp64 oracle on one (batch, head) problem of the workload,
    repeated until the time budget is spent.

    The problem is a single head with the workload's shape and input
    distribution (Nq x Nkv, d_qk, d_v, causal or not), drawn as its own
    1-head workload; the oracle runs it whole each time.  Returns
    (TFLOP/s, sample description, threads).  FLOPs of a head use the
    reported formula (4*Nq*Nkv*d, halved when causal; 2*Nq*Nkv*(d_qk+d_v)).
    """
    import numpy as np
    from oracle import attention_head
    cores = blas_threads()
    small = wl
    # the decode shape has one query per head; take whole batch rows at a time
    per_head = 2.0 * wl.Nq * wl.Nkv * (wl.d_qk + wl.d_v) / (2.0 if wl.causal else 1.0)
    done, flops, t0 = 0, 0.0, time.perf_counter()
    rng_heads = [(b, h) for b in range(small.B) for h in range(small.Hq)]
    one = syn.Workload(wl.name + "_head", 1, 1, 1, wl.Nq, wl.Nkv, wl.d_qk, wl.d_v, wl.causal, wl.scale,
                       wl.q_factor, wl.kv_factor, wl.v_aliases_k, wl.seed)
    inp = syn.make_inputs(one)      # one head of the same distribution
    q, k, v = inp.f64()
    elapsed = 0.0
    while done < len(rng_heads):
        s = time.perf_counter()
        if DROPOUT > 0.0:
            from oracle.dropout_fp64 import attention_dropout_head
            attention_dropout_head(q[0, 0], k[0, 0], v[0, 0], wl.causal, wl.scale, DROPOUT, DROPOUT_SEED, 0, 0)
        else:
            attention_head(q[0, 0], k[0, 0], v[0, 0], wl.causal, wl.scale)
        elapsed += time.perf_counter() - s
        done += 1
        flops += per_head
        if elapsed >= budget_s or time.perf_counter() - t0 > 2 * budget_s:
            break
    desc = ("one (batch, head) problem of %s's shape and distribution (%d x %d keys, d %d/%d%s), run %d times "
            "(the workload has %d such problems), full rows, fp64 numpy%s") % (
        wl.name, wl.Nq, wl.Nkv, wl.d_qk, wl.d_v, ", causal" if wl.causal else "", done, len(rng_heads),
        ", dropout %g" % DROPOUT if DROPOUT > 0.0 else "")
    return flops / elapsed / 1e12, desc, cores


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def single_thread_oracle(names=("tile_d64", "causal_d64_bigq"), budget_s: float = 3.0):
    """The fp64 oracle on whole small workloads in a child process whose BLAS
    and OpenMP pools are limited to one thread:
    {workload: {"tflops": ..., "seconds": ..., "runs": ...}}, or {} if the
    child fails."""
    code = (
        "import json, sys, time\n"
        "sys.path.insert(0, %r)\n"
        "from blackwell_programming_gb300 import synthetic as syn\n"
        "from oracle import attention\n"
        "res = {}\n"
        "for name in %r:\n"
        "    wl = syn.WORKLOADS[name]\n"
        "    q, k, v = syn.make_inputs(wl).f64()\n"
        "    runs, t0 = 0, time.perf_counter()\n"
        "    while True:\n"
        "        attention(q, k, v, wl.causal, wl.scale)\n"
        "        runs += 1\n"
        "        if time.perf_counter() - t0 >= %r:\n"
        "            break\n"
        "    secs = (time.perf_counter() - t0) / runs\n"
        "    res[name] = {'tflops': wl.flops / secs / 1e12, 'seconds': secs, 'runs': runs}\n"
        "print(json.dumps(res))\n") % (ROOT, tuple(names), budget_s)
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = "1"
    try:
        out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                             timeout=60 + 10 * budget_s * len(names))
        return json.loads(out.stdout.strip().splitlines()[-1]) if out.returncode == 0 else {}
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return {}


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ main

def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    t0 = time.time()
    tflops = []
    desc, cores = "", 1
    for _ in range(args.warmup):
        oracle_sample(wl, budget_s=1.0)
    for _ in range(args.steps):
        v, desc, cores = oracle_sample(wl, budget_s=args.ref_budget)
        tflops.append(v)
    value = statistics.median(tflops)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.time() - t0, 1)}
    print(json.dumps(line), flush=True)
    return 0


# O is written as fp32 (attn_fwd, the measured configuration) unless
# --out bf16 selects attn_fwd_bf16out.
O_DTYPE = "fp32"
# Dropout probability on the softmax weights (--dropout; attn_fwd_dropout when > 0).
DROPOUT = 0.0
DROPOUT_SEED = 0x5EED


def call_attn(q, k, v, wl, o, lse, stream):
    import blackwell_programming_gb300 as gb
    if DROPOUT > 0.0:
        return gb.attn_fwd_dropout(q, k, v, DROPOUT, DROPOUT_SEED, causal=wl.causal, scale=wl.scale, out=o, lse=lse,
                                   stream=stream)
    return gb.attn_fwd(q, k, v, causal=wl.causal, scale=wl.scale, out=o, lse=lse, stream=stream)


def o_torch_dtype():
    import torch
    return torch.bfloat16 if O_DTYPE == "bf16" else torch.float32


def algorithmic_bytes(wl) -> int:
    """Workload bytes with O in the selected output type."""
    o32 = wl.B * wl.Hq * wl.Nq * wl.d_v * 4
    return wl.algorithmic_bytes - (o32 // 2 if O_DTYPE == "bf16" else 0)


def workload_config(wl):
    return {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "Nq": wl.Nq, "Nkv": wl.Nkv,
            "d_qk": wl.d_qk, "d_v": wl.d_v, "causal": wl.causal, "scale": wl.scale,
            "inputs": "seeded N(0,1) bf16 (q x%g, k/v x%g)" % (wl.q_factor, wl.kv_factor),
            "l2": "flushed (256 MB write) before every step, outside the step events",
            "parallelism": "replicas", "o_dtype": O_DTYPE, "dropout": DROPOUT}


def measure_device(wl, steps, warmup, world, stream, flush, inputs):
    """Per-step event times (seconds) of attn_fwd with resident inputs."""
    import torch
    import blackwell_programming_gb300 as gb
    q, k, v = inputs
    o = torch.empty((wl.B, wl.Hq, wl.Nq, wl.d_v), dtype=o_torch_dtype(), device="cuda")
    lse = torch.empty((wl.B, wl.Hq, wl.Nq), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.fill_(1.0)
            call_attn(q, k, v, wl, o, lse, stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        for s, e in ev:
            flush.fill_(1.0)
            s.record(stream)
            call_attn(q, k, v, wl, o, lse, stream)
            e.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    assert gb.attn_check_device(stream) == 0, "kernel reported a timed-out wait"
    return [s.elapsed_time(e) / 1e3 for s, e in ev], o, lse


# parity bar of the path (fp32 O against the fp64 oracle)
O_MAX_ABS, O_MEAN_ABS, LSE_REL = 2e-2, 2e-3, 1e-3


def sampled_parity(wl, inp, o, lse, heads: int = 6, rows: int = 48, seed: int = 1):
    """The timed output against the fp64 oracle on sampled rows: `heads`
    random (batch, query head) pairs (8 x `rows` of them for a one-query
    decode), `rows` random query rows of each (all rows when Nq is smaller).  Returns max and mean |dO|, the max LSE error
    relative to max(1, |LSE|), the rows checked and whether the bar holds."""
    import numpy as np
    from oracle import attention_head, kv_head_of
    rng = np.random.default_rng(seed)
    if wl.Nq == 1:
        heads = max(heads, 8 * rows)     # decode: one row per head, so sample more heads
    f64 = syn.bf16_bits_to_f64
    dmax, dsum, n_el, lmax, n_rows = 0.0, 0.0, 0, 0.0, 0
    for _ in range(heads):
        b, h = int(rng.integers(wl.B)), int(rng.integers(wl.Hq))
        g = kv_head_of(h, wl.Hq, wl.Hkv)
        idx = np.sort(rng.choice(wl.Nq, size=min(rows, wl.Nq), replace=False))
        q = f64(inp.q[b, h, idx])
        k = f64(inp.k[b, g])
        v = k[:, : wl.d_v] if inp.v is None else f64(inp.v[b, g])
        if DROPOUT > 0.0:
            from oracle.dropout_fp64 import attention_dropout_head
            o_ref, lse_ref = attention_dropout_head(q, k, v, wl.causal, wl.scale, DROPOUT, DROPOUT_SEED, b, h,
                                                    row_index=idx, n_q=wl.Nq)
        else:
            o_ref, lse_ref = attention_head(q, k, v, wl.causal, wl.scale, row_index=idx, n_q=wl.Nq)
        o_gpu = o[b, h, idx].float().cpu().numpy().astype(np.float64)
        l_gpu = lse[b, h, idx].cpu().numpy().astype(np.float64)
        d = np.abs(o_gpu - o_ref)
        dmax, dsum, n_el = max(dmax, float(d.max())), dsum + float(d.sum()), n_el + d.size
        fin = np.isfinite(lse_ref)
        le = np.abs(l_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
        lmax = max(lmax, float(le.max()) if le.size else 0.0)
        n_rows += len(idx)
    mean = dsum / max(n_el, 1)
    # with dropout, kept weights are scaled by the keep factor, and so is the O bar
    f = 1.0
    if DROPOUT > 0.0:
        from oracle.dropout_fp64 import drop_threshold, keep_scale
        f = keep_scale(drop_threshold(DROPOUT))
    bar = {"max_abs_dO": O_MAX_ABS * f, "mean_abs_dO": O_MEAN_ABS * f, "lse_rel": LSE_REL}
    return {"max_abs_dO": dmax, "mean_abs_dO": mean, "max_lse_err": lmax, "rows": n_rows, "bar": bar,
            "ok": bool(dmax <= bar["max_abs_dO"] and mean <= bar["mean_abs_dO"] and lmax <= LSE_REL)}


def link_bandwidth(nbytes: int = 256 << 20, reps: int = 5):
    """Plain pinned host<->device copy bandwidth (GB/s, best of `reps`): host
    to device, device to host, and both directions at once on two streams."""
    import torch
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def best(fn):
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            fn()
            for st in (s1, s2):
                torch.cuda.current_stream().wait_stream(st)
            b.record()
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b) / 1e3)
        return min(t)

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    return {"h2d_gbs": nbytes / best(h2d) / 1e9, "d2h_gbs": nbytes / best(d2h) / 1e9,
            "bidir_gbs": 2 * nbytes / best(both) / 1e9, "bytes": nbytes}


def roofline_for(wl, per_launch: float, peaks, peak_src: str):
    """The roofline object of the attention workload's dominant kernel."""
    flops = wl.flops
    kind = ("decode" if wl.Nq == 1 else "latent_prefill") if wl.d_qk == 576 else "prefill"
    if kind in ("prefill", "latent_prefill"):
        achieved = flops / per_launch / 1e12
        kname = {64: "prefill_kernel<64>", 128: "prefill_kernel<128>"}.get(wl.d_qk, "latent_pair_kernel (prefill mode)")
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "peak_source": peak_src + " bf16_tflops (burst)",
                "kernel": kname, "algorithmic_flops_per_launch": flops}
    else:
        achieved = algorithmic_bytes(wl) / per_launch / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": peak_src + " hbm_gbs",
                "kernel": "latent_pair_kernel (decode mode) + combine_pair_kernel (one step)",
                "algorithmic_bytes_per_launch": algorithmic_bytes(wl),
                "tensor_tflops": flops / per_launch / 1e12}
    traffic_key = wl.name + ("_dropout%g" % DROPOUT if DROPOUT > 0.0 else "")
    roof["traffic"] = committed_traffic(kind, traffic_key) if O_DTYPE == "fp32" else None
    return roof, kind


def device_inputs(wl):
    """Seeded inputs of the workload: host bits, pinned host tensors and device tensors."""
    import numpy as np
    import torch
    inp = syn.make_inputs(wl)
    hq = torch.from_numpy(inp.q.view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = torch.from_numpy(inp.k.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = None if inp.v is None else torch.from_numpy(inp.v.view(np.int16)).view(torch.bfloat16).pin_memory()
    q, k = hq.cuda(), hk.cuda()
    v = k[..., : wl.d_v] if hv is None else hv.cuda()
    return inp, (hq, hk, hv), (q, k, v)


def also_entry(name, steps, warmup, world, stream, flush, peaks, peak_src):
    """Another workload of the path timed in the same run (device value,
    roofline and sampled parity; no CPU or host-buffer legs)."""
    wl = syn.WORKLOADS[name]
    inp, _, dev = device_inputs(wl)
    times, o, lse = measure_device(wl, steps, warmup, world, stream, flush, dev)
    per_launch = reduce_max(sum(times), world) / steps
    roof, _ = roofline_for(wl, per_launch, peaks, peak_src)
    return {"workload": name, "config": workload_config(wl), "ms_per_step": per_launch * 1e3,
            "value": aggregate(wl.flops, per_launch, world) / 1e12, "unit": "TFLOP/s", "roofline": roof,
            "step_ms": {"min": min(times) * 1e3, "median": statistics.median(times) * 1e3, "max": max(times) * 1e3},
            "parity": sampled_parity(wl, inp, o, lse), "gpu_launches": (2 if wl.Nq == 1 and wl.d_qk == 576 else 1) * steps}


E2E_SCHEDULE = "per step: H2D of its inputs, the call, D2H of its results; three streams, two device slots"
E2E_SERIAL = False


def pipelined_steps(steps, warmup, copy_in, compute, copy_out, nbuf=2):
    """Time `steps` end-to-end steps as a serving loop runs them: each step
    copies its inputs from pinned host memory into device slot i % nbuf
    (copy_in), runs the library call on that slot (compute) and copies its
    results back to pinned host memory (copy_out), on three streams, so one
    step's copies overlap its neighbours' compute.  Events keep a slot from
    being refilled before its compute and its copy-out are done.  Returns the
    seconds from the first copy in to the last copy out."""
    import torch
    if E2E_SERIAL:
        # one stream: each step's copies and call run back to back
        nbuf = 1
        s_in = s_c = s_out = torch.cuda.Stream()
    else:
        s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(nbuf)]
    c_done = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]

    def run(n):
        for i in range(n):
            b = i % nbuf
            with torch.cuda.stream(s_in):
                if i >= nbuf:
                    s_in.wait_event(c_done[b])
                copy_in(b)
                in_done[b].record(s_in)
            with torch.cuda.stream(s_c):
                s_c.wait_event(in_done[b])
                if i >= nbuf:
                    s_c.wait_event(out_done[b])
                compute(b, s_c)
                c_done[b].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(c_done[b])
                copy_out(b)
                out_done[b].record(s_out)

    run(warmup)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    run(steps)
    end.record(s_out)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def measure_e2e(wl, steps, warmup, stream, host):
    """Same metric with pinned host buffers: per step H2D of Q, K, V, the
    attention call, D2H of O and LSE (pipelined over steps, two slots)."""
    import torch
    hq, hk, hv = host
    nb = 2
    dq = [torch.empty_like(hq, device="cuda") for _ in range(nb)]
    dk = [torch.empty_like(hk, device="cuda") for _ in range(nb)]
    dv = [torch.empty_like(hv, device="cuda") for _ in range(nb)] if hv is not None else None
    ho = [torch.empty((wl.B, wl.Hq, wl.Nq, wl.d_v), dtype=o_torch_dtype()).pin_memory() for _ in range(nb)]
    hl = [torch.empty((wl.B, wl.Hq, wl.Nq), dtype=torch.float32).pin_memory() for _ in range(nb)]
    o = [torch.empty_like(ho[0], device="cuda") for _ in range(nb)]
    lse = [torch.empty_like(hl[0], device="cuda") for _ in range(nb)]

    def copy_in(b):
        dq[b].copy_(hq, non_blocking=True)
        dk[b].copy_(hk, non_blocking=True)
        if dv is not None:
            dv[b].copy_(hv, non_blocking=True)

    def compute(b, s):
        v = dv[b] if dv is not None else dk[b][..., : wl.d_v]
        call_attn(dq[b], dk[b], v, wl, o[b], lse[b], s)

    def copy_out(b):
        ho[b].copy_(o[b], non_blocking=True)
        hl[b].copy_(lse[b], non_blocking=True)

    secs = pipelined_steps(steps, warmup, copy_in, compute, copy_out, nb)
    h2d = hq.numel() * 2 + hk.numel() * 2 + (hv.numel() * 2 if hv is not None else 0)
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * 4
    return secs, h2d, d2h


def run_ours(args, wl):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    import blackwell_programming_gb300 as gb
    gb.build()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, cores = oracle_sample(wl, budget_s=args.ref_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "cpu_model": cpu_model(), "single_thread": single_thread_oracle()}

    inp, (hq, hk, hv), dev = device_inputs(wl)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    peaks, peak_src = load_peaks()
    also_names = [] if args.no_also else [n for n in args.also.split(",") if n and n != wl.name]

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = ClockSampler(int(vis[local]) if local < len(vis) and vis[local].strip().isdigit() else local)
    clocks.start()
    times, o, lse = measure_device(wl, args.steps, args.warmup, world, stream, flush, dev)
    also = [also_entry(n, args.steps, args.warmup, world, stream, flush, peaks, peak_src) for n in also_names]
    clk = clocks.stop()
    total = sum(times)
    t_max = reduce_max(total, world)
    flops = wl.flops
    value = aggregate(flops * args.steps, t_max, world) / 1e12
    parity = sampled_parity(wl, inp, o, lse) if rank == 0 else None
    del o, lse

    e2e = None
    if not args.no_e2e:
        e2e_secs, h2d, d2h = measure_e2e(wl, args.steps, args.warmup, stream, (hq, hk, hv))
        e2e_max = reduce_max(e2e_secs, world)
        e2e = {"value": aggregate(flops * args.steps, e2e_max, world) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "schedule": E2E_SCHEDULE}
        link = link_bandwidth()
        moved = (h2d + d2h) * args.steps / e2e_max / 1e9
        e2e["link"] = dict(link, achieved_gbs=moved, frac_of_bidir=moved / link["bidir_gbs"])

    per_launch = total / args.steps
    roof, kind = roofline_for(wl, per_launch, peaks, peak_src)
    launches = (2 if kind == "decode" else 1) * args.steps + sum(a["gpu_launches"] for a in also)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": workload_config(wl), "roofline": roof, "cpu_baseline": cpu,
                "e2e": e2e, "parity": parity,
                "gpu_launches": launches, "clocks": clk,
                "step_ms": {"min": min(times) * 1e3, "median": statistics.median(times) * 1e3,
                            "max": max(times) * 1e3}}
        if also:
            line["also"] = also
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------- projection GEMM

METRIC_GEMM = "projection GEMM TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak"
_GEMM_SAMPLE = {}


def gemm_oracle_sample(gw, budget_s: float):
    """Time the fp64 GEMM oracle on whole rows of the workload, bounded in time."""
    from oracle import gemm_nt
    if gw.name not in _GEMM_SAMPLE:
        # the first 256 rows of A and all of B, exactly as the GPU run draws them
        rows = min(gw.M, 256)
        a = syn.f32_to_bf16_bits(syn.normals_f32(gw.seed, 0, rows * gw.K)).reshape(rows, gw.K)
        b = syn.f32_to_bf16_bits(syn.normals_f32(gw.seed, gw.M * gw.K, gw.N * gw.K)).reshape(gw.N, gw.K)
        _GEMM_SAMPLE[gw.name] = (syn.bf16_bits_to_f64(a), syn.bf16_bits_to_f64(b))
    a64, b64 = _GEMM_SAMPLE[gw.name]
    rows, flops, t0 = 0, 0.0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s and rows < a64.shape[0]:
        blk = a64[rows:rows + 16]
        gemm_nt(blk, b64)
        rows += blk.shape[0]
        flops += 2.0 * blk.shape[0] * gw.N * gw.K
    secs = time.perf_counter() - t0
    return flops / secs / 1e12, "%d of %d rows of %s (all %d columns), fp64 numpy" % (rows, gw.M, gw.name, gw.N), \
        os.cpu_count() or 1


def gemm_config(gw):
    return {"workload": gw.name, "M": gw.M, "N": gw.N, "K": gw.K, "a": "bf16 [M, K]", "b": "bf16 [N, K]",
            "c": "bf16 [M, N]", "inputs": "seeded N(0,1) bf16",
            "l2": "flushed (256 MB write) before every step, outside the step events", "parallelism": "replicas"}


def run_gemm_reference(args, gw):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    t0 = time.time()
    vals, desc, cores = [], "", 1
    for _ in range(args.warmup):
        gemm_oracle_sample(gw, 0.5)
    for _ in range(args.steps):
        v, desc, cores = gemm_oracle_sample(gw, args.ref_budget)
        vals.append(v)
    value = statistics.median(vals)
    print(json.dumps({"impl": "reference", "metric": METRIC_GEMM, "value": value, "unit": "TFLOP/s",
                      "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": gemm_config(gw),
                      "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                       "sample": desc},
                      "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                      "wall_s": round(time.time() - t0, 1)}), flush=True)
    return 0


def run_gemm_ours(args, gw):
    import numpy as np
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    import blackwell_programming_gb300 as gb
    gb.build()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, cores = gemm_oracle_sample(gw, args.ref_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    a_bits, b_bits = syn.make_gemm_inputs(gw)
    ha = torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hb = torch.from_numpy(b_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    a, b = ha.cuda(), hb.cuda()
    c = torch.empty((gw.M, gw.N), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = ClockSampler(int(vis[local]) if local < len(vis) and vis[local].strip().isdigit() else local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            gb.gemm_nt(a, b, out=c, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        for s_ev, e_ev in ev:
            flush.fill_(1.0)
            s_ev.record(stream)
            gb.gemm_nt(a, b, out=c, stream=stream)
            e_ev.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    assert gb.attn_check_device(stream) == 0, "kernel reported a timed-out wait"
    clk = clocks.stop()
    times = [s_ev.elapsed_time(e_ev) / 1e3 for s_ev, e_ev in ev]
    total = sum(times)
    t_max = reduce_max(total, world)
    value = aggregate(gw.flops * args.steps, t_max, world) / 1e12

    e2e = None
    if not args.no_e2e:
        hc = [torch.empty((gw.M, gw.N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        da = [torch.empty_like(a) for _ in range(2)]
        db = [torch.empty_like(b) for _ in range(2)]
        dc = [c, torch.empty_like(c)]

        def copy_in(i):
            da[i].copy_(ha, non_blocking=True)
            db[i].copy_(hb, non_blocking=True)

        def copy_out(i):
            hc[i].copy_(dc[i], non_blocking=True)

        secs = pipelined_steps(args.steps, args.warmup, copy_in,
                               lambda i, s: gb.gemm_nt(da[i], db[i], out=dc[i], stream=s), copy_out)
        e2e_max = reduce_max(secs, world)
        e2e = {"value": aggregate(gw.flops * args.steps, e2e_max, world) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": 2 * (gw.M + gw.N) * gw.K, "d2h_bytes_per_step": 2 * gw.M * gw.N,
               "schedule": E2E_SCHEDULE}

    peaks, peak_src = load_peaks()
    per_launch = total / args.steps
    achieved = gw.flops / per_launch / 1e12
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "peak_source": peak_src + " bf16_tflops (burst)",
            "kernel": "gemm_kernel", "algorithmic_flops_per_launch": gw.flops,
            "traffic": committed_traffic("gemm", gw.name)}
    if rank == 0:
        print(json.dumps({"metric": METRIC_GEMM, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                          "config": gemm_config(gw), "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                          "gpu_launches": args.steps, "clocks": clk,
                          "step_ms": {"min": min(times) * 1e3, "median": statistics.median(times) * 1e3,
                                      "max": max(times) * 1e3}}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------ attention layer slice

METRIC_LAYER = "attention layer slice TFLOP/s (QKV GEMM + attention + O GEMM, bf16, 1 GB300)"
_LAYER_SAMPLE = {}


def layer_oracle_sample(lw, budget_s: float):
    """Time the fp64 layer oracle on sequence 0 of the workload: its K and V
    projections, then blocks of 32 query tokens (Q projection, attention
    rows of every head, O projection) until the budget is spent.  FLOPs are
    credited as the GPU line counts them (per token, the causal attention's
    halved average)."""
    import numpy as np
    from oracle import attention_head, gemm_nt, kv_head_of, round_bf16
    if lw.name not in _LAYER_SAMPLE:
        N, D = lw.N, lw.d_model
        x = syn.f32_to_bf16_bits(syn.normals_f32(lw.seed, 0, N * D)).reshape(N, D)
        x_all = lw.B * lw.N * D
        nw = lw.n_qkv * D
        wq = syn._draw(lw.seed, x_all, (lw.n_qkv, D), 1.0 / (D ** 0.5))
        wo = syn._draw(lw.seed, x_all + nw, (D, lw.Hq * lw.d), 1.0 / ((lw.Hq * lw.d) ** 0.5))
        _LAYER_SAMPLE[lw.name] = tuple(syn.bf16_bits_to_f64(t) for t in (x, wq, wo))
    x, wq, wo = _LAYER_SAMPLE[lw.name]
    Hq, Hkv, d, N = lw.Hq, lw.Hkv, lw.d, lw.N
    t0 = time.perf_counter()
    kv = round_bf16(gemm_nt(x, wq[Hq * d:]))
    flops = 2.0 * N * 2 * Hkv * d * lw.d_model
    per_tok = 2.0 * Hq * d * lw.d_model * 2 + 4.0 * Hq * d * N / (2.0 if lw.causal else 1.0)
    done = 0
    while time.perf_counter() - t0 < budget_s and done < N:
        toks = list(range(done, min(N, done + 32)))
        q = round_bf16(gemm_nt(x[toks], wq[:Hq * d]))
        o = np.zeros((len(toks), Hq * d))
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            o[:, h * d:(h + 1) * d], _ = attention_head(q[:, h * d:(h + 1) * d], kv[:, g * d:(g + 1) * d],
                                                        kv[:, (Hkv + g) * d:(Hkv + g + 1) * d], lw.causal,
                                                        lw.scale, row_index=toks, n_q=N)
        gemm_nt(round_bf16(o), wo)
        done += len(toks)
        flops += per_tok * len(toks)
    secs = time.perf_counter() - t0
    return flops / secs / 1e12, ("sequence 0 of %s: K/V projections of all %d tokens, then %d query tokens "
                                 "through Q projection, attention and O projection, fp64 numpy") % (
        lw.name, N, done), os.cpu_count() or 1


def layer_config(lw):
    return {"workload": lw.name, "B": lw.B, "N": lw.N, "d_model": lw.d_model, "Hq": lw.Hq, "Hkv": lw.Hkv,
            "d": lw.d, "causal": lw.causal, "scale": lw.scale,
            "x": "bf16 [B*N, d_model]", "w_qkv": "bf16 [(Hq+2Hkv)*d, d_model]", "w_o": "bf16 [d_model, Hq*d]",
            "qkv": "bf16 token-major, read in place by the attention", "o": "bf16 token-major", "y": "bf16",
            "inputs": "seeded N(0,1) X, N(0,1)/sqrt(fan-in) weights, bf16",
            "l2": "flushed (256 MB write) before every step, outside the step events", "parallelism": "replicas"}


def run_layer_reference(args, lw):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    t0 = time.time()
    vals, desc, cores = [], "", 1
    for _ in range(args.warmup):
        layer_oracle_sample(lw, 0.5)
    for _ in range(args.steps):
        v, desc, cores = layer_oracle_sample(lw, args.ref_budget)
        vals.append(v)
    value = statistics.median(vals)
    print(json.dumps({"impl": "reference", "metric": METRIC_LAYER, "value": value, "unit": "TFLOP/s",
                      "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": layer_config(lw),
                      "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                       "sample": desc},
                      "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                      "wall_s": round(time.time() - t0, 1)}), flush=True)
    return 0


def run_layer_ours(args, lw):
    import numpy as np
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    import blackwell_programming_gb300 as gb
    gb.build()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, cores = layer_oracle_sample(lw, args.ref_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    B, N, D, Hq, Hkv, d = lw.B, lw.N, lw.d_model, lw.Hq, lw.Hkv, lw.d
    T, nqkv, nq = B * N, lw.n_qkv, lw.Hq * lw.d
    x_bits, wq_bits, wo_bits = syn.make_layer_inputs(lw)
    pin = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hx, hwq, hwo = pin(x_bits), pin(wq_bits), pin(wo_bits)
    x, wq, wo = hx.cuda(), hwq.cuda(), hwo.cuda()
    qkv = torch.empty((T, nqkv), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((T, nq), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    L = gb.load_library()
    import ctypes
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + 2 * off)

    def qkv_gemm():
        return L.gemm_bf16_nt(P(x), P(wq), P(qkv), T, nqkv, D, 0, ctypes.c_void_p(sp))

    def attention():
        return L.attn_fwd_bshd(P(qkv), P(qkv, nq), P(qkv, nq + Hkv * d), P(o), None, B, Hq, Hkv, N, N, d,
                               nqkv, nqkv, nqkv, nq, 0, 1 if lw.causal else 0, ctypes.c_float(lw.scale),
                               ctypes.c_void_p(sp))

    def o_gemm():
        return L.gemm_bf16_nt(P(o), P(wo), P(y), T, D, nq, 0, ctypes.c_void_p(sp))

    parts = (("qkv_gemm", qkv_gemm), ("attention", attention), ("o_gemm", o_gemm))
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = ClockSampler(int(vis[local]) if local < len(vis) and vis[local].strip().isdigit() else local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            for _, fn in parts:
                assert fn() == 0
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        for e in ev:
            flush.fill_(1.0)
            e[0].record(stream)
            for i, (_, fn) in enumerate(parts):
                fn()
                e[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    assert gb.attn_check_device(stream) == 0, "kernel reported a timed-out wait"
    clk = clocks.stop()
    part_s = [[e[i].elapsed_time(e[i + 1]) / 1e3 for i in range(3)] for e in ev]
    times = [sum(p) for p in part_s]
    total = sum(times)
    t_max = reduce_max(total, world)
    value = aggregate(lw.flops * args.steps, t_max, world) / 1e12

    e2e = None
    if not args.no_e2e:
        hy = [torch.empty((T, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        dx = [torch.empty_like(x) for _ in range(2)]
        dqkv = [qkv, torch.empty_like(qkv)]
        do_ = [o, torch.empty_like(o)]
        dy = [y, torch.empty_like(y)]

        def copy_in(i):
            dx[i].copy_(hx, non_blocking=True)

        def compute(i, s):
            st = gb.attn_layer_raw(dx[i].data_ptr(), wq.data_ptr(), wo.data_ptr(), dqkv[i].data_ptr(),
                                   do_[i].data_ptr(), dy[i].data_ptr(), 0, B, N, D, Hq, Hkv, d, lw.causal, lw.scale,
                                   False, s.cuda_stream)
            assert st == 0

        def copy_out(i):
            hy[i].copy_(dy[i], non_blocking=True)

        secs = pipelined_steps(args.steps, args.warmup, copy_in, compute, copy_out)
        e2e_max = reduce_max(secs, world)
        e2e = {"value": aggregate(lw.flops * args.steps, e2e_max, world) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": 2 * T * D, "d2h_bytes_per_step": 2 * T * D,
               "api": "attn_layer_fwd (one call), weights resident", "schedule": E2E_SCHEDULE}

    # per-part FLOPs in the line's convention; the roofline is the slowest part's kernel
    att = 4.0 * B * Hq * N * N * d / (2.0 if lw.causal else 1.0)
    pflops = {"qkv_gemm": 2.0 * T * nqkv * D, "attention": att, "o_gemm": 2.0 * T * D * nq}
    mean_s = {name: sum(p[i] for p in part_s) / args.steps for i, (name, _) in enumerate(parts)}
    top = max(mean_s, key=mean_s.get)
    peaks, peak_src = load_peaks()
    achieved = pflops[top] / mean_s[top] / 1e12
    kern = {"qkv_gemm": ("gemm_kernel", "gemm", "gemm_qkv_proj"), "attention": ("prefill_kernel", "prefill", None),
            "o_gemm": ("gemm_kernel", "gemm", None)}[top]
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "peak_source": peak_src + " bf16_tflops (burst)",
            "kernel": kern[0] + " (" + top + ")", "algorithmic_flops_per_launch": pflops[top],
            "traffic": committed_traffic(kern[1], kern[2]) if kern[2] else None}
    if rank == 0:
        print(json.dumps({"metric": METRIC_LAYER, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic", "config": layer_config(lw), "roofline": roof, "cpu_baseline": cpu,
                          "e2e": e2e, "gpu_launches": 3 * args.steps, "clocks": clk,
                          "parts": {name: {"ms": mean_s[name] * 1e3,
                                           "tflops": pflops[name] / mean_s[name] / 1e12} for name, _ in parts},
                          "step_ms": {"min": min(times) * 1e3, "median": statistics.median(times) * 1e3,
                                      "max": max(times) * 1e3}}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(syn.WORKLOADS) + sorted(syn.GEMM_WORKLOADS) + sorted(syn.LAYER_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--also", default=None,
                    help="comma-separated attention workloads also timed in the same run (device value, roofline, "
                         "sampled parity); default: the long-context and decode workloads when the default "
                         "workload runs unmodified")
    ap.add_argument("--no-also", action="store_true", help="time the named workload only")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch size (profiling cases)")
    ap.add_argument("--heads", type=int, default=None, help="override the workload's query heads (profiling cases)")
    ap.add_argument("--out", default="fp32", choices=["fp32", "bf16"], help="O output type (fp32 is the measured configuration)")
    ap.add_argument("--dropout", type=float, default=0.0, help="dropout probability on the softmax weights (prefill shapes)")
    ap.add_argument("--e2e-schedule", default="pipelined", choices=["pipelined", "serial"],
                    help="e2e steps overlapped on three streams (default) or back to back on one")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)      # at least three untimed warm-up steps
    global O_DTYPE, DROPOUT, E2E_SERIAL, E2E_SCHEDULE
    O_DTYPE = args.out
    if args.e2e_schedule == "serial":
        E2E_SERIAL = True
        E2E_SCHEDULE = "per step: H2D of its inputs, the call, D2H of its results; one stream, back to back"
    DROPOUT = args.dropout
    if DROPOUT > 0.0 and O_DTYPE != "fp32":
        ap.error("--dropout writes fp32 O")
    if args.workload in syn.GEMM_WORKLOADS:
        gw = syn.GEMM_WORKLOADS[args.workload]
        return run_gemm_reference(args, gw) if args.impl == "reference" else run_gemm_ours(args, gw)
    if args.workload in syn.LAYER_WORKLOADS:
        lw = syn.LAYER_WORKLOADS[args.workload]
        if args.batch is not None:
            lw = lw.with_sizes(B=args.batch, name="%s_B%d" % (lw.name, args.batch))
        return run_layer_reference(args, lw) if args.impl == "reference" else run_layer_ours(args, lw)
    wl = syn.WORKLOADS[args.workload]
    if args.batch is not None:
        wl = wl.with_sizes(B=args.batch, name="%s_B%d" % (wl.name, args.batch))
    if args.heads is not None:
        wl = wl.with_sizes(Hq=args.heads, name="%s_H%d" % (wl.name, args.heads))
    if args.also is None:
        plain = (args.workload == DEFAULT_WORKLOAD and args.batch is None and args.heads is None
                 and DROPOUT == 0.0 and O_DTYPE == "fp32")
        args.also = "long_causal_d128,decode_d576" if plain else ""
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
