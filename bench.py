"""Benchmark of the Muse Glimmer decode output stage on GB300.

One step = one forward of the whole output stage (final RMSNorm, Q5_K LM-head
matvec, scale, soft cap, argmax) over one batch of synthetic input.  Default
workload: the full LM head, batch 1 (202,048 x 6,656 Q5_K weights, ~925 MB,
rows 0/777/200001 boosted so the cap bites).

Prints ONE JSON line (rank 0).  `value` is the achieved algorithmic bandwidth
(Q5_K weights + hidden + gamma + logits bytes per forward / device time per
forward), GB/s, with inputs resident in HBM.  Extra keys: us_per_forward,
logits_per_s, roofline (dominant kernel vs the measured HBM copy peak),
cpu_baseline (the f64 oracle on this host's cores, a bounded row sample), e2e
(the same metric through the host-buffer C-ABI call, copies included), clocks
sampled during the timed region, gpu_launches.

--impl reference times the f64 CPU oracle, as it stands, on the host cores, on
the same workload and metric.

Multi-GPU: each rank runs an independent replica of the output stage (no
sharding, no collective); --gpus N runs N of them, value = all ranks' bytes /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024   # GB300 L2 (per nvidia-smi/cudaDeviceProp order of magnitude)


def _measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (200 ms period)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ncu summaries that carry a per-launch DRAM traffic figure:
# (kernel path, workload) -> (file, kernel sources)
_B1_SRC = ("gemv_b1.cu", "common.cuh", "ptx.cuh")
_TC_SRC = ("gemm_tc.cu", "common.cuh", "ptx.cuh", "tc.cuh")
_PROFILED = {("gemv_b1", "lmhead_b1"): ("gemv_b1_lmhead.md", _B1_SRC),
             ("gemv_b1", "lmhead_q4k_b1"): ("gemv_b1_lmhead_q4k.md", _B1_SRC),
             ("gemm_tc", "lmhead_b8"): ("gemm_tc_lmhead_b8.md", _TC_SRC),
             ("gemm_tc", "sweep_b2"): ("gemm_tc_sweep_b2.md", _TC_SRC),
             ("gemm_tc", "dflash_verify_b16"): ("gemm_tc_dflash_verify_b16.md", _TC_SRC),
             ("gemm_tc", "sweep_b32"): ("gemm_tc_sweep_b32.md", _TC_SRC),
             ("gemv_b1_split", "ffn_down_q4k"): ("gemv_b1_split_ffn_down_q4k.md", _B1_SRC),
             ("gemm_tc", "lmhead_q4k_b8"): ("gemm_tc_lmhead_q4k_b8.md", _TC_SRC),
             ("gemv_b1_group", "ffn_gate_up_q4k"): ("gemv_b1_group_ffn_gate_up_q4k.md", _B1_SRC),
             ("gemv_b1", "tiny"): ("gemv_b1_small_shapes.md", _B1_SRC),
             ("gemv_b1", "attn_q"): ("gemv_b1_small_shapes.md", _B1_SRC),
             ("gemv_b1", "attn_k"): ("gemv_b1_small_shapes.md", _B1_SRC),
             ("gemv_b1", "attn_o"): ("gemv_b1_small_shapes.md", _B1_SRC),
             ("gemv_b1_group", "attn_qkvg"): ("gemv_b1_group_attn_qkvg.md", _B1_SRC)}


def kernel_code(name: str) -> str:
    """A kernel source file's code with comments and blank lines removed, the
    text the profile summaries' kernel-source hash covers (a comment edit does
    not change the profiled kernel)."""
    import re
    with open(os.path.join(ROOT, "q5_lm_head_gb300", "csrc", name)) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def _profile_fields(path: str, workload: str):
    """(kernel-source digest, traffic bytes per launch for `workload`) from an
    ncu summary: the plain traffic line, or the workload's own line in a
    summary covering several workloads; None for what is missing."""
    digest, traffic = None, None
    mine = f"traffic_bytes_per_launch[{workload}]:"
    with open(path) as fh:
        for line in fh:
            if line.startswith("kernel-source:"):
                digest = line.split()[1]
            elif line.startswith("traffic_bytes_per_launch:") or line.startswith(mine):
                traffic = int(line.split()[1])
    return digest, traffic


def _profiled_traffic(kernel_path: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when there
    is none for this kernel/workload or the kernel source changed since."""
    import hashlib
    ent = _PROFILED.get((kernel_path, workload))
    if not ent:
        return None
    h = hashlib.sha256()
    for f in ent[1]:
        h.update(kernel_code(f).encode())
    try:
        digest, traffic = _profile_fields(os.path.join(ROOT, "profiles", ent[0]), workload)
    except OSError:
        return None
    return traffic if digest and h.hexdigest().startswith(digest) else None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_aggregate(seconds: float, nbytes: int, device=None):
    """Whole-job throughput of independent replicas, one per rank: the bytes of
    every rank over the slowest rank's time (max over ranks; the identity at one
    rank).  Returns (GB/s, max seconds)."""
    import torch
    dist = torch.distributed
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    if ws > 1:
        t = torch.tensor([seconds], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        seconds = float(t.item())
    return ws * nbytes / seconds / 1e9, seconds


def _oracle_rate(wl, hidden, gamma, wq, target_s: float, threads: int | None = None):
    """Time the oracle, as it stands, on a bounded sample of the workload: the
    first `rows` weight rows (all of them when they fit the time budget), run
    repeatedly for `target_s` seconds on `threads` threads (all host cores by
    default).  Returns (bytes_per_s, rows, reps, cores, secs)."""
    import numpy as np
    import oracle
    cores = threads or oracle.default_threads()
    probe = min(2048, wl.n_rows)
    t0 = time.perf_counter()
    oracle.lmhead(hidden, gamma, wq[:probe], wl.scale, wl.cap, nthreads=cores, fmt=wl.fmt)
    dt = max(time.perf_counter() - t0, 1e-6)
    rows = int(min(wl.n_rows, max(probe, probe * target_s / dt)))
    sample = np.ascontiguousarray(wq[:rows])
    reps = 0
    t0 = time.perf_counter()
    while True:                  # whole passes until the time budget is spent
        oracle.lmhead(hidden, gamma, sample, wl.scale, wl.cap, nthreads=cores, fmt=wl.fmt)
        reps += 1
        secs = time.perf_counter() - t0
        if secs >= target_s:
            break
    bytes_sample = wl.algorithmic_bytes() * (rows / wl.n_rows) * reps
    return bytes_sample / secs, rows, reps, cores, secs


def run_reference(args, wl):
    """The oracle (f64 CPU) as the reference arm."""
    import q5k_synth as synth
    ws, rank, _ = _dist()
    if rank != 0:
        return
    group = isinstance(wl, synth.GroupWorkload)
    hidden, gamma, wq = synth.group_inputs(wl) if group else synth.inputs_for(wl)
    rate_fn = _oracle_rate_group if group else _oracle_rate
    per_step = max(0.5, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        rate_fn(wl, hidden, gamma, wq, per_step * 0.2)
    rates, rows_l, secs_l, cores, reps = [], [], [], 1, 1
    for _ in range(args.steps):
        r, rows, reps, cores, secs = rate_fn(wl, hidden, gamma, wq, per_step)
        rates.append(r)
        rows_l.append(rows)
        secs_l.append(secs)
    value = statistics.median(rates) / 1e9
    sample = (f"{int(statistics.median(rows_l))} of {wl.n_rows} weight rows x batch {wl.batch}, "
              f"{reps} pass(es) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.median(secs_l) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl, ws, _l2_mode(wl)),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "Q5_K LM-head forward us and achieved HBM GB/s (% of GB300 peak), batch 1-32"


def _big(wl) -> bool:
    """Whether a workload's bytes exceed L2 enough that every forward streams from HBM."""
    return wl.algorithmic_bytes() > 2 * L2_BYTES


def _l2_mode(wl) -> str:
    return ("inputs larger than L2 (weights stream from HBM every forward)" if _big(wl) else
            "L2 flushed before every timed forward (256 MiB write, then a 256 MiB read so that no "
            "write-back lands in the timed interval; both outside it)")


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or the platform string."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def _config(wl, ws, l2_mode):
    import q5k_synth as synth
    if isinstance(wl, synth.GroupWorkload):
        return {"workload": wl.name, "matrices": [[n, r] for (n, r, _, _, _) in wl.segments], "k": wl.k,
                "batch": 1, "weights": "Q5_K 176 B / 256 weights" if wl.fmt == "q5_k" else "Q4_K 144 B / 256 weights",
                "norm": wl.norm,
                "scale_cap": [[sc, cp] for (_, _, _, sc, cp) in wl.segments], "launches": 1, "l2": l2_mode,
                "parallelism": f"replicas x{ws}"}
    return {"workload": wl.name, "n_rows": wl.n_rows, "k": wl.k, "batch": wl.batch,
            "weights": "Q5_K 176 B / 256 weights" if wl.fmt == "q5_k" else "Q4_K 144 B / 256 weights", "final_norm": wl.norm, "scale": wl.scale, "cap": wl.cap,
            "argmax": wl.argmax, "l2": l2_mode, "parallelism": f"replicas x{ws}"}


def _e2e(args, wl, head, hidden, w_d, g_d, eps, stream, ws, nbytes):
    """Same metric through the C-ABI call muse_lmhead_forward_host (its
    same-named binding, pointers only): each step copies the pinned hidden rows
    in, the kernel writes logits + argmax into pinned host memory, and the call
    waits for them.  The LMHead wrapper's tensor checks (about 4.6 us of Python
    per call) are done once, by the warm-up calls."""
    import torch
    import q5_lm_head_gb300 as mlh
    h_pin = torch.from_numpy(hidden).pin_memory()
    l_pin = torch.empty((wl.batch, wl.n_rows), dtype=torch.float32, pin_memory=True)
    a_pin = torch.empty((wl.batch,), dtype=torch.int32, pin_memory=True)
    steps = max(3, min(args.steps, 50))
    for _ in range(2):
        head.forward_host(h_pin, w_d, g_d, eps, wl.scale, wl.cap, l_pin, a_pin, stream)
    call = mlh.load_library().muse_lmhead_forward_host
    argv = (head.handle, h_pin.data_ptr(), wl.batch, None if g_d is None else g_d.data_ptr(), float(eps),
            w_d.data_ptr(), float(wl.scale), float(wl.cap), l_pin.data_ptr(), a_pin.data_ptr(), stream.cuda_stream)
    if ws > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        if call(*argv) != 0:
            raise RuntimeError("muse_lmhead_forward_host failed")
    secs = (time.perf_counter() - t0) / steps
    value, secs = replica_aggregate(secs, nbytes, w_d.device)
    h2d = wl.batch * wl.k * 4
    d2h = wl.batch * wl.n_rows * 4 + wl.batch * 4
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "us_per_forward": round(secs * 1e6, 2)}


def _hold_cycles(steps: int, host_s_per_step: float = 0.3e-3, cap_s: float = 2.0) -> int:
    """GPU cycles to sleep while the host enqueues `steps` timed forwards
    (host_s_per_step of host work per step, at up to 2.1 GHz)."""
    return int(min(cap_s, host_s_per_step * (steps + 4)) * 2.1e9)


def _graph_times(fwd, stream, steps, l2_flush):
    """Median device time of one forward replayed from a captured CUDA graph,
    L2 flushed before each replay; None when capture fails."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fwd()
        torch.cuda.synchronize()
    except RuntimeError as e:   # capture unsupported: report, do not fail the bench
        return {"error": str(e).splitlines()[0][:200]}
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda._sleep(_hold_cycles(steps))
        for i in range(steps):
            l2_flush(i)
            starts[i].record(stream)
            g.replay()
            ends[i].record(stream)
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) * 1e3 for s, e in zip(starts, ends)]
    return {"us_per_forward_median": round(statistics.median(per), 2), "steps": steps}


def _e2e_group(args, wl, head, hidden, segs, g_d, eps, stream, nbytes):
    """The grouped forward end to end through muse_lmhead_forward_group_host:
    each step copies the pinned hidden row in, the kernel writes every
    matrix's output into pinned host buffers, and the call waits for it."""
    import torch
    h_pin = torch.from_numpy(hidden).reshape(-1).pin_memory()
    host_segs = [(w, n, sc, cp, torch.empty((n,), dtype=torch.float32, pin_memory=True))
                 for (w, n, sc, cp, _) in segs]
    steps = max(3, min(args.steps, 50))
    for _ in range(2):
        head.forward_group_host(h_pin, host_segs, g_d, eps, stream)
    t0 = time.perf_counter()
    for _ in range(steps):
        head.forward_group_host(h_pin, host_segs, g_d, eps, stream)
    secs = (time.perf_counter() - t0) / steps
    value, secs = replica_aggregate(secs, nbytes, g_d.device if g_d is not None else segs[0][0].device)
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": wl.k * 4,
            "d2h_bytes_per_step": wl.n_rows * 4, "us_per_forward": round(secs * 1e6, 2)}


def _e2e_logprobs(args, wl, head, hidden, w_d, g_d, eps, stream, nbytes):
    """The logprobs forward end to end: pinned hidden rows copied in, logprobs,
    lse and argmax copied out to pinned host buffers, stream synchronised."""
    import torch
    h_pin = torch.from_numpy(hidden).pin_memory()
    h_dev = torch.empty(h_pin.shape, dtype=torch.float32, device=w_d.device)
    lp_pin = torch.empty((wl.batch, wl.n_rows), dtype=torch.float32, pin_memory=True)
    lse_pin = torch.empty((wl.batch,), dtype=torch.float32, pin_memory=True)
    am_pin = torch.empty((wl.batch,), dtype=torch.int32, pin_memory=True)
    steps = max(3, min(args.steps, 50))

    def step():
        with torch.cuda.stream(stream):
            h_dev.copy_(h_pin, non_blocking=True)
            lp, lse, am = head.forward_logprobs(h_dev, w_d, g_d, eps, wl.scale, wl.cap, True, stream=stream)
            lp_pin.copy_(lp, non_blocking=True)
            lse_pin.copy_(lse, non_blocking=True)
            am_pin.copy_(am, non_blocking=True)
        stream.synchronize()

    for _ in range(2):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    secs = (time.perf_counter() - t0) / steps
    value, secs = replica_aggregate(secs, nbytes, h_dev.device)
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": wl.batch * wl.k * 4,
            "d2h_bytes_per_step": wl.batch * (wl.n_rows + 2) * 4, "us_per_forward": round(secs * 1e6, 2)}


def _oracle_rate_group(g, hidden, gamma, wqs, target_s: float, threads: int | None = None):
    """The oracle, as it stands, over every matrix of a group, whole passes for
    `target_s` seconds.  Returns (bytes_per_s, rows, reps, cores, secs)."""
    import oracle
    cores = threads or oracle.default_threads()
    reps = 0
    t0 = time.perf_counter()
    while True:
        for w, (_, n, _, sc, cp) in zip(wqs, g.segments):
            oracle.lmhead(hidden, gamma, w, sc, cp, nthreads=cores, fmt=g.fmt)
        reps += 1
        secs = time.perf_counter() - t0
        if secs >= target_s:
            break
    return g.algorithmic_bytes() * reps / secs, g.n_rows, reps, cores, secs


# The whole metric in one run ("batch 1-32" over the five workloads): each entry
# (workload, what it stands for).  The 202,048-row entries share two weight
# matrices, generated once: the boosted one (rows 0, 777, 200001) for the
# batch-1 / batch-8 / DFlash entries and the plain one for the batch sweep.
SWEEP = (("lmhead_b1", "full LM head, batch 1"), ("lmhead_b8", "full LM head, serving batch 8"),
         ("sweep_b2", "batch sweep"), ("sweep_b4", "batch sweep"), ("sweep_b8", "batch sweep"),
         ("sweep_b16", "batch sweep"), ("sweep_b32", "batch sweep"),
         ("dflash_verify_b16", "DFlash verify batch"),
         ("tiny", "tiny head, 2,048 rows"), ("attn_q", "attention projection"), ("attn_k", "attention projection"),
         ("attn_v", "attention projection"), ("attn_o", "attention projection"),
         ("attn_qkvg", "Q/K/V/gate group, one launch"))


def _time_forwards(fwd, stream, n, l2_flush=None):
    """Per-forward device times (ms) of n forwards enqueued behind a sleep
    kernel (no interval waits on the host), L2 flushed before each one when a
    flush is given."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(_hold_cycles(n, 0.1e-3, 1.0))
        for i in range(n):
            if l2_flush is not None:
                l2_flush(i)
            starts[i].record(stream)
            fwd()
            ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def _time_back_to_back(fwd, stream, n):
    """Device time (ms) per forward of n forwards enqueued back to back
    behind a sleep kernel, with one event before the first and one after the
    last (none in between)."""
    import torch
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(_hold_cycles(n, 0.1e-3, 1.0))
        t0.record(stream)
        for _ in range(n):
            fwd()
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / n


def run_sweep(args, dev, stream, local, peak, peak_kind, preset=None):
    """Every workload of the metric on this GPU, one entry each: device time
    per forward (CUDA events; inputs larger than L2, or L2 flushed before
    every forward), algorithmic GB/s, fraction of the measured copy peak,
    kernel path and the clocks sampled while it ran."""
    import torch
    import q5k_synth as synth
    import q5_lm_head_gb300 as mlh
    eps = synth.RMS_EPS
    mats = dict(preset or {})          # (weight tag, boosted rows) -> device matrix

    def weights(wl):
        key = (wl.weight_tag, wl.boost_rows)
        if key not in mats:
            mats[key] = torch.from_numpy(synth.weights_for(wl)).to(dev)
        return mats[key]

    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    evict = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def l2_flush(i):
        flush.fill_(i & 0xFF)
        evict.sum()

    entries = []
    for name, what in SWEEP:
        group = name in synth.GROUPS
        wl = synth.GROUPS[name] if group else synth.WORKLOADS[name]
        if group:
            hidden, gamma, wq = synth.group_inputs(wl)
            w_d = [torch.from_numpy(w).to(dev) for w in wq]
            head = mlh.LMHead(1, wl.k, max_batch=1, device=local, fmt=wl.fmt)
            segs = [(w, n, sc, cp, torch.empty((n,), dtype=torch.float32, device=dev))
                    for w, (_, n, _, sc, cp) in zip(w_d, wl.segments)]
            path = "gemv_b1_group"
        else:
            hidden, gamma = synth.hidden_for(wl), synth.gamma_for(wl)
            w_d = weights(wl) if wl.n_rows == synth.VOCAB else torch.from_numpy(synth.weights_for(wl)).to(dev)
            head = mlh.LMHead(wl.n_rows, wl.k, max_batch=wl.batch, device=local, fmt=wl.fmt)
            logits = torch.empty((wl.batch, wl.n_rows), dtype=torch.float32, device=dev)
            amax = torch.empty((wl.batch,), dtype=torch.int32, device=dev) if wl.argmax else None
            path = head.path_name(wl.batch)
        h_d = torch.from_numpy(hidden).to(dev)
        g_d = None if gamma is None else torch.from_numpy(gamma).to(dev)

        def fwd():
            if group:
                head.forward_group(h_d, segs, g_d, eps, stream)
            else:
                head.forward(h_d, w_d, g_d, eps, wl.scale, wl.cap, wl.argmax, logits, amax, stream)

        big = _big(wl)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fwd()
        torch.cuda.synchronize()
        probe = _time_forwards(fwd, stream, 5, None if big else l2_flush)
        est_ms = statistics.median(probe)
        # at least args.sweep_seconds of forwards, so the clock sampler sees the GPU under load
        n = int(max(args.steps, min(20000, args.sweep_seconds * 1e3 / max(est_ms, 1e-3))))
        if not big:
            n = min(n, 400)
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        wall_ms = _time_back_to_back(fwd, stream, n) if big else None
        per = _time_forwards(fwd, stream, n, None if big else l2_flush)
        clocks = sampler.stop()
        kern_ms = (sum(per) / len(per)) if big else statistics.median(per)
        ms = wall_ms if big else kern_ms
        nbytes = wl.algorithmic_bytes()
        gbs = nbytes / (ms * 1e-3) / 1e9
        entries.append({
            "workload": name, "what": what, "batch": wl.batch, "n_rows": wl.n_rows, "k": wl.k,
            "weights": "Q5_K" if wl.fmt == "q5_k" else "Q4_K", "kernel_path": path, "forwards": n,
            "us_per_forward": round(ms * 1e3, 2),
            "us_stat": "forwards back to back, two events around the run / forwards" if big else
                       "median of per-forward CUDA-event intervals, L2 flushed before each",
            "kernel_us": round(kern_ms * 1e3, 2),
            "kernel_us_stat": "mean of per-forward CUDA-event intervals" if big else
                              "median of per-forward CUDA-event intervals, L2 flushed before each",
            "algorithmic_bytes": nbytes, "gbs": round(gbs, 1),
            "frac_of_peak": round(nbytes / (kern_ms * 1e-3) / 1e9 / peak, 4),
            "logits_per_s": round(wl.batch * wl.n_rows / (ms * 1e-3), 1),
            "traffic": _profiled_traffic(path, name), "clocks": clocks, "device_status": head.device_status()})
        head.close()
    return {"peak_gbs": peak, "peak_source": f"{peak_kind} HBM copy bandwidth", "entries": entries}


def run_ours(args, wl):
    import numpy as np
    import torch
    import q5k_synth as synth
    import q5_lm_head_gb300 as mlh
    from q5_lm_head_gb300 import _build

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(mlh.LIB_PATH):
        _build.build()
    if ws > 1:
        torch.distributed.barrier()
    mlh.load_library()

    group = isinstance(wl, synth.GroupWorkload)
    stream = torch.cuda.Stream(dev)
    eps = synth.RMS_EPS
    if group:
        hidden, gamma, wq = synth.group_inputs(wl)     # wq: one weight matrix per segment
        w_d = [torch.from_numpy(w).to(dev) for w in wq]
        head = mlh.LMHead(1, wl.k, max_batch=1, device=local, fmt=wl.fmt)
        outs = [torch.empty((n,), dtype=torch.float32, device=dev) for (_, n, _, _, _) in wl.segments]
        segs = [(w, n, sc, cp, o) for w, o, (_, n, _, sc, cp) in zip(w_d, outs, wl.segments)]
        path, launches = "gemv_b1_group", 1
    else:
        hidden, gamma, wq = synth.inputs_for(wl)
        w_d = torch.from_numpy(wq).to(dev)
        head = mlh.LMHead(wl.n_rows, wl.k, max_batch=wl.batch, device=local, fmt=wl.fmt)
        logits = torch.empty((wl.batch, wl.n_rows), dtype=torch.float32, device=dev)
        amax = torch.empty((wl.batch,), dtype=torch.int32, device=dev) if wl.argmax else None
        path, launches = head.path_name(wl.batch), head.launches_per_forward(wl.batch, wl.norm)
        if args.logprobs:           # + the apply kernel (+ a pass over the logits off the fused path)
            launches += 1 if path in ("gemv_b1", "gemv_b1_split") else 2
            path = path + "+logprobs"
            lse_d = torch.empty((wl.batch,), dtype=torch.float32, device=dev)
    h_d = torch.from_numpy(hidden).to(dev)
    g_d = None if gamma is None else torch.from_numpy(gamma).to(dev)
    big = _big(wl)
    l2_mode = _l2_mode(wl)
    flush = None if big else torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    evict = None if big else torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)

    def l2_flush(i):
        flush.fill_(i & 0xFF)
        evict.sum()

    def fwd():
        if group:
            head.forward_group(h_d, segs, g_d, eps, stream)
        elif args.logprobs:
            head.forward_logprobs(h_d, w_d, g_d, eps, wl.scale, wl.cap, wl.argmax, logits, lse_d, amax, stream)
        else:
            head.forward(h_d, w_d, g_d, eps, wl.scale, wl.cap, wl.argmax, logits, amax, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            fwd()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall_ms = None
    if flush is None:
        # the timed steps: K forwards back to back behind a sleep kernel that
        # holds the GPU while the host enqueues them (no interval waits on the
        # host), two events around the whole run and none in between
        with torch.cuda.stream(stream):
            torch.cuda._sleep(_hold_cycles(args.steps))
            t_begin.record(stream)
            for _ in range(args.steps):
                fwd()
            t_end.record(stream)
        torch.cuda.synchronize()
        wall_ms = t_begin.elapsed_time(t_end)
    with torch.cuda.stream(stream):
        # per-forward device times (the kernel-only rate of the roofline; with
        # a flush, the timed steps themselves): an event pair around each
        # forward, L2 flushed before it when the inputs fit in L2
        torch.cuda._sleep(_hold_cycles(args.steps))
        for i in range(args.steps):
            if flush is not None:
                l2_flush(i)
            starts[i].record(stream)
            fwd()
            ends[i].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]     # ms, each forward
    kern_ms = sum(per) / len(per)
    step_ms = statistics.median(per) if flush is not None else wall_ms / args.steps

    # small workloads: the same forward replayed from a CUDA graph (launch cost off the host path)
    graph = None
    if flush is not None and not args.no_graph:
        graph = _graph_times(fwd, stream, args.steps, l2_flush)
    nbytes = wl.algorithmic_bytes()
    value, step_s = replica_aggregate(step_ms * 1e-3, nbytes, dev)
    step_ms = step_s * 1e3
    status = head.device_status()

    # end to end through the host-buffer entry point: pinned hidden in, logits + argmax out
    e2e = None
    if not args.no_e2e:
        if group:
            e2e = _e2e_group(args, wl, head, hidden, segs, g_d, eps, stream, nbytes)
        elif args.logprobs:
            e2e = _e2e_logprobs(args, wl, head, hidden, w_d, g_d, eps, stream, nbytes)
        else:
            e2e = _e2e(args, wl, head, hidden, w_d, g_d, eps, stream, ws, nbytes)

    peak, peak_kind = _measured_peaks()
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Q5_K weights and N(0,1) hidden rows; no checkpoint)",
        "config": _config(wl, ws, l2_mode),
        "us_per_forward": round(step_ms * 1e3, 2),
        "us_per_forward_stat": "median of per-forward CUDA-event intervals" if flush is not None
                               else "timed wall interval / steps",
        "cuda_graph": graph,
        "logits_per_s": round(ws * wl.batch * wl.n_rows / (step_ms * 1e-3), 1),
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "kernel_path": path,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": _profiled_traffic(path, wl.name),
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "kernel": path,
                     "algorithmic_bytes_per_launch": nbytes if launches == 1 else None},
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "device_status": status,
    }
    if not group and args.logprobs:
        line["config"]["output"] = "logprobs: log-softmax of the capped logits, plus lse and argmax"
    if ws == 1 and args.sweep:
        preset = {} if group else {(wl.weight_tag, wl.boost_rows): w_d}
        line["sweep"] = run_sweep(args, dev, stream, local, peak, peak_kind, preset)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate_fn = _oracle_rate_group if group else _oracle_rate
        rate, rows, reps, cores, secs = rate_fn(wl, hidden, gamma, wq, args.cpu_seconds)
        rate1, rows1, reps1, _, secs1 = rate_fn(wl, hidden, gamma, wq, args.cpu_seconds / 3, threads=1)
        line["cpu_baseline"] = {"value": round(rate / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": f"{rows} of {wl.n_rows} weight rows x batch {wl.batch}, {reps} pass(es), "
                                          f"{secs:.1f} s wall on {cores} threads",
                                "single_thread": {"value": round(rate1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                                                  "sample": f"{rows1} of {wl.n_rows} weight rows x batch "
                                                            f"{wl.batch}, {reps1} pass(es), {secs1:.1f} s wall"},
                                "cpu_model": cpu_model(), "host_cores": os.cpu_count()}
    head.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    import q5k_synth as synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="lmhead_b1", choices=sorted(synth.WORKLOADS) + sorted(synth.GROUPS))
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--logprobs", action="store_true",
                    help="time the logprobs forward (log-softmax of the capped logits) instead of the logits")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", dest="sweep", action="store_true", default=None,
                    help="also time every workload of the metric (default: on for the default workload)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--sweep-seconds", type=float, default=0.8,
                    help="timed seconds per large sweep entry (lets the clock sampler see each one)")
    ap.add_argument("--rows", type=int, default=0,
                    help="profiling: keep only the first ROWS weight rows of the workload")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep is None:
        args.sweep = args.workload == "lmhead_b1" and not args.rows and not args.logprobs
    wl = synth.GROUPS[args.workload] if args.workload in synth.GROUPS else synth.WORKLOADS[args.workload]
    if (args.rows or args.logprobs) and isinstance(wl, synth.GroupWorkload):
        ap.error("--rows and --logprobs apply to single-matrix workloads")
    if args.rows:
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name}[rows={args.rows}]", n_rows=args.rows,
                                 boost_rows=tuple(r for r in wl.boost_rows if r < args.rows))
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
