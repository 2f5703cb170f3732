"""Benchmark one decode step of the DSpark hot path: the K-step Markov drafting
loop plus rejection-sampling verification, on the MiniMax-like drafter
workload (vocab 200064, K = 7, markov_rank 256, fp32 logits and cache,
batch 32 by default), synthetic seeded data.

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle on
the host cores instead (the slow, obviously-correct restatement), on a
bounded sample of the same workload.

Timing: one CUDA graph of the two library calls (the Markov loop, then
verification) replayed once per step, CUDA events on the launching stream
around each replay; L2 is flushed (a 512 MiB write) before every step,
outside the timed events. The loop and the verifier are also timed as graphs
of their own, after the steps, to split the step (each half then pays its own
graph launch). For N > 1 (torchrun) every rank runs an independent replica
(no collectives on the data path); the barrier and the max over ranks use the
process group only for timing.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per decode step (K-step Markov loop + verify) and % of HBM roofline, 1×GB300"
PAGES_ROOFLINE_GBS = 8000.0  # the "8 TB/s" the workload's roofline is quoted against


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """SM clock and clock-event (throttle) samples during the timed region.

    NVML (the library behind nvidia-smi, loaded with ctypes) is polled every
    2 ms from a thread, so that even a timed region of a few tens of
    milliseconds gets samples; nvidia-smi -lms is the fallback. Read-only: no
    setting of the GPU is touched."""

    # NVML clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.samples = []      # (sm_mhz, max_mhz, reason bits)
        self.lines = []        # nvidia-smi fallback
        self.proc = None
        self._stop = threading.Event()
        self._t = None
        self._nvml = None
        self._h = None
        self.source = None

    def _uuid(self):
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.dev).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    def _nvml_open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        uuid = self._uuid()
        ok = uuid is not None and lib.nvmlDeviceGetHandleByUUID(uuid.encode(),
                                                                ctypes.byref(h)) == 0
        if not ok:
            return False
        self._nvml, self._h = lib, h
        self._reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return True

    def _nvml_sample(self):
        import ctypes
        sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(sm)) != 0:
            return
        self._nvml.nvmlDeviceGetMaxClockInfo(self._h, 1, ctypes.byref(mx))
        self._reason_fn(self._h, ctypes.byref(rs))
        self.samples.append((float(sm.value), float(mx.value), int(rs.value)))

    def _poll(self):
        while not self._stop.is_set():
            self._nvml_sample()
            time.sleep(0.002)

    def start(self):
        if self._nvml_open():
            self.source = "nvml"
            self._nvml_sample()
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
            return
        try:
            target = self._uuid() or str(self.dev)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.source == "nvml":
            self._stop.set()
            self._t.join(timeout=2)
            self._nvml_sample()
            reasons = set()
            for _, _, bits in self.samples:
                for bit, name in self.REASONS.items():
                    if bits & bit:
                        reasons.add(name)
            sm = [a for a, _, _ in self.samples]
            return {"sm_mhz": statistics.median(sm) if sm else None,
                    "sm_max_mhz": max(b for _, b, _ in self.samples) if self.samples else None,
                    "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def algorithmic_bytes(w):
    """Bytes the path must move at least once (the roofline's numerator):
    Markov loop per step: markov_w2 once, the base row and the cache row of
    every request, the Markov embeddings; verification: every target row and
    every draft-cache row once."""
    s_base = 2 if w.base_bf16 else 4
    s_cache = 2 if w.cache_bf16 else 4
    s_t = 2 if w.target_bf16 else 4
    per_markov_step = 2 * w.V * w.R + w.B * w.V * (s_base + s_cache) + 2 * w.B * w.R
    verify = w.B * (w.K + 1) * w.V * s_t + w.B * w.K * w.V * s_cache
    return per_markov_step, verify


def _subset(w, idx):
    import copy
    idx = np.asarray(idx)
    v = copy.copy(w)
    v.B = len(idx)
    v.base = np.ascontiguousarray(w.base[idx])
    v.anchor = np.ascontiguousarray(w.anchor[idx])
    v.req_state_idx = np.ascontiguousarray(w.req_state_idx[idx])
    v.positions = np.ascontiguousarray(w.positions[idx])
    v.target = np.ascontiguousarray(w.target[idx])
    return v


def time_oracle(w, n_req: int, threads: int = 1):
    """Seconds of the CPU oracle for the first n_req requests of w (loop,
    verify), on `threads` host threads (OpenMP over requests when > 1)."""
    import oracle
    oracle.build()
    sub = _subset(w, list(range(n_req)))
    t0 = time.perf_counter()
    tok, cache, _ = oracle.markov_sample(sub.base, sub.w1, sub.w2, sub.anchor,
                                         sub.req_state_idx, sub.positions, sub.temperature,
                                         sub.seeds, cache_rows=w.C, cache_bf16=w.cache_bf16,
                                         row_map=w.row_map, threads=threads)
    t1 = time.perf_counter()
    oracle.rejection_sample(tok, cache, sub.target, sub.req_state_idx, sub.positions,
                            sub.temperature, sub.top_p, sub.seeds, row_map=w.row_map,
                            threads=threads)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def host_threads() -> int:
    """The host cores this process may run on (nproc)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_threads() -> int:
    """Threads the parallel oracle leg uses: every host core, if the OpenMP
    build of the oracle exists, else 1."""
    import oracle
    n = host_threads()
    try:
        return oracle.threads_in_use(n)
    except RuntimeError:
        return 1


def cpu_baseline(w, budget_s: float = 20.0):
    """The oracle on the host cores: the parallel leg runs as many requests of
    the batch as fit the time budget (the whole batch if it does) on every
    core; the single-threaded leg runs request 0 alone, i.e. the workload at
    batch 1. Both as µs per decode step."""
    thr = oracle_threads()
    a1, b1 = time_oracle(w, 1, 1)
    one = (a1 + b1) * 1e6
    # requests the parallel leg can afford: about `budget_s` of wall time
    per_req_wall = (a1 + b1) / max(1, thr)
    n_req = int(max(1, min(w.B, budget_s / max(per_req_wall, 1e-9))))
    t0 = time.perf_counter()
    a, b = time_oracle(w, n_req, thr)
    wall = time.perf_counter() - t0
    scale = w.B / n_req
    return {"value": round((a + b) * scale * 1e6, 1), "unit": "us", "cores": thr,
            "kind": "oracle", "nproc": host_threads(),
            "sample": (f"{n_req} of {w.B} requests of one decode step (K-step loop + "
                       f"verification), OpenMP over requests on {thr} host threads" +
                       ("" if n_req == w.B else f", scaled by {w.B}/{n_req}")),
            "measured_wall_s": round(wall, 3), "extrapolation": round(scale, 3),
            "loop_us": round(a * scale * 1e6, 1), "verify_us": round(b * scale * 1e6, 1),
            "single_thread": {"value": round(one, 1), "unit": "us", "cores": 1,
                              "sample": "request 0 alone (the same workload at batch 1): "
                                        "K-step loop + verification, measured, not scaled",
                              "loop_us": round(a1 * 1e6, 1), "verify_us": round(b1 * 1e6, 1)}}


def build_workload(args):
    from verify_dspark_markov_step_gb300 import workloads as wl
    return wl.make(args.config, batch=args.batch)


def max_over_ranks(value: float, world: int, device: str) -> float:
    """The largest of every rank's value (the slowest replica sets a step's
    time); the value itself on one process. `device` holds the one-element
    tensor the process group reduces ("cuda" for NCCL, "cpu" for gloo)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle on the host cores (OpenMP over the
    requests on every core). Each step runs as many requests of the batch as
    keep the whole --warmup + --steps run within about two minutes -- the
    whole batch when they fit -- and the line says how many and by what
    factor the time was scaled."""
    if rank != 0:
        return
    w = build_workload(args)
    thr = oracle_threads()
    # size the per-step sample from one timed request on all threads
    a1, b1 = time_oracle(w, min(w.B, thr), thr)
    per_req = (a1 + b1) / min(w.B, thr)
    n_steps = max(1, args.steps) + max(0, args.warmup)
    n_req = int(max(1, min(w.B, 120.0 / n_steps / max(per_req, 1e-9))))
    for _ in range(max(0, args.warmup)):
        time_oracle(w, n_req, thr)
    loops, vers = [], []
    t0 = time.perf_counter()
    for _ in range(max(1, args.steps)):
        a, b = time_oracle(w, n_req, thr)
        loops.append(a)
        vers.append(b)
    wall = time.perf_counter() - t0
    scale = w.B / n_req
    loop_us = statistics.mean(loops) * scale * 1e6
    ver_us = statistics.mean(vers) * scale * 1e6
    val = loop_us + ver_us
    sample = (f"{n_req} of {w.B} requests per step (K-step loop + verification), OpenMP "
              f"over requests on {thr} host threads" +
              ("" if n_req == w.B else f", scaled by {w.B}/{n_req}"))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 1), "unit": "us",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(val / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, args),
        "loop_us": round(loop_us, 1), "verify_us": round(ver_us, 1),
        "requests_per_step_measured": n_req, "extrapolation": round(scale, 3),
        "measured_wall_s_timed_steps": round(wall, 3),
        "cpu_baseline": {"value": round(val, 1), "unit": "us", "cores": thr, "kind": "oracle",
                         "nproc": host_threads(), "sample": sample},
        "e2e": {"value": round(val, 1), "unit": "us", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w, args):
    topk = f", top-{args.draft_topk} Markov candidates" if args.draft_topk else ""
    topk += ", draft-row statistics recorded by the loop" if args.draft_stats else ""
    return {"workload": f"{w.name}-like drafter: batch {w.B}, K={w.K}, vocab {w.V}, "
                        f"markov_rank {w.R}, {'bf16' if w.base_bf16 else 'fp32'} logits, "
                        f"{'bf16' if w.cache_bf16 else 'fp32'} draft cache{topk}",
            "batch": w.B, "K": w.K, "vocab": w.V, "markov_rank": w.R,
            "l2": "flushed (512 MiB write) before every timed step",
            "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


def _capture(st, stream):
    """One decode step as one CUDA graph of both library calls (the Markov
    loop, then verification, on one stream), and each half as a graph of its
    own (to split the step)."""
    import torch
    with torch.cuda.stream(stream):
        st.run(stream=stream)
    stream.synchronize()
    g = {"step": torch.cuda.CUDAGraph(), "markov": torch.cuda.CUDAGraph(),
         "verify": torch.cuda.CUDAGraph()}
    with torch.cuda.graph(g["step"], stream=stream):
        st.markov(stream=stream)
        st.verify(stream=stream)
    with torch.cuda.graph(g["markov"], stream=stream):
        st.markov(stream=stream)
    with torch.cuda.graph(g["verify"], stream=stream):
        st.verify(stream=stream)
    return g


def _one_step(g, stream, flush):
    """L2 flush, then one timed replay of the whole step; returns its events."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        flush.fill_(1)
        ev[0].record(stream)
        g["step"].replay()
        ev[1].record(stream)
    return ev


def _split_step(g, stream, flush):
    """L2 flush, then the loop's graph and the verifier's, timed apart."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with torch.cuda.stream(stream):
        flush.fill_(1)
        ev[0].record(stream)
        g["markov"].replay()
        ev[1].record(stream)
        g["verify"].replay()
        ev[2].record(stream)
    return ev


# The workloads timed beside the headline one (same run, same timing rules):
# the drafter at batch 1 and 4, the verify-heavy bf16 workload, the long-draft
# stress workload and the odd vocabulary.
OTHER_CONFIGS = [("minimax", 1), ("minimax", 4), ("qwen", 256), ("long", 128), ("odd", 8)]


def other_configs(args, stream, flush, peak):
    """Each other workload: its step, loop and verifier times and the
    verifier's fraction of the HBM peak."""
    import torch
    from verify_dspark_markov_step_gb300 import workloads as wl
    from verify_dspark_markov_step_gb300.step import DecodeStep
    out = []
    steps = max(3, min(args.steps, 10))
    for name, batch in OTHER_CONFIGS:
        if (name, batch) == (args.config, args.batch):
            continue
        w = wl.make(name, batch=batch)
        st = DecodeStep(w, draft_topk=args.draft_topk, draft_stats=args.draft_stats)
        g = _capture(st, stream)
        for _ in range(3):
            _one_step(g, stream, flush)
            _split_step(g, stream, flush)
        evs = [_one_step(g, stream, flush) for _ in range(steps)]
        sev = [_split_step(g, stream, flush) for _ in range(steps)]
        torch.cuda.synchronize()
        step_us = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) * 1e3
        loop_us = statistics.mean(e[0].elapsed_time(e[1]) for e in sev) * 1e3
        ver_us = statistics.mean(e[1].elapsed_time(e[2]) for e in sev) * 1e3
        per_step, ver_bytes = algorithmic_bytes(w)
        out.append({
            "workload": f"{w.name}: batch {w.B}, K={w.K}, vocab {w.V}, markov_rank {w.R}",
            "steps": steps, "value": round(step_us, 2), "unit": "us",
            "loop_us": round(loop_us, 2), "verify_us": round(ver_us, 2),
            "loop_frac": round(per_step * w.K / (loop_us * 1e-6) / 1e9 / peak, 3),
            "verify_frac": round(ver_bytes / (ver_us * 1e-6) / 1e9 / peak, 3),
            "mean_accepted": round(st.num_accepted.float().mean().item(), 3),
            "status": st.status_code()})
        del g, st
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local):
    import torch
    from verify_dspark_markov_step_gb300 import build
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_device
    from verify_dspark_markov_step_gb300 import _lib

    torch.cuda.set_device(local)
    build.build()
    w = build_workload(args)
    st = DecodeStep(w, draft_topk=args.draft_topk, draft_stats=args.draft_stats)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    graphs = _capture(st, stream)
    for _ in range(args.warmup):
        _one_step(graphs, stream, flush)
        _split_step(graphs, stream, flush)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t0 = time.perf_counter()
    evs = [_one_step(graphs, stream, flush) for _ in range(args.steps)]
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms = max_over_ranks(statistics.mean(step_ms), world, "cuda")
    # the two halves, each its own graph (each pays its own graph launch)
    sev = [_split_step(graphs, stream, flush) for _ in range(args.steps)]
    torch.cuda.synchronize()
    clk = clocks.stop()
    loop_ms = [e[0].elapsed_time(e[1]) for e in sev]
    ver_ms = [e[1].elapsed_time(e[2]) for e in sev]
    status = st.status_code()
    nacc = st.num_accepted.float().mean().item()
    tokens = (st.num_accepted + 1).sum().item()

    # end to end through the public API with host buffers
    base_h = torch.from_numpy(np.ascontiguousarray(w.base)).pin_memory()
    tgt_h = torch.from_numpy(np.ascontiguousarray(w.target)).pin_memory()
    small_h = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
               for a in (w.anchor, w.req_state_idx, w.positions)]
    small_d = [st.anchor, st.rsi, st.pos]
    out_h = torch.empty((w.B, w.K + 1), dtype=torch.int32).pin_memory()
    nacc_h = torch.empty(w.B, dtype=torch.int32).pin_memory()
    h2d = base_h.numel() * base_h.element_size() + tgt_h.numel() * tgt_h.element_size() + \
        sum(t.numel() * t.element_size() for t in small_h)
    d2h = out_h.numel() * 4 + nacc_h.numel() * 4

    # The host-to-device link (about 207 GB/s here, the same with one copy
    # stream or several) bounds this measurement. The copies run in the order
    # they are needed on one copy stream: the small inputs and the base logits
    # first, at the link's full rate, then the target logits, which only the
    # verifier reads; the Markov loop starts as soon as the base logits are in
    # and runs beside the target copy.
    tstream = torch.cuda.Stream()

    def e2e_step(ev):
        base_in = torch.cuda.Event()
        with torch.cuda.stream(stream):
            flush.fill_(1)
            ev[0].record(stream)
            tstream.wait_event(ev[0])
            with torch.cuda.stream(tstream):
                for h, d in zip(small_h, small_d):
                    d.copy_(h, non_blocking=True)
                st.base.copy_(base_h, non_blocking=True)
                base_in.record(tstream)
                st.target.copy_(tgt_h, non_blocking=True)
            stream.wait_event(base_in)
            st.markov(stream=stream)
            stream.wait_stream(tstream)
            st.verify(stream=stream)
            out_h.copy_(st.out, non_blocking=True)
            nacc_h.copy_(st.num_accepted, non_blocking=True)
            ev[1].record(stream)

    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(3):
        e2e_step([torch.cuda.Event(enable_timing=True) for _ in range(2)])
    torch.cuda.synchronize()
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        e2e_step(eev[i])
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in eev), world,
                            "cuda")

    peak, peak_kind = _peaks()
    per_step, ver_bytes = algorithmic_bytes(w)
    per_launch = per_step * w.K  # one launch runs all K Markov steps
    loop_kernel = "markov_loop_tc (one launch = all K Markov steps)"
    if args.draft_topk:
        # top-k variant: the base logits read once and the cache rows written
        # once (candidate selection and -inf fill), the candidates' w2 rows
        # gathered, the embeddings; two launches
        s_base = 2 if w.base_bf16 else 4
        s_cache = 2 if w.cache_bf16 else 4
        k = min(args.draft_topk, w.V)
        per_launch = w.B * w.K * (w.V * (s_base + s_cache) + k * (2 * w.R + 8) + 2 * w.R)
        loop_kernel = "topk_rows + markov_topk_loop (candidate selection, then the K steps)"
    loop_us = statistics.mean(loop_ms) * 1e3
    ver_us = statistics.mean(ver_ms) * 1e3
    achieved = per_launch / (loop_us * 1e-6) / 1e9
    traffic = None if args.draft_topk or args.draft_stats else _traffic_from_profile(
        args, "markov_loop_tc_minimax_b32.md", ("markov_tc.cu", "common.cuh", "tc_ptx.cuh"))
    line = {
        "metric": METRIC, "value": round(ms * 1e3, 2), "unit": "us", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": _config(w, args),
        # the halves timed as graphs of their own (each with its own launch)
        "loop_us": round(loop_us, 2), "verify_us": round(ver_us, 2),
        "step_us_p10_p90": [round(float(np.percentile(step_ms, 10)) * 1e3, 2),
                            round(float(np.percentile(step_ms, 90)) * 1e3, 2)],
        "loop_us_p10_p90": [round(float(np.percentile(loop_ms, 10)) * 1e3, 2),
                            round(float(np.percentile(loop_ms, 90)) * 1e3, 2)],
        "verify_us_p10_p90": [round(float(np.percentile(ver_ms, 10)) * 1e3, 2),
                              round(float(np.percentile(ver_ms, 90)) * 1e3, 2)],
        "tokens_per_s": round(tokens * world / (ms * 1e-3), 1),
        "mean_accepted": round(nacc, 3),
        "hbm_frac_8tbs": {
            "loop": round(per_launch / (loop_us * 1e-6) / 1e9 / PAGES_ROOFLINE_GBS, 3),
            "verify": round(ver_bytes / (ver_us * 1e-6) / 1e9 / PAGES_ROOFLINE_GBS, 3)},
        "roofline": {"bound": "hbm", "kernel": loop_kernel,
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "peak_kind": peak_kind,
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": per_launch,
                     "verify_achieved": round(ver_bytes / (ver_us * 1e-6) / 1e9, 1),
                     "verify_frac": round(ver_bytes / (ver_us * 1e-6) / 1e9 / peak, 3)},
        "e2e": {"value": round(e2e_ms * 1e3, 1), "unit": "us", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        # per step: the Markov loop kernel (top-k: candidate selection, then
        # the loop) and the one verification kernel; the graph's memset nodes
        # (the loop's and the verifier's cleared control words) are not kernels
        "gpu_launches": args.steps * (3 if args.draft_topk else 2),
        "memset_nodes_per_step": 3 if args.draft_stats else 2,
        "clocks": clk, "status": status, "wall_s_timed_region": round(wall, 4),
    }
    vt = None if args.draft_topk or args.draft_stats else _traffic_from_profile(
        args, "verify_flat_minimax_b32.md",
        ("verify_stats.cu", "verify_draw.cuh", "verify_common.cuh", "common.cuh", "kernels.h"))
    line["roofline"]["verify_traffic"] = vt
    if rank == 0 and world == 1 and not args.no_other_configs:
        del graphs
        torch.cuda.empty_cache()
        line["other_configs"] = other_configs(args, stream, flush, peak)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def _traffic_from_profile(args, summary, sources):
    """DRAM bytes (read + write) per launch of a kernel from its committed ncu
    summary under profiles/, if it was taken on this workload (MiniMax-like,
    batch 32) and on the current kernel sources (its source hash matches);
    else None."""
    import hashlib
    import re
    if args.config != "minimax" or args.batch != 32:
        return None
    p = os.path.join(ROOT, "profiles", summary)
    try:
        with open(p) as f:
            txt = f.read()
        t = re.search(r"^traffic_bytes_per_launch: (\d+)", txt, re.M)
        h = re.search(r"^source_sha256: ([0-9a-f]+)", txt, re.M)
        if not t or not h:
            return None
        m = hashlib.sha256()
        for name in sources:
            with open(os.path.join(ROOT, "verify_dspark_markov_step_gb300", "csrc", name), "rb") as f:
                m.update(f.read())
        return int(t.group(1)) if m.hexdigest().startswith(h.group(1)) else None
    except OSError:
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="minimax")
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="time the named workload only (no other_configs block)")
    ap.add_argument("--draft-topk", type=int, default=0,
                    help="time the top-k variant of the Markov loop (0: the dense loop)")
    ap.add_argument("--draft-stats", action="store_true",
                    help="the Markov loop records each draft row's maximum and exp-mass "
                         "and the verifier uses them instead of reading the rows")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = _dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
