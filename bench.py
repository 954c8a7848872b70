#!/usr/bin/env python
"""Training steps/s (forward + backward) of the sparse-graph leaky-tanh
recurrence on one GB300, for the FlyGPT launch shape (connectome-kernels page,
"Why" table: N=5,000, E=524,324, B=32, T x microsteps = 64 x 2).

One step = ck_forward + ck_backward over the whole window, inputs resident in
HBM; the L2 is flushed (a 512 MB write) before every timed step and the flush
is outside the timed events.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference|torch-sparse]
                  [--config 0-4] [--microsteps M] [--graph-in-host-memory]

--config picks another of the five synthetic workloads (default 1, the FlyGPT
shape that the headline is quoted on); --microsteps overrides its M.
--graph-in-host-memory builds the graph with its edge-indexed arrays in pinned
host memory, read by the kernels over the CPU-GPU link.  --recompute times the
checkpointing forward and the recomputing backward instead of the regular
pair.  --ncu-steps K only runs K steps (for a profiler) and exits.
--barrier-probe times the grid-barrier schemes of ck_probe_grid_barrier on their
own (ns per crossing, 304 CTAs each writing 16 rows per crossing, and the
uncontended single-CTA floor) and prints one JSON line instead of the bench line.
--phase-profile loads the profiling build (libck_prof.so) and prints, for the
workload, the mean and slowest-CTA time of each phase of a microstep (part A,
the CTA sync, the finish, the grid barrier) instead of the bench line.

With N > 1 (under torchrun) every rank runs an independent replica of the
same step (the method has no exchange between replicas): weak scaling.
--impl reference times the CPU oracle (fp64) on whole steps, every batch
column, spread over all host cores with OpenMP.  --impl torch-sparse times, for
context only, the step written with torch.sparse.mm in a Python loop (the
baseline the page compares its fused kernels with); it is not part of the
library.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "train steps/sec (fwd+bwd) at N=5k,E=524k,B=32,T=64×2; % of HBM/L2 roofline"
PAGE_STEPS_PER_S = 1000.0 / 15.5  # the page's fused-kernel step time for this workload (B200)
HBM_FALLBACK = 6800.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK, "fallback"


def source_digest(path):
    """First 16 hex digits of the sha256 of a C/C++ source's code: comments
    removed and runs of whitespace collapsed, so that an edit to comments keeps
    a profile capture valid and any edit to the code voids it."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    tokens = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|//[^\n]*|/\*.*?\*/', re.S)
    code = tokens.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text)
    return hashlib.sha256(" ".join(code.split()).encode()).hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch of `kernel` ("forward"/"backward") from the committed ncu
    summary, or None when the kernel source's code has changed since that capture."""
    try:
        src = os.path.join(ROOT, "sparse_graph_recurrent_gb300", "csrc", "recurrence.cu")
        digest = source_digest(src)
        for line in open(os.path.join(ROOT, "profiles", "rec_kernel_flygpt.md")):
            if line.startswith("traffic_bytes_per_launch:"):
                kv = dict(x.split("=") for x in line.split(":", 1)[1].split())
                if kv.get("source_code_sha256_16") == digest:
                    return int(kv[kernel])
    except Exception:
        pass
    return None


def max_over_ranks(x, dist, device):
    """The largest of every rank's x: a job of replicas takes as long as its
    slowest rank."""
    if not dist:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(local_total_ms, steps, world, dist, device):
    """(job time in ms, whole-job steps/s) for `world` independent replicas
    that each timed `steps` steps: every replica's steps over the slowest
    rank's time."""
    total_ms = max_over_ranks(local_total_ms, dist, device)
    return total_ms, world * steps / (total_ms / 1e3)


def byte_model(N, E, B, T, M, n_in):
    """Algorithmic bytes per launch (every byte that must reach the SMs).

    Forward microstep: graph 8E + 4(N+1), gathered source rows 4EB, own row
    read plus state and pre-activation written 12NB, drives 4 n_in B.
    Backward microstep: transposed graph 8E + 4(N+1), edge-gradient
    read-modify-write 8E, gathered rows 4EB, own rows 16NB.
    Per input step: the output write (forward) and dOut read (backward), 4NB each.
    """
    S = T * M
    fwd = S * (8 * E + 4 * (N + 1) + 4 * E * B + 12 * N * B + 4 * n_in * B) + T * 4 * N * B
    bwd = S * (8 * E + 4 * (N + 1) + 8 * E + 4 * E * B + 16 * N * B) + T * 4 * N * B
    return fwd, bwd


L2_BYTES = 126 << 20  # about what of the 129 MB L2 a working set can keep


def hbm_bytes(N, E, B, T, M, n_in):
    """Compulsory DRAM bytes per step: saved activations written and read
    back, out, dOut, drives and their gradient, state0 and its gradient,
    parameters and their gradients, and the graph (both compressed-row copies)
    once per step if it fits in L2, else once per microstep of each pass."""
    S = T * M
    saved = 2 * 4 * (2 * S + 1) * N * B
    io = 4 * (2 * T * N * B + 2 * T * n_in * B + 2 * N * B + 2 * E + 4 * N)
    graph = 2 * (8 * E + 4 * (N + 1))
    return saved + io + (graph if graph <= L2_BYTES else S * graph)


def step_roofline(q_l2, q_hbm, bw_l2_gbs, bw_hbm_gbs, step_ms):
    """The step-level fraction: the roofline time max(Q_L2 / BW_L2, Q_HBM /
    BW_HBM) of a whole step over its measured time, and which bound sets it."""
    t_l2 = q_l2 / (bw_l2_gbs * 1e9) * 1e3
    t_hbm = q_hbm / (bw_hbm_gbs * 1e9) * 1e3
    bound, t = ("l2", t_l2) if t_l2 >= t_hbm else ("hbm", t_hbm)
    return {"bound": bound, "roofline_ms": t, "step_ms": step_ms, "frac": t / step_ms,
            "l2_ms": t_l2, "hbm_ms": t_hbm}


def memory_figures(N, E, B, T, n_in, graph_bytes, saved_b, scratch_b, ckpt_b, scratch_rc_b):
    """Device bytes one training step holds: the graph, the caller's inputs,
    outputs and gradients, and the saved activations and scratch of the
    regular pair or of the recomputing pair."""
    io = 4 * (E + 2 * N + T * n_in * B + B * N  # w, leak, bias, drives, state0
              + 2 * T * B * N                     # out, dOut
              + E + 2 * N + T * n_in * B + B * N)  # their gradients
    return {"graph_bytes": graph_bytes, "io_bytes": io, "saved_bytes": saved_b,
            "scratch_bytes": scratch_b, "step_bytes": graph_bytes + io + saved_b + scratch_b,
            "recompute": {"ckpt_bytes": ckpt_b, "scratch_bytes": scratch_rc_b,
                          "step_bytes": graph_bytes + io + ckpt_b + scratch_rc_b},
            "page_context": "connectome-kernels page, Why table (B200): fused kernels 0.55 GB, "
                            "torch.sparse 2.43 GB per training step"}


def flops_per_step(N, E, B, T, M):
    """Algorithmic floating-point operations of one step: per microstep about
    6EB (gather multiply-add forward; gather and edge-gradient dot backward)
    and 12NB elementwise."""
    return T * M * (6 * E * B + 12 * N * B)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons, kept for the
    samples taken inside the timed region (begin() .. end())."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index, interval_ms=50):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.index = index
        self.interval_ms = interval_ms
        self.t_begin = self.t_end = None

    def start(self):
        """Start the sampler and wait (up to 5 s) for its first line, so that
        the timed region that follows is covered from its start."""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        deadline = time.time() + 5.0
        while time.time() < deadline and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()
        if self.proc is not None:
            time.sleep(2 * self.interval_ms / 1e3)  # the sample in flight at the end

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.read().splitlines()
        os.unlink(self.path)
        return self.summarize(lines, self.t_begin, self.t_end)

    @classmethod
    def summarize(cls, lines, t_begin, t_end):
        """Median SM clock, maximum clock and the throttle reasons seen, over
        the samples whose timestamp lies in [t_begin, t_end] (epoch seconds);
        if none does (a region shorter than the interval), the sample nearest
        to the region stands in and "samples" says 0."""
        import datetime
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t_begin is not None and t_end is not None and t_begin <= r[0] <= t_end]
        use = inside
        if not use:
            mid = ((t_begin or 0.0) + (t_end or 0.0)) / 2
            use = [min(rows, key=lambda r: abs(r[0] - mid))]
        reasons = sorted({n for r in use for n, v in zip(cls.REASONS, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(inside), "interval_ms": None if not rows else
                round(1e3 * (rows[-1][0] - rows[0][0]) / max(len(rows) - 1, 1), 1)}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def oracle_step_seconds(c, threads):
    """Seconds of one whole oracle step (forward and backward over every batch
    column): the single-thread oracle for threads == 1, else its column-parallel
    statement on `threads` OpenMP threads."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    if threads == 1:
        oracle.run_case(c)
    else:
        oracle.step_columns(c, threads)
    return time.perf_counter() - t0


def cpu_baseline(c, omp_steps=3):
    """The oracle timed on this host: one whole single-thread step, and
    `omp_steps` whole steps over all cores (OpenMP across batch columns)."""
    import oracle
    oracle.build()
    cores = oracle.threads_available()
    single = oracle_step_seconds(c, 1)
    multi = [oracle_step_seconds(c, cores) for _ in range(omp_steps)]
    per = statistics.mean(multi)
    return {"value": 1.0 / per, "unit": "steps/s", "cores": cores, "threads": cores,
            "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"{omp_steps} whole steps (all {c['B']} batch columns, full graph and "
                      f"window), fp64, OpenMP over batch columns on {cores} threads",
            "single_thread": {"value": 1.0 / single, "unit": "steps/s", "threads": 1,
                              "sample": "one whole step on one thread (the oracle as it stands)"}}


def torch_sparse_step(c, dev, dtype):
    """One training step written with torch.sparse.mm in a Python loop over
    T x microsteps, the backward by autograd (connectome-kernels page, "Why":
    the torch.sparse COO baseline).  Returns (out [T, B, N], gradients of
    L = sum(out * dOut) w.r.t. w, leak, bias, drives, state0)."""
    import torch
    N = c["N"]
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a), device=dev, dtype=dtype)  # noqa: E731
    w, leak, bias = (t(c[k]).requires_grad_() for k in ("w", "leak", "bias"))
    drives, state0 = t(c["drives"]).requires_grad_(), t(c["state0"]).requires_grad_()
    dout = t(c["dout"])
    idx = torch.stack([torch.as_tensor(c["dst"], device=dev), torch.as_tensor(c["src"], device=dev)])
    inp = torch.as_tensor(c["input_nodes"], device=dev)
    T, M = drives.shape[0], c["M"]
    W = torch.sparse_coo_tensor(idx, w, (N, N), check_invariants=False).coalesce()  # W[dst][src]; repeated pairs add
    h = state0.t()
    outs = []
    for ti in range(T):
        drive = torch.zeros(N, h.shape[1], device=dev, dtype=dtype).index_put((inp,), drives[ti])
        for _ in range(M):
            p = torch.tanh(torch.sparse.mm(W, h) + drive + bias[:, None])
            h = (1 - leak[:, None]) * h + leak[:, None] * p
        outs.append(h.t())
    out = torch.stack(outs)
    (out * dout).sum().backward()
    return out.detach(), [x.grad for x in (w, leak, bias, drives, state0)]


def run_torch_sparse(args, c, rank):
    if rank != 0:
        return
    import torch
    dev = torch.device("cuda", 0)
    for _ in range(max(args.warmup, 1)):
        torch_sparse_step(c, dev, torch.float32)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        torch_sparse_step(c, dev, torch.float32)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({
        "impl": "torch-sparse", "context_only": True, "metric": METRIC, "value": 1e3 / ms,
        "unit": "steps/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "config": {"workload": _workload_name(c)},
        "note": "torch.sparse.mm in a Python loop over T x microsteps, autograd backward "
                "(the page's baseline: 207 ms on B200)"}), flush=True)


def run_reference(args, c, rank):
    """The reference arm: the CPU oracle, whole steps over all batch columns,
    OpenMP across columns on every host core (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.threads_available()
    for _ in range(args.warmup):
        oracle_step_seconds(c, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step_seconds(c, cores)
    per_step = (time.perf_counter() - t0) / args.steps
    value = 1.0 / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGE_STEPS_PER_S, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_name(c), "parallelism": "replicas",
                   "l2": "not applicable (CPU)"},
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "threads": cores,
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": f"{args.steps} whole steps (all {c['B']} batch columns), fp64, "
                                   f"OpenMP over batch columns on {cores} threads"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


CONFIG_NAMES = {0: "tiny", 1: "flygpt", 2: "ragged", 3: "wide", 4: "connectome"}


def _workload_name(c):
    name = CONFIG_NAMES.get(c.get("config_id", 1), "workload")
    return f"{name} N={c['N']} E={c['E']} B={c['B']} T={c['T']} M={c['M']}"


# Shapes of the dense L2 read probe swept for the roofline's denominator:
# (load bytes, loads in flight per thread, threads per CTA, CTAs per SM).
# Each keeps one pass of the whole grid (loads x threads x bytes) within half
# of the 64 MB buffer, so every thread runs its loads-in-flight loop.
L2_SWEEP = [(16, 4, 512, 2), (16, 8, 512, 2), (16, 16, 256, 2), (16, 8, 1024, 1),
            (32, 2, 512, 2), (32, 4, 256, 4), (32, 4, 512, 2), (32, 2, 512, 4),
            (32, 8, 256, 2), (32, 4, 1024, 1), (32, 2, 256, 8)]
L2_SWEEP_BYTES = 64 << 20


def l2_read_sweep(timed, buf, sink):
    """GB/s of the dense L2 read probe for each swept shape (and the fixed
    ck_probe_read); `timed(fn)` returns the rate of 10 reads of `buf`."""
    from sparse_graph_recurrent_gb300 import _ck
    out = [{"shape": "ck_probe_read (16-byte loads, 4 in flight, 2 x 512 threads per SM)",
            "gbs": timed(lambda: _ck.ck_probe_read(buf, 10, sink))}]
    for lb, depth, thr, cps in L2_SWEEP:
        out.append({"shape": f"{lb}-byte loads, {depth} in flight, {cps} x {thr} threads per SM",
                    "gbs": timed(lambda: _ck.ck_probe_read_shape(buf, 10, lb, depth, thr, cps,
                                                                 sink))})
    return out


BARRIER_CASES = [
    # (scheme, CTAs per SM (0: a single CTA), cluster)
    ("BARRIER_COUNTER", 0, 1), ("BARRIER_COUNTER", 1, 1), ("BARRIER_COUNTER", 2, 1),
    ("BARRIER_COUNTER_RETURNING", 2, 1), ("BARRIER_COUNTER_RELAXED", 2, 1),
    ("BARRIER_FLAG", 2, 1), ("BARRIER_FLAGS8", 2, 1),
    ("BARRIER_CLUSTER_SYNC", 2, 2), ("BARRIER_CLUSTER_SYNC", 2, 8),
    ("BARRIER_CLUSTER_MBARRIER", 2, 2), ("BARRIER_CLUSTER_MBARRIER", 2, 8),
]


def run_barrier_probe(crossings=4000, rows_per_cta=16):
    """`--barrier-probe`: ns per grid-barrier crossing for each scheme, timed
    with CUDA events on the launching stream (second of two runs)."""
    import torch

    from sparse_graph_recurrent_gb300 import _ck
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = torch.zeros(2 * sms * rows_per_cta * 32, dtype=torch.float32, device=dev)
    words = torch.zeros(_ck.PROBE_BARRIER_WORDS, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = []
    for name, cps, cluster in BARRIER_CASES:
        ctas = 1 if cps == 0 else cps * sms
        rec = {"scheme": name.lower(), "ctas": ctas, "cluster": cluster}
        try:
            ns = None
            for _ in range(2):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                _ck.ck_probe_grid_barrier(getattr(_ck, name), ctas, cluster, crossings,
                                          rows_per_cta, rows, words, status)
                e1.record()
                torch.cuda.synchronize()
                if int(status.item()) != 0:
                    raise RuntimeError("a wait ran out")
                ns = e0.elapsed_time(e1) * 1e6 / crossings
            rec["ns_per_crossing"] = round(ns, 1)
        except (_ck.CKError, RuntimeError) as ex:
            rec["error"] = str(ex)
        out.append(rec)
    print(json.dumps({"barrier_probe": out, "crossings": crossings, "rows_per_cta": rows_per_cta,
                      "threads_per_cta": 256, "gpu": torch.cuda.get_device_name(0)}))


def run_phase_profile(args, c, steps=5):
    """`--phase-profile`: per-phase microstep times from the profiling build
    (ck_phase_profile_read), over `steps` forward + backward steps after one
    warm-up step."""
    import torch

    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    if _ck.library_variant() != "prof":
        raise SystemExit("--phase-profile needs CK_LIBRARY_VARIANT=prof before the library loads")
    dev = torch.device("cuda", 0)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    g = pkg.SparseGraph(tt(c["src"]), tt(c["dst"]), c["N"], tt(c["input_nodes"]),
                        edges_in_host_memory=args.graph_in_host_memory)
    w, leak, bias, drives, state0, dout = (tt(c[k]) for k in ("w", "leak", "bias", "drives",
                                                              "state0", "dout"))
    B, T, M = c["B"], c["T"], c["M"]
    for i in range(steps + 1):
        if i == 1:
            _ck.ck_phase_profile_read(clear=True)
        _, saved, scratch = pkg.forward(g, w, leak, bias, drives, state0, M)
        pkg.backward(g, w, leak, B, T, M, saved, dout, scratch)
    _ck.ck_query_status(scratch)
    data = _ck.ck_phase_profile_read(clear=True)
    out = {}
    for d, name in ((0, "forward"), (1, "backward")):
        ctas = [q for q in data[d] if q[4] > 0]
        per = {
            "part_a": [q[0] / q[4] / 1e3 for q in ctas],
            "cta_sync": [(q[1] - q[0]) / q[4] / 1e3 for q in ctas],
            "finish": [q[2] / q[4] / 1e3 for q in ctas],
            "part_a_sync_finish": [(q[1] + q[2]) / q[4] / 1e3 for q in ctas],
            "barrier": [q[3] / q[5] / 1e3 for q in ctas if q[5] > 0],
        }
        out[name] = {"ctas": len(ctas), "microsteps_per_cta": ctas[0][4] // steps if ctas else 0,
                     **{k: {"mean_us": round(statistics.fmean(v), 3), "slowest_cta_us": round(max(v), 3)}
                        for k, v in per.items() if v}}
    print(json.dumps({"phase_profile": out, "steps": steps, "library": "libck_prof.so",
                      "config": {"workload": _workload_name(c)},
                      "note": "per CTA, mean over its microsteps; %globaltimer stamps add one CTA "
                              "sync per microstep"}))


def run_plain_steps(args, c):
    """`--ncu-steps K`: K forward + backward steps through the public API and
    nothing else (no probes, no timing), for a profiler to capture; prints one
    line when done."""
    import torch

    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck
    dev = torch.device("cuda", 0)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    g = pkg.SparseGraph(tt(c["src"]), tt(c["dst"]), c["N"], tt(c["input_nodes"]),
                        edges_in_host_memory=args.graph_in_host_memory)
    w, leak, bias, drives, state0, dout = (tt(c[k]) for k in ("w", "leak", "bias", "drives",
                                                              "state0", "dout"))
    B, T, M = c["B"], c["T"], c["M"]
    for _ in range(args.ncu_steps):
        _, saved, scratch = pkg.forward(g, w, leak, bias, drives, state0, M)
        pkg.backward(g, w, leak, B, T, M, saved, dout, scratch)
    _ck.ck_query_status(scratch)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_steps": args.ncu_steps, "config": {"workload": _workload_name(c)}}))


def run_ours(args, c, rank, world, dist):
    import torch

    import sparse_graph_recurrent_gb300 as pkg
    from sparse_graph_recurrent_gb300 import _ck

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    N, E, B, T, M, n_in = c["N"], c["E"], c["B"], c["T"], c["M"], c["n_in"]
    g = pkg.SparseGraph(tt(c["src"]), tt(c["dst"]), N, tt(c["input_nodes"]),
                        edges_in_host_memory=args.graph_in_host_memory)
    w, leak, bias, drives, state0, dout = (tt(c[k]) for k in ("w", "leak", "bias", "drives",
                                                              "state0", "dout"))
    saved_b, scratch_b = g.workspace_size(B, T, M)
    ckpt_b, scratch_rc_b = _ck.ck_workspace_size_recompute(g.handle, B, T, M)
    mem = memory_figures(N, E, B, T, n_in, _ck.ck_graph_memory(g.handle)[0], saved_b, scratch_b,
                         ckpt_b, scratch_rc_b)
    # --recompute: the checkpointing forward and the recomputing backward, with
    # their own workspace (checkpoints instead of saved activations)
    saved = torch.empty(ckpt_b if args.recompute else saved_b, dtype=torch.uint8, device=dev)
    scratch = torch.empty(scratch_rc_b if args.recompute else scratch_b, dtype=torch.uint8,
                          device=dev)
    out = torch.empty((T, B, N), device=dev)
    dw, dl, db = (torch.empty(n, device=dev) for n in (E, N, N))
    dd = torch.empty((T, n_in, B), device=dev)
    dh = torch.empty((B, N), device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    launches = [0]

    def fwd_call():
        if args.recompute:
            _ck.ck_forward_checkpointed(g.handle, w, leak, bias, drives, state0, M, out, saved,
                                        scratch)
        else:
            _ck.ck_forward(g.handle, w, leak, bias, drives, state0, M, out, saved, scratch)
        launches[0] += _ck.ck_last_launch_count()

    def bwd_call():
        if args.recompute:
            _ck.ck_backward_recompute(g.handle, w, leak, bias, drives, B, T, M, saved, dout, dw,
                                      dl, db, dd, dh, scratch)
        else:
            _ck.ck_backward(g.handle, w, leak, B, T, M, saved, dout, dw, dl, db, dd, dh, scratch)
        launches[0] += _ck.ck_last_launch_count()

    def step():
        fwd_call()
        bwd_call()

    for _ in range(args.warmup):
        step()
    _ck.ck_query_status(scratch)
    torch.cuda.synchronize()

    # L2 peaks in this run: dense read of a 64 MB buffer, and a gather of
    # random 128-byte rows from a state-sized table (the forward's pattern)
    sink = torch.zeros(1, device=dev)
    buf = torch.ones(L2_SWEEP_BYTES // 4, device=dev)
    rows = torch.ones((N, 32), device=dev)
    idx = torch.randint(0, N, (E,), dtype=torch.int32, device=dev)

    def probe(fn, nbytes, reps=20):
        fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return nbytes / (e0.elapsed_time(e1) / 1e3 / reps) / 1e9

    l2_sweep = l2_read_sweep(lambda f: probe(f, buf.numel() * 4 * 10), buf, sink)
    l2_best = max(l2_sweep, key=lambda r: r["gbs"])
    l2_read = l2_best["gbs"]
    l2_gather = probe(lambda: _ck.ck_probe_gather(rows, idx, sink), E * 128)

    clocks = Clocks(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches[0] = 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks.begin()
    for k in range(args.steps):
        flush.fill_(k & 0xff)
        ev[k][0].record(stream)
        fwd_call()
        ev[k][1].record(stream)
        bwd_call()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    clocks.end()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    _ck.ck_query_status(scratch)
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c2) for _, b, c2 in ev]
    total_ms, value = replica_throughput(sum(a.elapsed_time(c2) for a, _, c2 in ev), args.steps,
                                         world, dist, dev)
    ms_per_step = total_ms / args.steps

    # end to end through the public API: host inputs in, host results out
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    h_in = {k: pin(c[k]) for k in ("w", "leak", "bias", "drives", "state0", "dout")}
    h_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (out, dw, dl, db, dd, dh)]
    h2d = sum(x.numel() * 4 for x in h_in.values())
    d2h = sum(x.numel() * 4 for x in h_out)

    # The two large copies overlap compute on a second stream, as a user
    # would pipeline them: dOut (needed only by the backward) goes in during
    # the forward, and the states come back during the backward.
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()

    def e2e_step():
        d = {k: h_in[k].to(dev, non_blocking=True)
             for k in ("w", "leak", "bias", "drives", "state0")}
        side.wait_stream(main)
        with torch.cuda.stream(side):
            d_out = h_in["dout"].to(dev, non_blocking=True)
        d_out.record_stream(main)
        dout_in = side.record_event()
        if args.recompute:
            o, sv, sc = pkg.forward_checkpointed(g, d["w"], d["leak"], d["bias"], d["drives"],
                                                 d["state0"], M)
        else:
            o, sv, sc = pkg.forward(g, d["w"], d["leak"], d["bias"], d["drives"], d["state0"], M)
        fwd_done = main.record_event()
        with torch.cuda.stream(side):
            side.wait_event(fwd_done)
            h_out[0].copy_(o, non_blocking=True)
        o.record_stream(side)
        main.wait_event(dout_in)
        if args.recompute:
            grads = pkg.backward_recompute(g, d["w"], d["leak"], d["bias"], d["drives"], B, T, M,
                                           sv, d_out, sc)
        else:
            grads = pkg.backward(g, d["w"], d["leak"], B, T, M, sv, d_out, sc)
        for hdst, src in zip(h_out[1:], grads):
            hdst.copy_(src, non_blocking=True)
        main.wait_stream(side)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)

    if rank != 0:
        return
    fb, bb = byte_model(N, E, B, T, M, n_in)
    f_mean, b_mean = statistics.mean(fwd_ms), statistics.mean(bwd_ms)
    dom, dom_bytes, dom_ms = ("backward", bb, b_mean) if b_mean >= f_mean else ("forward", fb, f_mean)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    hbm_peak, hbm_src = _peaks()
    q_hbm = hbm_bytes(N, E, B, T, M, n_in)
    headline = (c.get("config_id", 1) == 1 and M == 2 and not args.graph_in_host_memory
                and not args.recompute)
    props = torch.cuda.get_device_properties(dev)
    sm_mhz = (clk or {}).get("sm_max_mhz") or 2070.0
    fp32_peak = props.multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12  # 128 FP32 lanes per SM
    gflop = flops_per_step(N, E, B, T, M) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGE_STEPS_PER_S if headline else None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": _workload_name(c), "parallelism": "replicas",
                   "l2": "flushed by a 512 MB write before every timed step (outside the events)",
                   **({"graph": "edge-indexed arrays in pinned host memory"}
                      if args.graph_in_host_memory else {}),
                   **({"pass_pair": "checkpointing forward + recomputing backward"}
                      if args.recompute else {})},
        "roofline": {"bound": "l2", "kernel": dom, "achieved": achieved, "peak": l2_read,
                     "unit": "GB/s", "frac": achieved / l2_read,
                     "traffic": ncu_traffic(dom) if headline else None,
                     "peak_source": "measured in this run: the fastest of a sweep of dense L2 "
                                    "reads of a 64 MB buffer (" + l2_best["shape"] + ")"},
        "roofline_hbm": {"bound": "hbm", "achieved": q_hbm / (ms_per_step / 1e3) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": q_hbm / (ms_per_step / 1e3) / 1e9 / hbm_peak,
                         "peak_source": f"{hbm_src} (MEASURED_PEAKS.json hbm_gbs)",
                         "bytes_per_step": q_hbm},
        "roofline_step": step_roofline(fb + bb, q_hbm, l2_read, hbm_peak, ms_per_step),
        "l2_probe": {"dense_read_gbs": l2_read, "row_gather_gbs": l2_gather,
                     "sweep": [{"shape": r["shape"], "gbs": round(r["gbs"], 1)} for r in l2_sweep]},
        "flops": {"gflop_per_step": gflop, "achieved_tflops": gflop / ms_per_step,
                  "fp32_fma_peak_tflops": fp32_peak, "frac": gflop / ms_per_step / fp32_peak},
        "kernels": {"forward_ms": f_mean, "backward_ms": b_mean,
                    "forward_gbs": fb / (f_mean / 1e3) / 1e9, "backward_gbs": bb / (b_mean / 1e3) / 1e9,
                    "forward_bytes": fb, "backward_bytes": bb},
        "e2e": {"value": world / (e2e_ms / 1e3), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches[0],
        "memory": mem,
        "clocks": clk,
        "samples_ms": [round(a + b, 4) for a, b in zip(fwd_ms, bwd_ms)],
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(c)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference", "torch-sparse"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--config", type=int, choices=range(5), default=1)
    ap.add_argument("--microsteps", type=int, default=None)
    ap.add_argument("--graph-in-host-memory", action="store_true")
    ap.add_argument("--recompute", action="store_true",
                    help="time the checkpointing forward and the recomputing backward")
    ap.add_argument("--ncu-steps", type=int, default=0,
                    help="run this many steps and nothing else (for a profiler), then exit")
    ap.add_argument("--barrier-probe", action="store_true",
                    help="time the grid-barrier schemes on their own and exit")
    ap.add_argument("--phase-profile", action="store_true",
                    help="per-phase microstep times from the profiling build, then exit")
    args = ap.parse_args()
    if args.phase_profile:
        os.environ["CK_LIBRARY_VARIANT"] = "prof"  # before the library first loads
    if args.barrier_probe:
        run_barrier_probe()
        return

    import workloads
    c = workloads.make(args.config, M=args.microsteps)
    c["config_id"] = args.config
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, c, rank)
        return
    if args.impl == "torch-sparse":
        run_torch_sparse(args, c, rank)
        return
    if args.ncu_steps > 0:
        run_plain_steps(args, c)
        return
    if args.phase_profile:
        run_phase_profile(args, c)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    run_ours(args, c, rank, world, dist)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
