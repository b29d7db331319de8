#!/usr/bin/env python
"""Benchmark of the GB300 verify step of speculative decoding.

A step is one pass of the whole hot path over one batch: the row-statistics
pass over every logit (phase 1) and the accept test + final draw (phase 2),
for the default workload "linear_b256_g8_v128256_bf16" (B=256 requests,
gamma=8 drafts, V=128256, bf16 logits, Zipf-shaped logits at T=0.7).

Prints ONE JSON line (rank 0):
  value      verified draft positions / s over all ranks (B * gamma per step),
             inputs resident in HBM, CUDA events on the launching stream;
  e2e        the same metric through the C-ABI host-buffer call with pinned
             HOST buffers: host->device copy of the step's inputs, the verify
             and the device->host copy of its outputs inside the timed region;
  roofline   the dominant kernel: algorithmic bytes per launch / its
             CUDA-event time against the measured HBM copy peak.  The kernel
             times come from steps issued as separate phases with events
             around each, AFTER the timed region (the timed steps are plain
             verify calls only);
  workloads  the other named workloads, each measured the same way in this
             process (step time, positions/s, requests/s, GB/s, fractions);
  cpu_baseline  the float64 oracle on the host cores, on a bounded sample.

--impl reference times the oracle (the only other implementation there is)
on the host cores instead.  Multi-rank (torchrun): every rank verifies its
own batch (weak scaling, no collective on the data path); the timing is the
max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_64_gb300 import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "linear_b256_g8_v128256_bf16"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
METRIC = "verified draft positions/sec and HBM GB/s (fraction of 8 TB/s) per verify step"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the end-to-end timing (default: enough for ~4 GB of "
                         "host-to-device copies, 20 to 2000 steps)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--topk", type=int, default=0,
                    help="linear workloads: time specdec_verify_linear_topk (the top-k residual "
                         "approximation) with this many candidates instead of the exact step")
    ap.add_argument("--alpha", action="store_true",
                    help="linear workloads: also time specdec_row_alpha (the opt-in acceptance-rate "
                         "pass) on the same inputs and report its bandwidth")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="skip timing the step replayed from CUDA graphs (reported beside the "
                         "eager value, never instead of it)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other named workloads (measured after the headline one, "
                         "reported under 'workloads')")
    ap.add_argument("--workload-steps", type=int, default=400,
                    help="timed steps of each of the other workloads")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (a smaller case for profiling; not a bench line)")
    ap.add_argument("--vocab", type=int, default=None,
                    help="override V (a smaller case for profiling; not a bench line)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------
# distributed plumbing (weak scaling: one independent batch per rank)
# ----------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float, device) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "row_stats_kernel": ("row_stats.cu", "stats_role.cuh", "stats_stage.cuh", "common.cuh"),
}


def kernel_source_hash(kernel: str = "row_stats_kernel") -> str:
    src = os.path.join(ROOT, "speculative_decoding_verification_64_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(src, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str = "row_stats_kernel"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", kernel.replace("_kernel", "") + "_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    want = kernel_source_hash(kernel)
    for ln in lines:
        if ln.startswith("#") or not ln.strip():
            continue
        kv = dict(x.split("=", 1) for x in ln.split() if "=" in x)
        if kv.get("workload") == workload and kv.get("kernel_sha") == want:
            try:
                return float(kv["bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [ln for t, ln in self.lines if self.t0 is not None and self.t0 <= t <= (self.t1 or t) + 0.06]
        if not rows:
            rows = [ln for _, ln in self.lines[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in rows:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def algorithmic_bytes(w, n_accepted_rows_rejected: float) -> dict:
    """Bytes the method must move per step: every logit once, the q row of
    each rejected request, the gathered p/q values and the small per-request
    inputs and outputs."""
    es = w.elem_bytes
    R = w.rows
    gamma = R - 1 if isinstance(w, W.LinearWorkload) else R - 1
    logits = w.B * R * w.V * es
    q_rows = n_accepted_rows_rejected * w.V * es
    small = w.B * gamma * (2 * es + 4) + w.B * R * 4 + w.B * 4 + w.B * (R + 4) * 4
    return dict(logits=logits, q_rows=q_rows, small=small, total=logits + q_rows + small)


def _verify_fn(binding, w, linear, out, ws, topk):
    """One public verify call on an input set (the step), on a given stream."""
    def verify(x, on):
        if topk:
            binding.verify_linear_topk(*x, topk, out=out, workspace=ws, stream=on)
        elif linear:
            binding.verify_linear(*x, out=out, workspace=ws, stream=on)
        else:
            binding.verify_tree(*x, w.max_depth, out=out, workspace=ws, stream=on)
    return verify


def _phase_fns(binding, w, linear, out, ws):
    """The two phases of the two-launch path, issued separately (per-kernel times)."""
    def stats(x, on):
        if linear:
            binding.row_stats(x[0], x[3], ws, q=x[1], draft_tokens=x[2], stream=on)
        else:
            binding.row_stats(x[0], x[4], ws, stream=on)

    def finalize(x, on):
        if linear:
            binding.linear_finalize(*x, out, ws, stream=on)
        else:
            binding.tree_finalize(*x, w.max_depth, out, ws, stream=on)
    return stats, finalize


class Setup:
    """A workload's resident input sets, outputs and workspace on the device."""

    def __init__(self, binding, w, device, topk=0):
        self.w = w
        self.linear = isinstance(w, W.LinearWorkload)
        inputs = (binding.linear_inputs_to_device(w, device) if self.linear
                  else binding.tree_inputs_to_device(w, device))
        # resident input sets used in turn, enough of them that a step's inputs
        # were last touched at least 3 x L2 bytes of other inputs ago (two for
        # the large workloads, many copies of the small ones)
        set_bytes = sum(t.numel() * t.element_size() for t in inputs)
        self.n_sets, self.l2_note = input_rotation(set_bytes)
        self.sets = [inputs] + [tuple(t.clone() for t in inputs) for _ in range(self.n_sets - 1)]
        self.dt = binding.dtype_code(inputs[0])
        self.ws = binding.alloc_workspace(w.B, w.rows, w.V, self.dt, device)
        self.out = (binding.LinearOut.empty(w.B, w.gamma, device) if self.linear
                    else binding.TreeOut.empty(w.B, w.N, w.max_depth, device))
        self.topk = topk if self.linear else 0
        self.units = w.B * w.gamma if self.linear else w.B * (w.N - 1)
        self.verify = _verify_fn(binding, w, self.linear, self.out, self.ws, self.topk)
        self.stats, self.finalize = _phase_fns(binding, w, self.linear, self.out, self.ws)
        # launches of one verify call: 1 (one kernel) or 2 (stats pass, then the draw)
        if self.topk:
            self.launches, self.path = 2, binding.PATH_TWO_LAUNCHES
        elif self.linear:
            self.launches = binding.verify_linear_launches(inputs[0], inputs[1])
            self.path = binding.verify_linear_path(inputs[0], inputs[1])
        else:
            self.launches, self.path = 2, binding.PATH_TWO_LAUNCHES
        self.binding = binding

    def marshal(self, stream):
        """The C-ABI verify call of every input set with its arguments marshalled
        once (as a C caller holds them), so that the timed steps measure the
        library, not the Python binding's per-call checks."""
        import ctypes
        b, w, o, ws = self.binding, self.w, self.out, self.ws
        lib = b.load_library()
        P = b._ptr
        sp = ctypes.c_void_p(stream.cuda_stream)
        calls = []
        for x in self.sets:
            if self.topk:
                fn = lib.specdec_verify_linear_topk
                a = (P(x[0]), P(x[1]), self.dt, P(x[2]), P(x[3]), P(x[4]), w.B, w.gamma, w.V,
                     self.topk, P(o.n_accepted), P(o.out_tokens), P(o.final_token),
                     P(o.is_bonus), P(o.row_status), P(o.p_draft), P(ws), ws.numel(), sp)
            elif self.linear:
                fn = lib.specdec_verify_linear
                a = (P(x[0]), P(x[1]), self.dt, P(x[2]), P(x[3]), P(x[4]), w.B, w.gamma, w.V,
                     P(o.n_accepted), P(o.out_tokens), P(o.final_token), P(o.is_bonus),
                     P(o.row_status), P(o.p_draft), P(ws), ws.numel(), sp)
            else:
                fn = lib.specdec_verify_tree
                a = (P(x[0]), P(x[1]), self.dt, P(x[2]), P(x[3]), P(x[4]), P(x[5]), w.B, w.N,
                     w.V, w.max_depth, P(o.n_accepted), P(o.path_nodes), P(o.out_tokens),
                     P(o.final_token), P(o.is_bonus), P(o.row_status), P(o.p_node), P(ws),
                     ws.numel(), sp)
            calls.append((fn, a))
        self.calls = calls

    def call(self, s):
        fn, a = self.calls[s % self.n_sets]
        rc = fn(*a)
        if rc != 0:
            raise RuntimeError(f"{fn.__name__}: {self.binding.status_string(rc)}")


PAUSE_CYCLES = 200_000  # ~0.1 ms at 2 GHz
# Warm-up: the requested steps (at least 3), and at least this much wall time
# of steps.  A 20-step timed region after 3 warm-up steps measured 0.7 us a
# step slower than after 400 (about 50 ms): the GPU needs that long under load
# to settle (the SM clock read 2070 MHz throughout).
WARM_SECONDS = 0.1


def time_steps(torch, st, K, warmup, stream, dist, sampler=None):
    """K verify calls back to back between two events (after the warm-up
    calls); every call is the public C entry point, nothing else is issued in
    between.  Sets st.warmup_run to the number of warm-up calls made."""
    st.marshal(stream)
    # the requested warm-up steps, timed; then, back to back with no wait in
    # between, as many more as fill WARM_SECONDS at that rate
    n0 = max(warmup, 3)
    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for s in range(n0):
        st.call(s)
    w1.record(stream)
    torch.cuda.synchronize()
    per_step = max(w0.elapsed_time(w1) / 1e3 / n0, 1e-6)
    n = max(n0, int(WARM_SECONDS / per_step))
    for s in range(n0, n):
        st.call(s)
    torch.cuda.synchronize()
    # and one untimed run of the timed region's own shape (K steps from a
    # synchronised start): the first such run after the warm-up measured
    # slower than the ones after it
    for s in range(K):
        st.call(s)
    st.warmup_run = n + K
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("begin")
    # A device-side pause (torch's bounded sleep kernel, ~0.1 ms) ahead of the
    # start event, so that the host has queued the first calls when the timed
    # region starts: the host's latency in issuing the first call is not
    # device time of a step (the e2e figure counts the host).
    if hasattr(torch.cuda, "_sleep"):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(PAUSE_CYCLES)
    t0.record(stream)
    for s in range(K):
        st.call(s)
    t1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("end")
    dist.barrier()
    return t0.elapsed_time(t1)


def time_phases(torch, st, n, stream):
    """Per-kernel times, measured apart from the timed steps: `n` steps issued
    as separate phases with events around each (two-launch path), or the
    one-kernel call between two events.  Medians in ms."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for s in range(n):
        x = st.sets[s % st.n_sets]
        e0, e1, e2 = ev[s]
        e0.record(stream)
        if st.launches == 1 or st.topk:
            st.verify(x, stream)
            e1.record(stream)
        else:
            st.stats(x, stream)
            e1.record(stream)
            st.finalize(x, stream)
        e2.record(stream)
    torch.cuda.synchronize()
    a = float(np.median([e[0].elapsed_time(e[1]) for e in ev]))
    b = float(np.median([e[1].elapsed_time(e[2]) for e in ev]))
    return a, b


def kernel_names(st):
    if st.topk:
        return "row_stats_kernel + topk_draw_kernel"
    return st.binding.PATH_KERNELS[st.path]


def workload_line(torch, binding, st, ms_per_step, k1_ms, k2_ms, peak, name):
    """Per-workload figures: step time, throughput, algorithmic GB/s and the
    dominant kernel's roofline (from the separately timed phases)."""
    w = st.w
    nb = st.out.is_bonus.cpu().numpy()
    rejected = 0.0 if st.topk else float((nb == 0).sum())
    ab = algorithmic_bytes(w, rejected)
    gbs = ab["total"] / (ms_per_step / 1e3) / 1e9
    es = w.elem_bytes
    spr = -(-w.V * es // 8192)
    kname = kernel_names(st)
    if st.launches == 1 and not st.topk:
        # the step is that one kernel: its time is the step's (events around
        # single launches would add the launch gap of an idle GPU)
        k1_ms = ms_per_step
    if st.topk or st.launches == 1:
        k_bytes, traffic = ab["total"], None
    else:
        k_bytes = ab["logits"] + w.B * w.rows * spr * 16
        traffic = ncu_traffic(name, kname)
    k_gbs = k_bytes / (k1_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(k_gbs, 1),
                "peak": peak, "unit": "GB/s", "frac": round(k_gbs / peak, 4),
                "traffic": traffic, "algorithmic_bytes_per_launch": int(k_bytes),
                "avg_launch_us": round(k1_ms * 1e3, 2)}
    if k1_ms > ms_per_step * 1.0001:
        # a kernel cannot take longer than the step it belongs to: the phase
        # timing is not trustworthy, so no fraction is claimed
        roofline.update(achieved=None, frac=None,
                        note=f"kernel median {k1_ms * 1e3:.2f} us > step {ms_per_step * 1e3:.2f} us")
    if st.topk:
        phase = {"verify_topk": round(k1_ms * 1e3, 2)}
    elif st.launches == 1:
        phase = {"verify_one_launch": round(k1_ms * 1e3, 2)}
    else:
        phase = {"row_stats": round(k1_ms * 1e3, 2), "finalize": round(k2_ms * 1e3, 2)}
    return dict(ab=ab, gbs=gbs, roofline=roofline, phase=phase)


PHASE_STEPS = 64  # separately issued phase-split steps for the per-kernel medians


def run_ours(args, dist):
    import torch
    from speculative_decoding_verification_64_gb300 import binding
    from speculative_decoding_verification_64_gb300 import build as builder

    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    dist.init("nccl")
    if dist.local_rank == 0:
        builder.build()
    dist.barrier()
    binding.load_library()

    w = W.make_workload(args.workload, B=args.batch, V=args.vocab, seed_offset=1000 * dist.rank)
    st = Setup(binding, w, device, args.topk)
    linear = st.linear
    launches, l2_note = st.launches, st.l2_note
    stream = torch.cuda.current_stream(device)
    K = args.steps
    peak, peak_kind = measured_peaks()

    sampler = ClockSampler(dist.local_rank) if dist.rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    total_ms = time_steps(torch, st, K, args.warmup, stream, dist, sampler)
    warmup_run = st.warmup_run
    clocks = sampler.stop() if sampler else None
    # outputs of the last timed step (its rejected requests set the q-row bytes)
    torch.cuda.synchronize()
    n_acc_sum = float(st.out.n_accepted.sum().item())
    k1_ms, k2_ms = time_phases(torch, st, max(PHASE_STEPS, 1), stream)

    total_ms = dist.max(total_ms, device)
    ms_per_step = total_ms / K
    value = dist.sum(st.units, device) * K / (total_ms / 1e3)
    line = workload_line(torch, binding, st, ms_per_step, k1_ms, k2_ms, peak,
                         _workload_name(args))
    roofline = dict(line["roofline"], peak_kind=peak_kind)

    # ---- the same steps replayed from CUDA graphs (launch-bound sizes) ----
    graph = None
    if args.graph and not st.topk:
        # a serving loop replays one graph on fixed buffers: up to 4 graphs here
        # (fewer than the eager rotation leaves the small inputs warm in L2)
        n_graphs = min(st.n_sets, 4)
        graphs = []
        for i in range(n_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                st.verify(st.sets[i], None)
            graphs.append(g)
        for s_ in range(max(args.warmup, 3)):
            graphs[s_ % n_graphs].replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize()
        g0.record()
        for s_ in range(K):
            graphs[s_ % n_graphs].replay()
        g1.record()
        torch.cuda.synchronize()
        g_ms = dist.max(g0.elapsed_time(g1), device)
        graph = {"ms_per_step": round(g_ms / K, 5),
                 "value": round(dist.sum(st.units, device) * K / (g_ms / 1e3), 1),
                 "unit": "positions/s", "graphs": n_graphs, "l2_warm": n_graphs < st.n_sets}
        del graphs

    # ---- the opt-in acceptance-rate pass, timed on its own ----
    alpha = None
    if args.alpha and linear:
        alpha = time_alpha(torch, binding, st, K, stream, peak)

    # ---- e2e: pinned host buffers through the public verify call ----
    e2e = run_e2e(args, w, linear, device, stream, dist, st.units)

    # ---- the other workloads, each measured the same way in this process ----
    others = None
    if (not args.no_workloads and dist.world == 1 and args.batch is None
            and args.vocab is None and not args.topk):
        others = {}
        del st
        torch.cuda.empty_cache()
        for name in sorted(W.WORKLOADS):
            if name == args.workload:
                continue
            others[name] = measure_other(torch, binding, name, device, stream, dist, peak,
                                         args.workload_steps)
            torch.cuda.empty_cache()

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, linear, w.B * w.gamma if linear else w.B * (w.N - 1),
                           args.cpu_seconds)

    ab = line["ab"]
    gbs = line["gbs"]
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "positions/s",
        "n_gpus": dist.world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "warmup_run": warmup_run,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": _config(w, _workload_name(args), linear, l2_note, args.topk if linear else 0),
        "requests_per_s": round(dist.sum(w.B, device) * K / (total_ms / 1e3), 1),
        "accepted_tokens_per_s": round(dist.sum(n_acc_sum + w.B, device) * K / (total_ms / 1e3), 1),
        "gbs": round(gbs, 1),
        "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
        "frac_of_measured_hbm": round(gbs / peak, 4),
        "algorithmic_bytes_per_step": int(ab["total"]),
        "phase_us": dict(line["phase"], steps=PHASE_STEPS,
                         how="median of separately issued steps after the timed region"),
        "roofline": roofline,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": launches * K,
        "graph": graph,
        "alpha_pass": alpha,
        "workloads": others,
        "clocks": clocks,
    }
    if dist.rank == 0:
        print(json.dumps(res), flush=True)
    dist.close()


def time_alpha(torch, binding, st, K, stream, peak):
    """The opt-in acceptance-rate pass on the workspace of a verify call on set 0
    (it reads only M and S of each row from it, so the passes over the other
    sets move the same bytes)."""
    w = st.w
    x0 = st.sets[0]
    binding.verify_linear(*x0, out=st.out, workspace=st.ws, stream=stream)
    for s_ in range(3):
        x = st.sets[s_ % st.n_sets]
        binding.row_alpha(x[0], x[1], x[3], st.ws, stream=stream)
    torch.cuda.synchronize()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    n_a = max(1, min(K, 200))
    a0.record(stream)
    for s_ in range(n_a):
        x = st.sets[s_ % st.n_sets]
        binding.row_alpha(x[0], x[1], x[3], st.ws, stream=stream)
    a1.record(stream)
    torch.cuda.synchronize()
    a_us = a0.elapsed_time(a1) / n_a * 1e3
    a_bytes = 2 * w.B * w.gamma * w.V * w.elem_bytes
    return {"kernel": "row_alpha_kernel", "avg_launch_us": round(a_us, 2),
            "bytes_per_launch": int(a_bytes), "achieved_gbs": round(a_bytes / a_us / 1e3, 1),
            "peak_gbs": peak, "frac": round(a_bytes / a_us / 1e3 / peak, 4), "launches": n_a}


def measure_other(torch, binding, name, device, stream, dist, peak, steps):
    """One of the other named workloads, measured in the same process as the
    headline: resident input sets used in turn (cold L2), `steps` timed verify
    calls, then the separately issued phase steps for the kernel times."""
    w = W.make_workload(name)
    st = Setup(binding, w, device)
    ms = time_steps(torch, st, steps, 10, stream, dist) / steps
    k1_ms, k2_ms = time_phases(torch, st, PHASE_STEPS, stream)
    line = workload_line(torch, binding, st, ms, k1_ms, k2_ms, peak, name)
    res = {"B": w.B, "V": w.V, "dtype": w.dtype,
           "gamma" if st.linear else "N": w.gamma if st.linear else w.N,
           "steps": steps, "us_per_step": round(ms * 1e3, 2),
           "positions_per_s": round(st.units / (ms / 1e3), 1),
           "requests_per_s": round(w.B / (ms / 1e3), 1),
           "gbs": round(line["gbs"], 1),
           "frac_of_8tbs": round(line["gbs"] / NOMINAL_HBM_GBS, 4),
           "frac_of_measured_hbm": round(line["gbs"] / peak, 4),
           "algorithmic_bytes_per_step": int(line["ab"]["total"]),
           "launches_per_step": st.launches,
           "phase_us": line["phase"], "roofline": line["roofline"], "l2": st.l2_note}
    del st
    return res


L2_BYTES = 129_000_000  # GB300 L2
def input_rotation(set_bytes: int):
    """How many resident copies of a step's inputs to use in turn so that a
    step's inputs were last touched at least 3 x L2 bytes of other inputs ago."""
    n = max(2, -(-3 * L2_BYTES // set_bytes) + 1)
    return n, (f"{n} resident input sets used in turn, {set_bytes * n / 1e6:.0f} MB in all; "
               f"a step's inputs were last touched >= 3 x L2 ago")


def _workload_name(args):
    name = args.workload
    if args.batch is not None or args.vocab is not None:
        name += f" (override B={args.batch} V={args.vocab})"
    return name


def _host_set_bytes(w) -> int:
    """Bytes of one step's inputs as the GPU arm holds them on the device."""
    arrs = ([w.logits, w.q, w.draft_tokens, w.temperature, w.uniforms]
            if isinstance(w, W.LinearWorkload)
            else [w.logits, w.q, w.node_tokens, w.parent, w.temperature, w.uniforms])
    return int(sum(a.nbytes for a in arrs))


def _config(w, name, linear, l2_note, topk=0):
    c = {"workload": name, "B": w.B, "V": w.V, "dtype": w.dtype, "l2": l2_note}
    if topk:
        c["topk_residual"] = topk  # the approximate correction draw, not the exact method
    if linear:
        c["gamma"] = w.gamma
        c["greedy_requests"] = int((w.temperature == 0).sum())
    else:
        c["N"] = w.N
        c["max_depth"] = w.max_depth
    return c


def run_e2e(args, w, linear, device, stream, dist, units):
    """The C-ABI host-buffer call (specdec_verify_linear_host / _tree_host):
    every step copies its inputs from page-locked host memory, verifies and
    copies its outputs back.  Two staging buffers on two streams, used in turn,
    so that step i+1's copies may overlap step i's kernels; the arguments are
    marshalled once, outside the timed region."""
    import ctypes
    import torch
    from speculative_decoding_verification_64_gb300 import binding

    lib = binding.load_library()
    host_in = (binding.linear_inputs_to_host(w) if linear else binding.tree_inputs_to_host(w))
    dt = binding.dtype_code(host_in[0])
    P = binding._ptr
    streams = [torch.cuda.Stream(device) for _ in range(2)]
    calls = []
    for j in range(2):
        if linear:
            out = binding._host_out(None, lambda: binding.LinearOut.empty(w.B, w.gamma, "cpu"))
            nbytes = binding.linear_staging_size(w.B, w.gamma, w.V, dt)
        else:
            out = binding._host_out(None, lambda: binding.TreeOut.empty(w.B, w.N, w.max_depth,
                                                                        "cpu"))
            nbytes = binding.tree_staging_size(w.B, w.N, w.V, w.max_depth, dt)
        st = torch.empty(nbytes, dtype=torch.uint8, device=device)
        sp = ctypes.c_void_p(streams[j].cuda_stream)
        if linear:
            a = (P(host_in[0]), P(host_in[1]), dt, P(host_in[2]), P(host_in[3]), P(host_in[4]),
                 w.B, w.gamma, w.V, P(out.n_accepted), P(out.out_tokens), P(out.final_token),
                 P(out.is_bonus), P(out.row_status), P(out.p_draft), P(st), nbytes, sp)
            fn = lib.specdec_verify_linear_host
        else:
            a = (P(host_in[0]), P(host_in[1]), dt, P(host_in[2]), P(host_in[3]), P(host_in[4]),
                 P(host_in[5]), w.B, w.N, w.V, w.max_depth, P(out.n_accepted),
                 P(out.path_nodes), P(out.out_tokens), P(out.final_token), P(out.is_bonus),
                 P(out.row_status), P(out.p_node), P(st), nbytes, sp)
            fn = lib.specdec_verify_tree_host
        calls.append((fn, a, st, out))
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(v.numel() * v.element_size() for v in vars(calls[0][3]).values() if v is not None)

    def one(i):
        fn, a = calls[i % 2][:2]
        rc = fn(*a)
        if rc != 0:
            raise RuntimeError(f"{fn.__name__}: {binding.status_string(rc)}")

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    n = args.e2e_steps
    if n is None:  # about 4 GB of host-to-device copies
        n = min(2000, max(20, -(-4_000_000_000 // h2d)))
    n = max(1, min(n, args.steps))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for s in streams:
        s.wait_event(e0)
    for i in range(n):
        one(i)
    for s in streams:
        ev = torch.cuda.Event()
        ev.record(s)
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(e0.elapsed_time(e1), device)
    val = dist.sum(units, device) * n / (ms / 1e3)
    return {"value": round(val, 1), "unit": "positions/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "ms_per_step": round(ms / n, 4),
            "h2d_gbs": round(h2d * n / (ms / 1e3) / 1e9, 1),
            "call": fn_name(linear),
            "pipelined": "two staging buffers on two streams in turn: step i+1's copies may "
                         "overlap step i's kernels"}


def fn_name(linear):
    return "specdec_verify_linear_host" if linear else "specdec_verify_tree_host"


# ----------------------------------------------------------------------------
# the oracle on the host cores
# ----------------------------------------------------------------------------

def _oracle_run(o, w, linear):
    if linear:
        return o.verify_linear_workload(w, diagnostics=False)
    return o.verify_tree_workload(w, diagnostics=False)


def cpu_baseline(w, linear, units, seconds):
    import oracle
    oracle.build()
    per_req = units / w.B
    # size the sample: time a few requests, then take enough for ~`seconds`
    probe = w.subset(np.arange(min(w.B, max(1, oracle.num_threads()))))
    t = time.perf_counter()
    _oracle_run(oracle, probe, linear)
    dt = max(time.perf_counter() - t, 1e-6)
    reps = max(1, int(seconds / dt))
    n_req = probe.B * reps
    t = time.perf_counter()
    for _ in range(reps):
        _oracle_run(oracle, probe, linear)
    el = time.perf_counter() - t
    cores = oracle.num_threads()
    # the same code on one thread, on a shorter sample (about a fifth of the time)
    oracle.set_threads(1)
    one = w.subset(np.arange(1))
    t = time.perf_counter()
    _oracle_run(oracle, one, linear)
    d1 = max(time.perf_counter() - t, 1e-6)
    reps1 = max(1, int(seconds / 5 / d1))
    t = time.perf_counter()
    for _ in range(reps1):
        _oracle_run(oracle, one, linear)
    el1 = time.perf_counter() - t
    oracle.set_threads(cores)
    return {"value": round(n_req * per_req / el, 1), "unit": "positions/s",
            "cores": cores, "kind": "oracle",
            "sample": f"{n_req} requests ({reps} x the first {probe.B} of the workload), "
                      f"{el:.1f} s, float64 C with OpenMP over requests",
            "single_thread": {"value": round(reps1 * per_req / el1, 1), "unit": "positions/s",
                              "sample": f"{reps1} x the first request, {el1:.1f} s"}}


def run_reference(args, dist):
    if dist.rank != 0:
        return
    import oracle
    oracle.build()
    w = W.make_workload(args.workload, B=args.batch, V=args.vocab)
    linear = isinstance(w, W.LinearWorkload)
    units_per_req = w.gamma if linear else w.N - 1
    cores = oracle.num_threads()
    # one step = `cores` requests of the workload (one per thread), cycling through the batch
    per_step = max(1, min(cores, w.B))
    subsets = [w.subset((np.arange(per_step) + i * per_step) % w.B)
               for i in range(max(1, w.B // per_step))]
    for s in range(max(args.warmup, 3)):
        _oracle_run(oracle, subsets[s % len(subsets)], linear)
    t = time.perf_counter()
    for s in range(args.steps):
        _oracle_run(oracle, subsets[s % len(subsets)], linear)
    el = time.perf_counter() - t
    value = args.steps * per_step * units_per_req / el
    sample = (f"{per_step} requests per step ({args.steps} steps), float64 C oracle, "
              f"OpenMP over requests")
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "positions/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, _workload_name(args), linear, input_rotation(_host_set_bytes(w))[1]),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 1), "unit": "positions/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
        return 0
    run_ours(args, dist)
    return 0


if __name__ == "__main__":
    sys.exit(main())
