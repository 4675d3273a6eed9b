"""Benchmark of the decode-sized weight-only quantized linear layer on GB300.

One "step" is one pass of the whole hot path over the pages' shapes: every
entry point once per (shape, M), each call on its own copy of the packed
weights so that every call streams its weights from HBM:

  * W8 GEMV 8192 x 8192, M = 1                       ("gpt-fast issue #114")
  * W4A16 (256,768), M = 1 (the tiny case)
  * W4A16 (8448,6656) (6656,4096) (6656,19968) (256,6656), M = 1..4
  * W4A8  (39936,6656), M = 1..4, one activation scale per row, and the
    same with one per (row, group of 32)
  * W4A16 (39936,6656) (6656,19968) (1536,512), M = 16, 64
    ("test_int4_quantized_gemm.py": MODEL_SHAPES, SMALL_SHAPES, buckets)

Metric: effective weight GB/s = (bytes of weights + scales + zeros every call
of the step must read) / step time; the JSON line also carries each call's
microseconds, GB/s and fraction of the measured HBM copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --summarize-ncu LAUNCHES.csv   # launch-list shares of an ncu --csv log
"""
from __future__ import annotations

import argparse
import csv
import hashlib
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

import workloads  # noqa: E402

METRIC = "effective weight GB/s and % of GB300 HBM roofline per call at M=1/4/16/64"
UNIT = "GB/s"
WORKLOAD = "decode_linear_suite"

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# the main kernel of a call, from one ncu capture (profiles/ has the command
# and the counters).  Each figure holds only for the kernel sources it was
# taken on: the sha256 of those files, concatenated, must still match, else
# the roofline reports traffic as null.
W4_SOURCES = ("gemv_w4.cu", "w4_stage.cuh", "common.cuh", "timeline.cuh")
W4_DIGEST = "28b51b9b1f50293ac7cddc35fd6e60c4782a0177563e7c532fd45e7a4c405dee"
UMMA_SOURCES = ("gemv_w4_umma.cu", "common.cuh", "tcgen05.cuh", "timeline.cuh")
UMMA_DIGEST = "2378dafd783ae7ce4e982bd07d29ee1dc94c984069c173ab5d24492e4901e06b"
CLUSTER_SOURCES = ("gemv_w4_cluster.cu", "w4_stage.cuh", "common.cuh", "timeline.cuh")
CLUSTER_DIGEST = "12ba6469113f29f542150a022ed4d8ae255622d65df32f6e1a0babdf7db8ff0e"
W8_SOURCES = ("w8.cu", "common.cuh", "timeline.cuh")
W8_DIGEST = "c6e56b97f1283748b2bf5c9a038b70b960b7d278db5cb60df3b6318449743f01"
W8TC_SOURCES = ("gemv_w8_umma.cu", "common.cuh", "tcgen05.cuh")
W8TC_DIGEST = "14fa3efbc3a7d18b41a13f47a384408feab13e645da2e80d2fc489429baf64fb"
MEASURED_TRAFFIC = {
    "w4a8r N=39936 K=6656 M=1": (160875264, W4_SOURCES, W4_DIGEST),
    "w4a8r N=39936 K=6656 M=4": (161396224, W4_SOURCES, W4_DIGEST),
    "w4a16 N=6656 K=4096 M=1": (16232960, CLUSTER_SOURCES, CLUSTER_DIGEST),
    "w4a16 N=39936 K=6656 M=16": (161338624, UMMA_SOURCES, UMMA_DIGEST),
    "w4a16 N=39936 K=6656 M=64": (164112896, UMMA_SOURCES, UMMA_DIGEST),
    "w8 N=8192 K=8192 M=1": (67285760, W8_SOURCES, W8_DIGEST),
    "w8 N=8192 K=8192 M=16": (67767808, W8TC_SOURCES, W8TC_DIGEST),
    "w8 N=8192 K=8192 M=64": (69326080, W8TC_SOURCES, W8TC_DIGEST),
}


def measured_traffic(call):
    """The ncu traffic figure for this call, or None when there is none or
    the kernel sources changed since it was taken."""
    entry = MEASURED_TRAFFIC.get(call)
    if entry is None:
        return None
    nbytes, files, digest = entry
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gemv_w4a16_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest() == digest else None
PAGES_W8_GBS = 1277.19   # "gpt-fast issue #114": compiled int8 GEMV, 8192^2, M=1 (HW unstated)


# ----------------------------------------------------------------- workload

def step_calls():
    """(kind, N, K, M) of one step, in launch order.  Kinds: w8, w4a16, w4a8r
    (W4A8, one activation scale per row), w4a8 (one per group of 32), w4a16c
    (W4A16 with the compact metadata)."""
    calls = [("w8", workloads.W8_GEMV["N"], workloads.W8_GEMV["K"], 1),
             ("w4a16", workloads.TINY_W4A16["N"], workloads.TINY_W4A16["K"], 1)]
    for (N, K) in workloads.W4A16_GEMV_SHAPES:
        for M in workloads.W4A16_GEMV_MS:
            calls.append(("w4a16", N, K, M))
    N, K = workloads.W4A8_SHAPE
    for kind in ("w4a8r", "w4a8"):
        for M in workloads.W4A8_MS:
            calls.append((kind, N, K, M))
    # the compact metadata (uint8 scale / zero codes on fp16 row steps)
    for (N, K) in ((6656, 19968), (8448, 6656)):
        calls.append(("w4a16c", N, K, 1))
    for (N, K) in workloads.TC_SHAPES:
        for M in workloads.TC_MS:
            calls.append(("w4a16", N, K, M))
    for M in workloads.W8_TC_MS:
        calls.append(("w8", workloads.W8_GEMV["N"], workloads.W8_GEMV["K"], M))
    return calls


def weight_bytes(kind, N, K):
    """Bytes of weights + scales + zeros the call must read (the metric)."""
    if kind == "w8":
        return N * K + 2 * N
    if kind == "w4a16c":
        return N * K // 2 + 2 * N * K // 32 + 4 * N
    return N * K // 2 + 3 * N * K // 32


def algorithmic_bytes(kind, N, K, M):
    """Every byte the call must move: weights + scales + zeros, x and out."""
    return weight_bytes(kind, N, K) + 2 * M * K + 2 * M * N


def call_label(kind, N, K, M):
    return "%s N=%d K=%d M=%d" % (kind, N, K, M)


def kernel_name(kind, M, launches=None):
    """The call's main kernel; `launches` (the library's launch count for the
    call) tells the one-launch cluster kernel from the stream-K kernel."""
    if kind == "w8":
        return "w8_kernel<M=%d>" % M if launches == 1 else "w8_umma_kernel<NP=%d>" % ((M + 15) // 16 * 16)
    if kind == "w4a16" and M >= 9:
        return "w4_umma_kernel<NP=%d>" % ((M + 15) // 16 * 16)
    if kind == "w4a16c":
        return "w4_cluster_kernel<A16,compact>"
    mode = "A16" if kind == "w4a16" else "A8"
    if launches == 1:
        return "w4_cluster_kernel<%s>" % mode
    return "w4_kernel<NB=1,%s>" % mode


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = set()
        for _, _, flags in rows:
            for name, flag in zip(names, flags[1:]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


# ---------------------------------------------------------------- GPU arm

class Suite:
    """Device buffers for every call of the step, with rotation pools."""

    def __init__(self, dev, l2_bytes):
        import torch
        from gemv_w4a16_gemm_gb300 import w4q
        self.torch, self.w4q, self.dev = torch, w4q, dev
        self.calls = step_calls()
        self.pools = {}        # (kind, N, K) -> list of weight buffers (copies)
        self.extra = {}        # (kind, N, K) -> scales (w8)
        self.x = {}            # call index -> x (device)
        self.x_host = {}       # call index -> pinned host x (a view of x_host_all)
        self.out = {}          # call index -> out (device)
        self.out_host = {}
        self.ws = {}
        users = {}
        for kind, N, K, M in self.calls:
            key = self.wkey(kind, N, K)
            users[key] = users.get(key, 0) + 1
        for key, n_users in users.items():
            kind, N, K = key
            per = weight_bytes("w4a16c" if kind == "w4c" else kind, N, K)
            copies = max(n_users + 1, -(-3 * l2_bytes // per), 4)
            if kind == "w8":
                W, sc, _ = workloads.w8_inputs(N=N, K=K, M=1)
                base = W.to(dev)
                self.extra[key] = sc.to(dev)
            else:
                W = workloads.w4_weight(N, K).to(dev)
                base = w4q.w4_pack_weights_compact(W) if kind == "w4c" else w4q.w4_pack_weights(W)
                del W
            pool = [base] + [base.clone() for _ in range(copies - 1)]
            self.pools[key] = pool
        # Every call's x and out live in one flat buffer each (on the device
        # and pinned on the host), at 256-byte aligned offsets, so that the
        # end-to-end step moves its inputs and results in one copy each.
        def offsets(sizes):
            offs, o = [], 0
            for n in sizes:
                offs.append(o)
                o += (n + 127) // 128 * 128  # bf16 elements: 256 bytes
            return offs, o
        x_off, x_len = offsets([M * K for _, _, K, M in self.calls])
        o_off, o_len = offsets([M * N for _, N, _, M in self.calls])
        self.x_host_all = torch.zeros(x_len, dtype=torch.bfloat16).pin_memory()
        self.x_all = torch.zeros(x_len, dtype=torch.bfloat16, device=dev)
        self.out_host_all = torch.zeros(o_len, dtype=torch.bfloat16).pin_memory()
        self.out_all = torch.zeros(o_len, dtype=torch.bfloat16, device=dev)
        for i, (kind, N, K, M) in enumerate(self.calls):
            x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
            self.x_host[i] = self.x_host_all[x_off[i]:x_off[i] + M * K].view(M, K)
            self.x_host[i].copy_(x)
            self.x[i] = self.x_all[x_off[i]:x_off[i] + M * K].view(M, K)
            self.out[i] = self.out_all[o_off[i]:o_off[i] + M * N].view(M, N)
            self.out_host[i] = self.out_host_all[o_off[i]:o_off[i] + M * N].view(M, N)
        self.x_all.copy_(self.x_host_all)
        for i, (kind, N, K, M) in enumerate(self.calls):
            if kind == "w8":
                self.ws[i] = torch.empty(max(w4q.w8_workspace_bytes(M, N, K), 16),
                                         dtype=torch.uint8, device=dev)
            elif kind != "w4a16c":
                nbytes = max(w4q.workspace_bytes(M, N, K), 16)
                self.ws[i] = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    @staticmethod
    def wkey(kind, N, K):
        """The weight pool a call reads (the W4 kinds share the packed format,
        except the compact one)."""
        return ("w8" if kind == "w8" else ("w4c" if kind == "w4a16c" else "w4"), N, K)

    def launch(self, i, copy_index, x=None, out=None):
        kind, N, K, M = self.calls[i]
        pool = self.pools[self.wkey(kind, N, K)]
        w = pool[copy_index % len(pool)]
        x = self.x[i] if x is None else x
        out = self.out[i] if out is None else out
        if kind == "w8":
            self.w4q.w8_gemm(x, w, self.extra[self.wkey(kind, N, K)], out=out, workspace=self.ws[i])
        elif kind == "w4a16":
            self.w4q.w4a16_gemm(x, w, N, K, out=out, workspace=self.ws[i])
        elif kind == "w4a8r":
            self.w4q.w4a8_gemm_rowscale(x, w, N, K, out=out, workspace=self.ws[i])
        elif kind == "w4a16c":
            self.w4q.w4a16_gemm_compact(x, w, N, K, out=out)
        else:
            self.w4q.w4a8_gemm(x, w, N, K, out=out, workspace=self.ws[i])

    def call_launches(self, kind, N, K, M):
        """Kernels the library launches for one call."""
        if kind == "w4a16c":
            return 1
        if kind == "w8":
            return self.w4q.w8_kernel_launches(M, N, K)
        return self.w4q.kernel_launches(M, N, K, {"w4a16": False, "w4a8": "group", "w4a8r": "row"}[kind])

    def launches_per_step(self):
        return sum(self.call_launches(*c) for c in self.calls)

    def step_copy_index(self, i):
        """Distinct copy per call within a step (calls of one shape rotate)."""
        kind, N, K, M = self.calls[i]
        key = self.wkey(kind, N, K)
        same = [j for j, c in enumerate(self.calls[:i]) if self.wkey(*c[:3]) == key]
        return len(same)


def _graph(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def measure_calls(suite, reps=3):
    """Per call: R back-to-back launches in one CUDA graph, rotating over
    weight copies (>= 3x L2), timed with CUDA events; median of reps."""
    torch = suite.torch
    res = []
    for i, (kind, N, K, M) in enumerate(suite.calls):
        pool = suite.pools[suite.wkey(kind, N, K)]
        R = max(50, len(pool))
        g = _graph(torch, lambda: [suite.launch(i, r) for r in range(R)])
        times = []
        for _ in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3 / R)
        us = statistics.median(times[1:])
        launches = suite.call_launches(kind, N, K, M)
        res.append(dict(call=call_label(kind, N, K, M), kind=kind, N=N, K=K, M=M,
                        kernel=kernel_name(kind, M, launches), us=us,
                        weight_gbs=weight_bytes(kind, N, K) / us / 1e3,
                        alg_gbs=algorithmic_bytes(kind, N, K, M) / us / 1e3))
        del g
    return res


def run_gpu(args, rank, world, dist):
    import torch
    from gemv_w4a16_gemm_gb300 import w4q

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    peaks = _peaks()
    suite = Suite(dev, l2)

    per_call = measure_calls(suite)
    calls = suite.calls
    step_weight = sum(weight_bytes(k, N, K) for k, N, K, M in calls)

    # the step: every call once on its own weight copy, captured in one graph
    use_ext = True
    try:
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(calls) + 1)]
    except TypeError:
        use_ext, ev = False, None

    def step():
        for i in range(len(calls)):
            suite.launch(i, suite.step_copy_index(i))

    def step_with_events():  # the same calls with an event between each (for the shares)
        for i in range(len(calls)):
            ev[i].record()
            suite.launch(i, suite.step_copy_index(i))
        ev[-1].record()

    # The timed graph holds the calls alone: event nodes between them would
    # break the programmatic launch chaining from one call to the next.
    g = _graph(torch, step)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("w4q_timed_steps")
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(args.steps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    if dist:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    ms = _max_over_ranks(ms, dist)
    in_step_us = None
    if use_ext:
        gi = _graph(torch, step_with_events)
        acc = [0.0] * len(calls)
        for r in range(3 + 5):
            gi.replay()
            torch.cuda.synchronize()
            if r >= 3:
                for i in range(len(calls)):
                    acc[i] += ev[i].elapsed_time(ev[i + 1]) * 1e3 / 5
        in_step_us = acc
        del gi

    # end to end through the public API with host buffers
    # one copy of every call's x in, one of every call's out back (the flat
    # buffers, alignment padding included)
    h2d = suite.x_host_all.numel() * 2
    d2h = suite.out_host_all.numel() * 2

    def e2e_step(s):
        suite.x_all.copy_(suite.x_host_all, non_blocking=True)
        for i in range(len(calls)):
            suite.launch(i, suite.step_copy_index(i))
        suite.out_host_all.copy_(suite.out_all, non_blocking=True)

    for s in range(args.warmup):
        e2e_step(s)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(args.steps):
        e2e_step(s)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / args.steps, dist)
    if dist:
        dist.barrier()
    assert w4q.device_error() == 0, "a kernel reported a bounded-wait timeout"

    if rank != 0:
        return None
    # shares of the step by call (live, inside the timed graph when available)
    step_us = in_step_us if in_step_us else [c["us"] for c in per_call]
    total = sum(step_us)
    for c, u in zip(per_call, step_us):
        c["in_step_us"] = u
        c["share"] = u / total
        c["frac_hbm"] = c["alg_gbs"] / peaks["hbm_gbs"]
    by_kernel = {}
    for c in per_call:
        by_kernel[c["kernel"]] = by_kernel.get(c["kernel"], 0.0) + c["share"]
    roofline = dominant_kernel_roofline(per_call, peaks, args.traffic)
    dom = max(per_call, key=lambda c: c["share"])
    dom_alg = algorithmic_bytes(dom["kind"], dom["N"], dom["K"], dom["M"])
    achieved = dom_alg / dom["us"] / 1e3
    roofline_call = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": measured_traffic(dom["call"]), "kernel": dom["kernel"],
                     "call": dom["call"], "algorithmic_bytes_per_launch": dom_alg,
                     "us_per_launch": round(dom["us"], 3), "peak_source": peaks["source"]}
    tensor = [{"call": c["call"], "kernel": c["kernel"],
               "achieved": round(2.0 * c["M"] * c["N"] * c["K"] / c["us"] / 1e6, 1),
               "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
               "frac": round(2.0 * c["M"] * c["N"] * c["K"] / c["us"] / 1e6 / peaks["bf16_tflops"], 4),
               "peak_source": peaks["source"].replace("copy", "cuBLAS bf16 GEMM, burst")}
              for c in per_call if (c["kind"] == "w4a16" and c["M"] >= 9) or "umma" in c["kernel"]]
    value = replica_value(world, step_weight, ms)
    w8 = next(c for c in per_call if c["kind"] == "w8")
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded randn / randint of the pages' shapes)",
        "config": {"workload": WORKLOAD, "calls_per_step": len(calls),
                   "weight_bytes_per_step": step_weight,
                   "l2": "inputs larger than L2: each call reads its own weight copy; "
                         "the step streams %.2f GB" % (step_weight / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline,
        "roofline_largest_call": roofline_call,
        "tensor_roofline": tensor,
        "e2e": {"value": round(world * step_weight / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "path": "eager calls of the Python binding -> C ABI; every call's x in from pinned host memory in one copy, every out back in one copy"},
        "gpu_launches": suite.launches_per_step() * args.steps,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"]},
        "per_call": [{"call": c["call"], "us": round(c["us"], 3),
                      "in_step_us": round(c["in_step_us"], 3),
                      "weight_gbs": round(c["weight_gbs"], 1),
                      "frac_hbm": round(c["frac_hbm"], 4), "share": round(c["share"], 4)}
                     for c in per_call],
        "kernel_shares": {k: round(v, 4) for k, v in sorted(by_kernel.items())},
        "context": {"pages_w8_compiled_gbs": PAGES_W8_GBS,
                    "w8_8192_ratio_to_pages": round(w8["weight_gbs"] / PAGES_W8_GBS, 2),
                    "pages_hardware": "unstated (W8); A100 (INT4 decode kernels)"},
    }
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def dominant_kernel_roofline(per_call, peaks, traffic_override=None):
    """Roofline of the kernel with the largest share of the step, over all its
    calls: algorithmic bytes per launch (their mean) over its mean launch
    duration (each call's per-launch CUDA-event time), against the measured
    copy bandwidth; traffic = ncu DRAM bytes per launch when every one of its
    calls has a current figure, else null."""
    kern = {}
    for c in per_call:
        k = kern.setdefault(c["kernel"], {"share": 0.0, "bytes": 0, "us": 0.0, "calls": []})
        k["share"] += c["share"]
        k["bytes"] += algorithmic_bytes(c["kind"], c["N"], c["K"], c["M"])
        k["us"] += c["us"]
        k["calls"].append(c["call"])
    name = max(kern, key=lambda n: kern[n]["share"])
    k = kern[name]
    n = len(k["calls"])
    achieved = k["bytes"] / k["us"] / 1e3
    traffic, traffic_calls = None, []
    if traffic_override is not None:
        traffic = traffic_override
    else:
        t = {c: measured_traffic(c) for c in k["calls"]}
        traffic_calls = [c for c, v in t.items() if v is not None]
        if traffic_calls:
            # per launch: the mean over the calls of this kernel with a
            # current capture (their algorithmic bytes are within 0.1% of
            # the kernel's mean)
            traffic = sum(t[c] for c in traffic_calls) / len(traffic_calls)
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
            "traffic_calls": traffic_calls,
            "kernel": name, "share_of_step": round(k["share"], 4), "launches_per_step": n,
            "calls": k["calls"], "algorithmic_bytes_per_launch": round(k["bytes"] / n),
            "us_per_launch": round(k["us"] / n, 3), "peak_source": peaks["source"]}


def replica_value(world, step_bytes, ms_max):
    """Whole-job GB/s of `world` replicas that each stream `step_bytes` per
    step, timed by the slowest rank (`ms_max`, milliseconds per step)."""
    return world * step_bytes / (ms_max * 1e-3) / 1e9


def _max_over_ranks(v, dist):
    if not dist:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured (MEASURED_PEAKS.json: STREAM-style copy)"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ----------------------------------------------------------- CPU baseline

def _oracle_sample(frac_rows):
    """A bounded sample of the step: for every call, the first rows of its
    weight (whole 16-row tiles), computed by the CPU oracle from the packed
    bytes (unpack, dequant, fp64 matmul).  Returns (run, weight bytes)."""
    import numpy as np
    import oracle
    jobs = []
    total = 0
    cache = {}
    for kind, N, K, M in step_calls():
        rows = max(16, int(N * frac_rows) // 16 * 16)
        rows = min(rows, N)
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
        if kind == "w8":
            W, sc, _ = workloads.w8_inputs(N=N, K=K, M=1)
            Wr = W[:rows].numpy().copy()
            scr = sc[:rows].clone()
            jobs.append(("w8", x, (Wr, scr), rows, K))
        elif kind == "w4a16c":
            Wd = workloads.w4_weight(N, K)[:rows].contiguous()
            jobs.append((kind, x, oracle.pack_w4c(*oracle.quantize_w4c(Wd, rows, K)), rows, K))
        else:
            key = (N, K)
            if key not in cache:
                Wd = workloads.w4_weight(N, K)
                rr = min(N, max(16, int(N * frac_rows) // 16 * 16))
                q, s, z = oracle.quantize_w4(Wd[:rr].contiguous(), rr, K)
                cache[key] = oracle.pack_w4(q, s, z)
            packed = cache[key][: (rows // 16) * (K // 256) * 2432]
            jobs.append((kind, x, packed, rows, K))
        total += weight_bytes(kind, rows, K)

    def run():
        for kind, x, data, rows, K in jobs:
            if kind == "w8":
                oracle.w8(x, data[0], data[1])
                continue
            if kind == "w4a16c":
                oracle.w4a16c(x, *oracle.unpack_w4c(data, rows, K))
                continue
            q, s, z = oracle.unpack_w4(data, rows, K)
            if kind == "w4a16":
                oracle.w4a16(x, q, s, z)
            elif kind == "w4a8r":
                xq, sx = oracle.act_quant_row(x, K)
                oracle.w4a8_row(xq, sx, q, s, z)
            else:
                xq, sx = oracle.act_quant(x, K)
                oracle.w4a8(xq, sx, q, s, z)
        return None

    del np
    return run, total


def _timed_sample(seconds, start_frac=0.002):
    """Time the oracle on a sample grown to about `seconds` of host work."""
    run, nbytes = _oracle_sample(start_frac)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    frac = min(1.0, start_frac * max(1.0, seconds / max(dt, 1e-3)))
    if frac > start_frac * 1.5:
        run, nbytes = _oracle_sample(frac)
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, dt, frac


def cpu_baseline(seconds):
    """The oracle on the host cores: OpenMP over all of them, and one thread."""
    import oracle
    cores = oracle.set_threads(0)
    value, dt, frac = _timed_sample(seconds)
    oracle.set_threads(1)
    value1, dt1, frac1 = _timed_sample(seconds / 3, start_frac=0.001)
    oracle.set_threads(cores)
    sample = ("first %.2f%% of the rows (whole 16-row tiles, >= 16) of every call of "
              "the step: unpack + dequant + fp64 matmul on the host")
    return {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": round(dt, 2), "sample": sample % (100 * frac),
            "single_thread": {"value": round(value1, 4), "unit": UNIT, "cores": 1,
                              "seconds": round(dt1, 2), "sample": sample % (100 * frac1)}}


def run_reference(args, rank):
    """The oracle as the reference arm: K timed steps of a bounded sample."""
    if rank != 0:
        return None
    import oracle
    cores = oracle.set_threads(0)
    frac = 0.01
    run, nbytes = _oracle_sample(frac)
    for _ in range(max(1, args.warmup)):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    sample = ("first %.1f%% of the rows (whole 16-row tiles, >= 16) of every call of the step, "
              "unpack + dequant + fp64 matmul on the host" % (100 * frac))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, the pages' shapes)",
        "config": {"workload": WORKLOAD, "sample_weight_bytes_per_step": nbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def profile_call(spec, launches):
    """Launch one call configuration `launches` times after two warm-ups (for
    an ncu capture of that kernel; prints no bench line)."""
    import torch
    from gemv_w4a16_gemm_gb300 import w4q
    kind, N, K, M = spec.split(",")
    N, K, M = int(N), int(K), int(M)
    dev = torch.device("cuda", 0)
    x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M)).to(dev)
    if kind == "w8":
        W, sc, _ = workloads.w8_inputs(N=N, K=K, M=1)
        W, sc = W.to(dev), sc.to(dev)
        ws = torch.empty(max(w4q.w8_workspace_bytes(M, N, K), 16), dtype=torch.uint8, device=dev)
        fn = lambda: w4q.w8_gemm(x, W, sc, workspace=ws)  # noqa: E731
    else:
        if kind == "w4a16c":
            packed = w4q.w4_pack_weights_compact(workloads.w4_weight(N, K).to(dev))
            fn = lambda: w4q.w4a16_gemm_compact(x, packed, N, K)  # noqa: E731
        else:
            packed = w4q.w4_pack_weights(workloads.w4_weight(N, K).to(dev))
            op = {"w4a16": w4q.w4a16_gemm, "w4a8": w4q.w4a8_gemm,
                  "w4a8r": w4q.w4a8_gemm_rowscale}[kind]
            ws = torch.empty(max(w4q.workspace_bytes(M, N, K), 16), dtype=torch.uint8, device=dev)
            fn = lambda: op(x, packed, N, K, workspace=ws)  # noqa: E731
    for _ in range(2 + launches):
        fn()
    torch.cuda.synchronize()
    assert w4q.device_error() == 0
    print("profiled %s x %d" % (spec, launches))


# ----------------------------------------------------------- ncu summary

def summarize_ncu(path):
    """Per-kernel launches, total time and share from an ncu --csv launch list
    (metric gpu__time_duration.sum)."""
    per = {}
    with open(path, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    hdr_i = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    hdr = rows[hdr_i]
    ki, mi, vi, ui = (hdr.index("Kernel Name"), hdr.index("Metric Name"),
                      hdr.index("Metric Value"), hdr.index("Metric Unit"))
    for r in rows[hdr_i + 1:]:
        if len(r) <= vi or r[mi] != "gpu__time_duration.sum":
            continue
        v = float(r[vi].replace(",", ""))
        unit = r[ui]
        ns = v * {"nsecond": 1, "usecond": 1e3, "msecond": 1e6, "second": 1e9}.get(unit, 1)
        name = r[ki]
        n, t = per.get(name, (0, 0.0))
        per[name] = (n + 1, t + ns)
    total = sum(t for _, t in per.values())
    out = []
    for name, (n, t) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        out.append("%-90s %6d launches %12.1f us total %6.2f%%" % (name[:90], n, t / 1e3,
                                                                  100 * t / total))
    return "\n".join(out)


# ------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=int(os.environ.get("WORLD_SIZE", "1")))
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the dominant kernel, when known")
    ap.add_argument("--summarize-ncu", metavar="CSV")
    ap.add_argument("--profile-call", metavar="KIND,N,K,M",
                    help="launch one call config only (for ncu); prints no bench line")
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args(argv)
    if args.summarize_ncu:
        print(summarize_ncu(args.summarize_ncu))
        return 0
    if args.profile_call:
        profile_call(args.profile_call, args.launches)
        return 0
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
    if args.impl == "reference":
        line = run_reference(args, rank)
    else:
        line = run_gpu(args, rank, world, dist)
    if dist:
        dist.destroy_process_group()
    if line is not None and rank == 0:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
