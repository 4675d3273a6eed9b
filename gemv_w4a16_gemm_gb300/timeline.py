"""Per-call timelines of back-to-back calls (profiling build).

Builds libw4q_timeline.so: the library compiled with -DW4Q_TIMELINE, whose
kernels stamp %globaltimer at fixed points (csrc/timeline.cuh).  For each
requested call, a CUDA graph of R back-to-back launches rotating over copies
of the weight (more than L2 in total) is replayed; the stamps of one replay
are grouped by call (the k-th stamp of an event from a block belongs to the
k-th call) and every event is placed relative to the end of the previous
call's last CTA.  The table gives, per event, the median over the calls of
its first / median / last CTA.  Stamping adds an atomic per event, so the
calls run a little slower than in the ordinary build.

    python gemv_w4a16_gemm_gb300/timeline.py KIND,N,K,M[,SPLIT] ...
        KIND: w4a16, w4a8 (scale per group), w4a8r (scale per row), w8

Runs on one GPU.
"""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

LIB = os.path.join(HERE, "libw4q_timeline.so")
READERS = ("w4q_timeline_read_w4", "w4q_timeline_read_cluster", "w4q_timeline_read_w8",
           "w4q_timeline_read_umma")
EVENTS = {
    1: "prologue (counter reset): start", 2: "prologue (counter reset): waited",
    4: "prologue (act_prep): start", 5: "prologue (act_prep): waited",
    10: "stream-K kernel: CTA start", 11: "stream-K: producer waited",
    13: "stream-K: first stage full", 14: "stream-K: last stage done",
    15: "stream-K: chunk flushed", 16: "stream-K: CTA end",
    20: "cluster kernel: CTA start", 21: "cluster: waited", 22: "cluster: activations ready",
    23: "cluster: last stage done", 25: "cluster: CTA end",
    30: "w8 kernel: CTA start", 31: "w8: waited", 32: "w8: last stage done",
    40: "tcgen05 kernel: CTA start", 41: "tcgen05: x producer waited", 42: "tcgen05: CTA end",
    44: "prologue (B operand): start", 45: "prologue (B operand): waited",
    47: "partial-sum launch: waited", 48: "partial-sum launch: block end",
}
END_EVENTS = (16, 25, 32, 42)


def build_lib():
    from gemv_w4a16_gemm_gb300 import build as b
    b.BUILD = os.path.join(HERE, "_build", "timeline")
    b.LIB = LIB
    orig = b._flags
    b._flags = lambda extra=(): orig(("-DW4Q_TIMELINE", *extra))
    return b.build()


def _group_by_call(stamps):
    t = stamps[:, 0].astype(np.int64)
    ev = (stamps[:, 1] >> 32).astype(np.int64)
    blk = (stamps[:, 1] & 0xFFFFFFFF).astype(np.int64)
    calls = {}
    for e in np.unique(ev):
        m = ev == e
        tt, bb = t[m], blk[m]
        order = np.lexsort((tt, bb))
        tt, bb = tt[order], bb[order]
        k = np.zeros(len(bb), np.int64)
        for i in range(1, len(bb)):
            k[i] = k[i - 1] + 1 if bb[i] == bb[i - 1] else 0
        for kk in np.unique(k):
            calls.setdefault(int(kk), {})[int(e)] = tt[k == kk]
    return calls


def summarize(stamps):
    """Rows (event, first, median, last CTA in us after the previous call's
    last CTA end, medians over calls) and the call period in us."""
    calls = _group_by_call(stamps)
    n = len(calls)
    end = next((e for e in END_EVENTS if e in calls.get(0, {})), None)
    rows, periods = {}, []
    for k in range(3, n - 2):
        prev = calls[k - 1].get(end)
        if prev is None:
            continue
        ref = prev.max()
        for e, tt in calls[k].items():
            rows.setdefault(e, []).append(((tt.min() - ref) / 1e3, np.median(tt - ref) / 1e3,
                                           (tt.max() - ref) / 1e3))
        if end in calls[k]:
            periods.append((calls[k][end].max() - ref) / 1e3)
    table = [(EVENTS.get(e, str(e)), *np.median(np.array(v), axis=0)) for e, v in sorted(rows.items())]
    return table, (float(np.median(periods)) if periods else None)


def run(specs, R=20):
    import torch
    import workloads
    from gemv_w4a16_gemm_gb300 import w4q
    w4q.LIB_PATH = LIB
    lib = w4q.lib()
    for name in READERS:
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]

    def read():
        out = []
        for name in READERS:
            buf = np.zeros(2 << 18, np.uint64)
            n = ctypes.c_uint32(0)
            assert getattr(lib, name)(buf.ctypes.data, ctypes.byref(n)) == 0
            out.append(buf[: 2 * n.value].reshape(-1, 2))
        return np.concatenate(out)

    dev = torch.device("cuda", 0)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
    for spec in specs:
        parts = spec.split(",")
        kind, N, K, M = parts[0], int(parts[1]), int(parts[2]), int(parts[3])
        split = int(parts[4]) if len(parts) > 4 else None
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M)).to(dev)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        if kind == "w8":
            W, sc, _ = workloads.w8_inputs(N=N, K=K, M=1)
            base, sc = W.to(dev), sc.to(dev)
            ws = torch.empty(max(w4q.w8_workspace_bytes(M, N, K), 16), dtype=torch.uint8, device=dev)
        else:
            base = w4q.w4_pack_weights(workloads.w4_weight(N, K).to(dev))
            ws = torch.empty(max(w4q.workspace_bytes(M, N, K, split_k=split), 16),
                             dtype=torch.uint8, device=dev)
        pool = [base] + [base.clone() for _ in range(max(4, -(-3 * l2 // base.numel())) - 1)]
        op = {"w4a16": w4q.w4a16_gemm, "w4a8": w4q.w4a8_gemm,
              "w4a8r": w4q.w4a8_gemm_rowscale}.get(kind)

        def calls():
            for r in range(R):
                w = pool[r % len(pool)]
                if kind == "w8":
                    w4q.w8_gemm(x, w, sc, out=out, workspace=ws)
                else:
                    op(x, w, N, K, split_k=split, out=out, workspace=ws)

        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            calls()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        read()
        g.replay()
        torch.cuda.synchronize()
        table, period = summarize(read())
        assert w4q.device_error() == 0
        print("\n### %s N=%d K=%d M=%d split=%s: period %.2f us per call (stamped build)\n"
              % (kind, N, K, M, "library" if split is None else split, period or float("nan")))
        print("| event | first CTA | median CTA | last CTA |\n|---|---:|---:|---:|")
        for name, a, b, c in table:
            print("| %s | %.2f | %.2f | %.2f |" % (name, a, b, c))
        sys.stdout.flush()
        del g, pool
        torch.cuda.empty_cache()


if __name__ == "__main__":
    build_lib()
    run(sys.argv[1:])
