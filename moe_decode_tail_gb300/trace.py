"""Per-CTA timeline of the decode tail's kernels, from the trace build.

The trace build (build.build(trace=True) -> _build/libmoetail_trace.so,
include/moe_tail_trace.h) has every CTA record %globaltimer at entry, at up to
four marks and at exit.  This module attaches a record buffer, runs work, and
turns the records into per-launch spans and the GEMM epilogue's phases.

    python -m moe_decode_tail_gb300.trace          # one bench.py decode step (b = 64), timed as the bench times it
    python -m moe_decode_tail_gb300.trace --latent-one-kernel   # the latent tail's one-kernel form, b = 1, 4, 16

prints, for one step in the middle of a graph replay of ten steps: each
kernel launch's first and last CTA start and its end (µs from the step's
first CTA), the median CTA duration, and for the GEMMs the median time from
CTA start to accumulator complete (the K loop) and the median epilogue
phases (staging, waiting for cluster peers, reduction and stores, second
barrier, exit).  Set MOE_TAIL_LIBRARY before the first library call, as
main() does; records are 64 bytes.
"""
from __future__ import annotations

import collections
import ctypes
import importlib.util
import os
import statistics

import torch

KERNELS = {10: "ep_finalize (route-parallel)", 11: "tp_finalize (route-parallel)", 12: "latent_norm",
           20: "tp_finalize (staged)", 21: "latent_norm (staged)", 30: "up-projection GEMM", 31: "gate/up GEMM",
           32: "down GEMM", 33: "latent tail (one kernel)", 40: "ep_finalize"}
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class Tracer:
    """Owns the device record buffer of an attached trace build."""

    def __init__(self, mt, capacity: int = 1 << 16):
        self.mt, self.L = mt, mt.lib()
        if not hasattr(self.L, "moe_tail_trace_attach"):
            raise RuntimeError("the loaded library is not the trace build (set MOE_TAIL_LIBRARY first)")
        self.L.moe_tail_trace_attach.argtypes = [ctypes.c_void_p, ctypes.c_uint]
        self.L.moe_tail_trace_counts.argtypes = [ctypes.POINTER(ctypes.c_uint)] * 2
        self.capacity = capacity
        self.buf = torch.zeros((capacity, 8), dtype=torch.int64, device="cuda")

    def attach(self):
        if self.L.moe_tail_trace_attach(ctypes.c_void_p(self.buf.data_ptr()), self.capacity) != 0:
            raise RuntimeError("moe_tail_trace_attach failed")

    def records(self) -> list[tuple]:
        g, f = ctypes.c_uint(), ctypes.c_uint()
        if self.L.moe_tail_trace_counts(ctypes.byref(g), ctypes.byref(f)) != 0:
            raise RuntimeError("moe_tail_trace_counts failed")
        half = self.capacity // 2
        rows = torch.cat([self.buf[:min(g.value, half)], self.buf[half:half + min(f.value, self.capacity - half)]])
        out = []
        for t0, m0, m1, m2, m3, t1, ids, _ in rows.cpu().tolist():
            out.append((ids >> 48, ids & 0xFFFFFFFF, (ids >> 32) & 0xFFFF, t0, (m0, m1, m2, m3), t1))
        return out


def launches(records) -> list[tuple[int, int, list]]:
    """(kernel id, ordinal, CTA records) per launch: a kernel's records sorted
    by start time, cut into consecutive groups of its grid size."""
    by = collections.defaultdict(list)
    for r in records:
        by[r[0]].append(r)
    out = []
    for kid, rs in by.items():
        n = max(r[1] for r in rs) + 1
        rs.sort(key=lambda r: r[3])
        out += [(kid, i // n, rs[i:i + n]) for i in range(0, len(rs), n)]
    return out


def describe(group: list[tuple[int, int, list]]) -> list[str]:
    """Lines for one set of launches (times in µs from their earliest CTA)."""
    base = min(r[3] for _, _, rs in group for r in rs)
    lines = []
    for kid, _, rs in sorted(group, key=lambda x: min(r[3] for r in x[2])):
        p50 = lambda f: statistics.median(f(r) for r in rs) / 1e3
        line = (f"{KERNELS.get(kid, kid):30s} CTAs {len(rs):4d}  first start {(min(r[3] for r in rs) - base) / 1e3:6.1f}"
                f"  last start {(max(r[3] for r in rs) - base) / 1e3:6.1f}  end {(max(r[5] for r in rs) - base) / 1e3:6.1f}"
                f"  CTA p50 {p50(lambda r: r[5] - r[3]):5.1f}")
        if kid == 33 and all(r[4][0] and r[4][1] and r[4][2] for r in rs):  # marks 1, 2: x formed, y ready
            line += (f"  x formed p50 {p50(lambda r: r[4][1] - r[3]):5.1f}  y ready {p50(lambda r: r[4][2] - r[3]):5.1f}"
                     f"  accumulator {p50(lambda r: r[4][0] - r[3]):5.1f}")
        elif kid in (20, 21) and all(r[4][2] and r[4][3] for r in rs):  # staged finalize, first pass
            line += (f"  first rows p50 {p50(lambda r: r[4][0] - r[3]):5.1f}  pass consumed "
                     f"{p50(lambda r: r[4][2] - r[3]):5.1f}  after cluster barrier {p50(lambda r: r[4][3] - r[3]):5.1f}")
        elif kid in (30, 31, 32) and all(r[4][0] for r in rs):
            line += f"  K loop p50 {p50(lambda r: r[4][0] - r[3]):5.1f}"
            if all(r[4][3] for r in rs):
                line += (f"  epilogue: stage {p50(lambda r: r[4][1] - r[4][0]):.1f}"
                         f" peers {p50(lambda r: r[4][2] - r[4][1]):.1f} reduce {p50(lambda r: r[4][3] - r[4][2]):.1f}"
                         f" barrier+exit {p50(lambda r: r[5] - r[4][3]):.1f}")
        lines.append(line)
    return lines


def latent_one_kernel(mt, sizes=(1, 4, 16), calls: int = 6) -> None:
    """The latent tail's one-kernel form (MOE_TAIL_LATENT_FUSED=1) at the decode
    shape (tp = 8 latent slots, L = 3584, H = 7168, 9 shared slots), each call
    alone (synchronised after it), without and with both promises: per call the
    CTA spans and the median times from CTA start to x formed, y ready and
    accumulator complete.  The weights rotate over six copies (> 2x L2)."""
    dev = torch.device("cuda", 0)
    L, H, TP, TPS = 3584, 7168, 8, 9
    g = torch.Generator(device=dev).manual_seed(7)
    wc = [(0.02 * torch.randn(H, L, device=dev, generator=g)).to(torch.bfloat16) for _ in range(6)]
    gamma = (1 + 0.05 * torch.randn(L, device=dev, generator=g)).to(torch.bfloat16)
    tracer = Tracer(mt)
    prev = os.environ.get("MOE_TAIL_LATENT_FUSED")
    os.environ["MOE_TAIL_LATENT_FUSED"] = "1"
    try:
        for b in sizes:
            lat = (0.5 * torch.randn(TP, b, L, device=dev, generator=g)).to(torch.bfloat16)
            sh = (0.5 * torch.randn(TPS, b, H, device=dev, generator=g)).to(torch.bfloat16)
            y = torch.empty((b, L), dtype=torch.bfloat16, device=dev)
            out = torch.empty((b, H), dtype=torch.bfloat16, device=dev)
            for promises in (False, True):
                def call(i):
                    mt.moe_tail_latent_up_flags(lat, gamma, wc[i % len(wc)], sh, out, y, inputs_ready=promises,
                                                weights_static=promises)
                for i in range(calls):  # warm-up
                    call(i)
                torch.cuda.synchronize()
                tracer.attach()
                for i in range(calls):
                    call(i)
                    torch.cuda.synchronize()
                print(f"-- b = {b}, promises {promises}")
                for kid, i, rs in launches(tracer.records())[1:3]:
                    print("  " + describe([(kid, i, rs)])[0])
    finally:
        if prev is None:
            os.environ.pop("MOE_TAIL_LATENT_FUSED", None)
        else:
            os.environ["MOE_TAIL_LATENT_FUSED"] = prev


def main() -> None:
    import sys

    from moe_decode_tail_gb300 import build as cuda_build

    os.environ["MOE_TAIL_LIBRARY"] = cuda_build.build(trace=True)
    import moe_decode_tail_gb300 as mt

    if "--latent-one-kernel" in sys.argv[1:]:
        torch.cuda.set_device(0)
        latent_one_kernel(mt)
        if mt.moe_tail_take_device_error() != 0:
            raise RuntimeError("a kernel wait expired")
        return

    spec = importlib.util.spec_from_file_location("bench_trace", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cpu, w = bench.make_workload(dev)
    stream = torch.cuda.Stream(dev, priority=-1)
    side = torch.cuda.Stream(dev, priority=0)
    tracer = Tracer(mt)
    with torch.cuda.stream(stream):
        for _ in range(3):
            bench.run_step(mt, w, stream, side=side)
    torch.cuda.synchronize()
    steps = 10
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(steps):
            bench.run_step(mt, w, stream, side=side)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    tracer.attach()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    print(f"{steps} steps: {a.elapsed_time(b) * 1e3 / steps:.1f} us per step (trace build)")
    ls = launches(tracer.records())
    for step in (steps // 2 - 1, steps // 2):
        print(f"-- step {step}")
        for line in describe([x for x in ls if x[1] == step]):
            print("  " + line)
    if mt.moe_tail_take_device_error() != 0:
        raise RuntimeError("a kernel wait expired")


if __name__ == "__main__":
    main()
