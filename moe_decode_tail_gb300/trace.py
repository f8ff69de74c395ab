"""Per-CTA timeline of the decode tail's kernels, from the trace build.

The trace build (build.build(trace=True) -> _build/libmoetail_trace.so,
include/moe_tail_trace.h) has every CTA record %globaltimer at entry, at up to
four marks and at exit.  Tracer attaches a record buffer and reads the
records back; launches() groups them into launches and describe() prints
each launch's first and last CTA start and its end (µs from the earliest
CTA), the median CTA duration, and for the GEMMs the median time from CTA
start to accumulator complete (the K loop) and the median epilogue phases.
Load the trace build by setting MOE_TAIL_LIBRARY before the first library
call; records are 64 bytes.  bench.py --trace runs it on the decode step.
"""
from __future__ import annotations

import collections
import ctypes
import statistics

import torch

KERNELS = {10: "ep_finalize (route-parallel)", 11: "tp_finalize (route-parallel)", 12: "latent_norm",
           20: "tp_finalize (staged)", 21: "latent_norm (staged)", 30: "up-projection GEMM", 31: "gate/up GEMM",
           32: "down GEMM", 33: "latent tail (one kernel)", 34: "down + up-projection GEMM", 40: "ep_finalize"}


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
        elif kid == 40 and all(r[4][0] and r[4][1] and r[4][2] and r[4][3] for r in rs):  # EP finalize
            line += (f"  route list p50 {p50(lambda r: r[4][0] - r[3]):5.1f}  rows summed {p50(lambda r: r[4][1] - r[3]):5.1f}"
                     f"  after cluster barrier {p50(lambda r: r[4][2] - r[3]):5.1f}"
                     f"  products {p50(lambda r: r[4][3] - r[3]):5.1f}")
        elif kid in (30, 31, 32, 34) and all(r[4][0] for r in rs):
            line += f"  K loop p50 {p50(lambda r: r[4][0] - r[3]):5.1f}"
            if all(r[4][3] for r in rs):
                line += (f"  epilogue: stage {p50(lambda r: r[4][1] - r[4][0]):.1f}"
                         f" peers {p50(lambda r: r[4][2] - r[4][1]):.1f} reduce {p50(lambda r: r[4][3] - r[4][2]):.1f}"
                         f" barrier+exit {p50(lambda r: r[5] - r[4][3]):.1f}")
        lines.append(line)
    return lines
