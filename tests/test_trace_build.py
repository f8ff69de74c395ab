"""The trace build (libmoetail_trace.so): it exports the two trace calls of
include/moe_tail_trace.h beside the normal ones, and on a GPU every CTA of a
traced call leaves one record (run in a child process, which loads the trace
build through MOE_TAIL_LIBRARY)."""
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, torch
import moe_decode_tail_gb300 as mt
from moe_decode_tail_gb300 import synth
from moe_decode_tail_gb300.trace import Tracer, launches
tr = Tracer(mt, capacity=4096)
d = synth.config(2)
out = torch.empty((d["b"], d["P"]), dtype=torch.bfloat16, device="cuda")
args = (d["rows"].cuda(), d["idx"].cuda(), d["w"].cuda(), d["gamma"].cuda(), out)
mt.moe_tail_ep_finalize(*args)
torch.cuda.synchronize()
tr.attach()
mt.moe_tail_ep_finalize(*args)
s = synth.config(5, b=16)
ws = torch.empty(mt.moe_tail_workspace_bytes(1, 16, 6144), dtype=torch.uint8, device="cuda")
o2 = torch.zeros((16, 7168), dtype=torch.bfloat16, device="cuda")
mt.moe_shared_expert(s["x"].cuda(), s["w_gate"].cuda(), s["w_up"].cuda(), s["w_down"].cuda(), o2, ws)
torch.cuda.synchronize()
ls = launches(tr.records())
kinds = sorted((k, len(rs)) for k, _, rs in ls)
print(kinds)
assert [k for k, _ in kinds] == [31, 32, 40], kinds
assert all(n > 0 for _, n in kinds)
assert all(r[3] <= r[4][0] <= r[5] for k, _, rs in ls if k in (31, 32) for r in rs)
assert mt.moe_tail_take_device_error() == 0
print("trace ok")
"""


@pytest.fixture(scope="module")
def trace_lib():
    from moe_decode_tail_gb300 import build as cuda_build

    return cuda_build.build(trace=True)


def test_trace_build_exports(trace_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", trace_lib], capture_output=True, text=True).stdout
    names = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert {"moe_tail_trace_attach", "moe_tail_trace_counts", "moe_tail_ep_finalize"} <= names


@pytest.mark.gpu
def test_traced_calls_leave_one_record_per_cta(trace_lib):
    env = dict(os.environ, MOE_TAIL_LIBRARY=trace_lib, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "trace ok" in r.stdout


def _rec(kid, cta, sm, t0, marks, t1):
    return (kid, cta, sm, t0, tuple(marks), t1)


def test_launches_cut_records_into_grids():
    # two launches of a 3-CTA kernel and one of a 2-CTA kernel, records out of
    # order: grouped per kernel by start time, in consecutive grid-sized groups
    from moe_decode_tail_gb300.trace import launches

    recs = [_rec(40, 1, 0, 1010, [0] * 4, 2000), _rec(31, 0, 3, 100, [0] * 4, 900),
            _rec(40, 0, 1, 1000, [0] * 4, 2100), _rec(40, 2, 2, 5, [0] * 4, 800),
            _rec(40, 0, 2, 0, [0] * 4, 700), _rec(40, 1, 5, 3, [0] * 4, 650), _rec(40, 2, 4, 1020, [0] * 4, 2050),
            _rec(31, 1, 4, 110, [0] * 4, 950)]
    ls = launches(recs)
    by_kernel = {}
    for kid, ordinal, rs in ls:
        by_kernel.setdefault(kid, []).append((ordinal, sorted(r[1] for r in rs), min(r[3] for r in rs)))
    assert sorted(by_kernel) == [31, 40]
    assert by_kernel[31] == [(0, [0, 1], 100)]
    assert sorted(by_kernel[40]) == [(0, [0, 1, 2], 0), (1, [0, 1, 2], 1000)]


def test_describe_reads_gemm_and_one_kernel_marks():
    # a GEMM launch: marks 0 (accumulator), 1 (staged), 2 (peers), 3 (stores);
    # the one-kernel latent tail: marks 1 (x formed), 2 (y ready), 0 (accumulator)
    from moe_decode_tail_gb300.trace import describe

    gemm = [_rec(30, c, c, 1000 * c, [1000 * c + 9000, 1000 * c + 9400, 1000 * c + 10400, 1000 * c + 12400],
                 1000 * c + 13800) for c in range(3)]
    fused = [_rec(33, c, c, 500 * c, [500 * c + 11000, 500 * c + 2000, 500 * c + 6500, 0], 500 * c + 14000)
             for c in range(3)]
    lines = describe([(30, 0, gemm), (33, 0, fused)])
    gemm_line = next(line for line in lines if line.startswith("up-projection GEMM"))
    fused_line = next(line for line in lines if line.startswith("latent tail (one kernel)"))
    assert "K loop p50   9.0" in gemm_line
    assert "stage 0.4 peers 1.0 reduce 2.0 barrier+exit 1.4" in gemm_line
    assert "x formed p50   2.0  y ready   6.5  accumulator  11.0" in fused_line
    assert "CTAs    3" in gemm_line and "CTA p50  13.8" in gemm_line


def test_describe_reads_ep_finalize_marks():
    # EP finalize: marks 0 (route list), 1 (rows summed), 2 (cluster barrier), 3 (products)
    from moe_decode_tail_gb300.trace import describe

    ep = [_rec(40, c, c, 100 * c, [100 * c + 900, 100 * c + 2500, 100 * c + 3100, 100 * c + 3600], 100 * c + 4000)
          for c in range(3)]
    line = describe([(40, 0, ep)])[0]
    assert "route list p50   0.9  rows summed   2.5  after cluster barrier   3.1  products   3.6" in line
