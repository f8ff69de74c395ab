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
