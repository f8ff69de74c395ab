#!/usr/bin/env python
"""Benchmark of the GB300 MoE decode tail.

One step = one decode batch of b = 64 tokens through every row of the tail's
hot path, each call on its decode shape:
  1. EP finalize        rows [8, *, 4096] (top-8 of 128 experts, 16 per slot) -> out [64, 4096]
  2. expert-TP finalize K-partials [8, 512, 4096] (top-8) -> out [64, 4096]
  3. latent tail        latent [8, 64, 3584] -> RMS norm -> y . W_up^T [7168 x 3584]
                        + shared partials [8, 64, 7168] -> out [64, 7168]
  4. shared expert      x [64, 7168]; W_gate, W_up [6144, 7168]; W_down [7168, 6144];
                        added into the latent tail's output
By default (--composition two_branch_fused) 3 and 4 run on a side stream as
the shared expert's gate/up, the latent norm, then one kernel streaming the
down projection and the up-projection (moe_tail_up_project_shared_down); 1
and 2 run beside them on a high-priority stream.  Gate/up and the norm take
the inputs-ready promise (their inputs are the step's own), the GEMMs the
static-weights promise.
Inputs are seeded and synthetic (random-init weights); every input is resident
in device memory before timing.  A step touches about 390 MB, three times the
L2, so every input is read cold without flushing.  Steps are replayed from a
CUDA graph whose timed replays carry no events; one more replay after the
timed region carries per-call CUDA events (in every tenth step) for each
call's duration.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference]

Under torchrun every rank runs an independent replica (the tail shards by
token with no exchange on one GPU); the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "MoE-tail tokens/s and µs/layer at b; achieved HBM GB/s vs ~8 TB/s peak"
NOMINAL_HBM_GBS = 8000.0  # the metric's nominal peak; fractions are also given against the measured copy rate
B = 64                    # decode tokens per step
TP, P, K_ROUTES, E = 8, 4096, 8, 128
L, H, I = 3584, 7168, 6144

# Algorithmic bytes per call (reads + writes the method needs; intermediates
# such as y and h that a fused kernel would keep on chip are not counted).
BYTES = {
    "ep_finalize": B * K_ROUTES * P * 2 + TP * B * K_ROUTES * 4 + B * K_ROUTES * 4 + P * 2 + B * P * 2,
    "tp_finalize": TP * B * K_ROUTES * P * 2 + B * K_ROUTES * 4 + B * K_ROUTES * 4 + P * 2 + B * P * 2,
    "latent_up": TP * B * L * 2 + L * 2 + H * L * 2 + TP * B * H * 2 + B * H * 2,
    "shared_expert": 3 * I * H * 2 + B * H * 2 + 2 * B * H * 2,
}
FLOPS = {"latent_up": 2 * B * H * L, "shared_expert": 2 * B * 3 * I * H}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--graph-steps", type=int, default=50, help="steps captured per CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload isolated timings")
    ap.add_argument("--composition", default="two_branch_fused",
                    choices=["two_branch_fused", "two_branch", "two_branch_one_call", "latent_main"],
                    help="how the step orders the weight-streaming calls (see run_step)")
    ap.add_argument("--only-config", type=int, choices=[1, 2, 3, 4, 5, 6, 7], default=None,
                    help="run one workload's call alone --calls times and exit (for profiling the call); 6: the "
                         "default step's side-stream calls at b = 64 (gate/up, latent norm, up-projection with the "
                         "down projection); 7: config 5's down projection as the K-split GEMM and as the "
                         "persistent kernel on 56 CTAs")
    ap.add_argument("--calls", type=int, default=4)
    ap.add_argument("--trace", choices=["step", "latent"], default=None,
                    help="per-CTA timeline from the trace build: ten decode steps as one graph (step), or the latent "
                         "tail's one-kernel form alone at b = 1, 4, 16 (latent)")
    ap.add_argument("--sequential", action="store_true",
                    help="run the four calls in order on one stream (shared expert accumulating into out)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist if world > 1 else None


def aggregate(seconds: float, units: float, dist=None, device="cpu"):
    """(max seconds over ranks, total units over ranks)."""
    if dist is None:
        return seconds, units
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        try:
            ident = str(self.dev)
            try:
                uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
                ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            except Exception:
                pass
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, sm_max = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            try:
                power = float(parts[2])
            except ValueError:  # "[N/A]": the clock sample still counts
                power = None
            rows.append((sm, sm_max, power, parts[3:]))
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        powers = [r[2] for r in rows if r[2] is not None]
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(powers) if powers else None, "samples": len(rows), "reasons": reasons}


# ----------------------------------------------------------------------------- workload

def make_workload(dev, b=B, weights=None):
    """The step's inputs at b tokens (seeded; config 2's EP shape, config 3's
    expert-TP shape, the latent tail and the shared expert), with the
    workspaces, output buffers and events.  weights: a workload whose weight
    tensors (W_up, W_gate, W_up of the shared expert, W_down) to share."""
    from moe_decode_tail_gb300 import synth

    ep = synth.config(2, b=b)                             # tp=8, P=4096, top-8 of 128
    tp = synth.config(3, b=b)                             # expert-TP
    lat = synth.latent_up_inputs(synth.SEED_BASE + 4, b=b, with_weight=weights is None)
    sh = synth.config(5, b=b, with_weights=weights is None)  # H=7168, I=6144
    cpu = dict(ep=ep, tp=tp, lat=lat, sh=sh)
    g = lambda t: t.to(dev)
    w = dict(
        ep_rows=g(ep["rows"]), ep_idx=g(ep["idx"]), ep_w=g(ep["w"]), ep_gamma=g(ep["gamma"]),
        tp_part=g(tp["partials"]), tp_idx=g(tp["idx"]), tp_w=g(tp["w"]), tp_gamma=g(tp["gamma"]),
        latent=g(lat["latent"]), lat_gamma=g(lat["gamma"]), shared=g(lat["shared"]), x=g(sh["x"]),
    )
    if weights is None:
        w.update(w_up=g(lat["w_up"]), w_gate=g(sh["w_gate"]), w_up_s=g(sh["w_up"]), w_down=g(sh["w_down"]))
    else:
        w.update({k: weights[k] for k in ("w_up", "w_gate", "w_up_s", "w_down")})
    import moe_decode_tail_gb300 as mt

    w["out_ep"] = torch.empty((b, P), dtype=torch.bfloat16, device=dev)
    w["out_tp"] = torch.empty((b, P), dtype=torch.bfloat16, device=dev)
    w["out"] = torch.empty((b, H), dtype=torch.bfloat16, device=dev)
    w["ws_lat"] = torch.empty(mt.moe_tail_workspace_bytes(0, b, L), dtype=torch.uint8, device=dev)
    w["y"] = w["ws_lat"][: b * L * 2].view(torch.bfloat16).view(b, L)
    w["ws_sh"] = torch.empty(mt.moe_tail_workspace_bytes(1, b, I), dtype=torch.uint8, device=dev)
    # the latent tail's shared partials plus one slot that receives the shared expert's output;
    # "shared" is a view of the first TP slots, so data copied into it reaches both compositions
    w["shared9"] = torch.empty((TP + 1, b, H), dtype=torch.bfloat16, device=dev)
    w["shared9"][:TP].copy_(w["shared"])
    w["shared"] = w["shared9"][:TP]
    w["d_slot"] = w["shared9"][TP]
    w["fork"], w["join"], w["normed"] = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    w["h_ready"] = torch.cuda.Event()
    return cpu, w


EVENTS_PER_STEP = 12  # (start, end) of EP, TP, latent norm, up-projection, shared gate/up (or all), down


def run_step(mt, w, stream, events=None, side=None):
    """The four calls of one step.  events: optional list of EVENTS_PER_STEP
    events, a (start, end) pair per call recorded on the call's stream (the
    latent tail has two pairs, for when its norm and up-projection run as
    separate calls; in one call the second pair is empty).

    With a side stream the weight-streaming calls run beside the routed
    finalize calls, as the Kimi-K3 tail runs its shared expert (its output is
    pushed into the tail's reduce-scatter partials).  The default,
    "two_branch_fused": on the side stream moe_shared_gate_up (static
    weights, inputs ready), moe_tail_latent_norm (inputs ready), then
    moe_tail_up_project_shared_down (static weights), which adds bf16(d)
    after the shared partials.  "two_branch": on the side stream the
    shared expert's two calls, moe_shared_gate_up and moe_shared_down, with
    static weights (each requests its first weight tiles before waiting for
    the preceding kernel), write d = bf16(down(h)) into the last of the
    latent tail's shared-partial slots ("two_branch_one_call": one
    moe_shared_expert call instead); then moe_tail_latent_up_flags follows
    with both promises -- inputs ready (the latent partials are read while
    the down projection drains) and static weights -- and adds d with the
    other slots in its epilogue; the call enqueues the norm and the
    up-projection.  With "latent_main" the latent tail runs on the main
    stream after the finalize calls, beside the shared expert's gate/up, and
    the down projection then adds d into its output.
    EP and expert-TP finalize run on the main stream, which joins the side
    stream at the end of the step.  Without a side stream the calls run in
    order (moe_tail_latent_up in one call) and the shared expert accumulates
    into the latent tail's output."""
    ev = events or [None] * EVENTS_PER_STEP

    def rec(i, st):
        if ev[i] is not None:
            ev[i].record(st)

    ready = w.get("finalize_ready", False)  # EP and TP with the inputs-ready promise

    def ep(st):
        rec(0, st)
        mt.moe_tail_ep_finalize_flags(w["ep_rows"], w["ep_idx"], w["ep_w"], w["ep_gamma"], w["out_ep"],
                                      gain_center=1.0, eps=1e-6, weight_before_norm=True, inputs_ready=ready,
                                      stream=st)
        rec(1, st)

    def tp(st):
        rec(2, st)
        mt.moe_tail_tp_finalize_flags(w["tp_part"], w["tp_idx"], w["tp_w"], w["tp_gamma"], w["out_tp"],
                                      gain_center=1.0, eps=1e-6, weight_before_norm=True, inputs_ready=ready,
                                      stream=st)
        rec(3, st)

    def shared_expert(st, out, accumulate):
        rec(8, st)
        mt.moe_shared_expert(w["x"], w["w_gate"], w["w_up_s"], w["w_down"], out, w["ws_sh"], accumulate=accumulate,
                             stream=st)
        rec(9, st)
        rec(10, st)
        rec(11, st)

    if side is None:
        ep(stream)
        tp(stream)
        rec(4, stream)
        mt.moe_tail_latent_up(w["latent"], w["lat_gamma"], w["w_up"], w["shared"], w["out"], w["ws_lat"], eps=1e-6,
                              stream=stream)
        rec(5, stream)
        rec(6, stream)
        rec(7, stream)
        shared_expert(stream, w["out"], True)
        return
    comp = w.get("composition", "two_branch_fused")
    if comp == "latent_main":
        # the latent tail on the finalize stream after EP and TP, beside the
        # shared expert's gate/up; the down projection then adds d into the
        # latent tail's output (out = bf16(out + bf16(d)), the sequential
        # composition's arithmetic) once both are done
        bx = w["x"].shape[0]
        ws_h = w["ws_sh"][: bx * I * 2].view(torch.bfloat16).view(bx, I)
        w["fork"].record(stream)
        side.wait_event(w["fork"])
        rec(8, side)
        mt.moe_shared_gate_up(w["x"], w["w_gate"], w["w_up_s"], ws_h, weights_static=True, stream=side)
        rec(9, side)
        w["h_ready"].record(side)
        ep(stream)
        tp(stream)
        rec(4, stream)
        mt.moe_tail_latent_up_flags(w["latent"], w["lat_gamma"], w["w_up"], w["shared"], w["out"], w["y"], eps=1e-6,
                                    inputs_ready=True, weights_static=True, stream=stream)
        rec(5, stream)
        rec(6, stream)
        rec(7, stream)
        stream.wait_event(w["h_ready"])
        rec(10, stream)
        mt.moe_shared_down(ws_h, w["w_down"], w["out"], accumulate=True, weights_static=True, stream=stream)
        rec(11, stream)
        return
    if comp == "two_branch_fused":
        # the shared expert's gate/up, the latent norm, then the down projection
        # and the up-projection in one kernel (d added after the shared partials).
        # Gate/up takes both promises: its weights are static and x, the step's
        # input, is complete before the previous step's last kernel ends, so its
        # whole K loop may run while that kernel drains (h is written after it).
        bx = w["x"].shape[0]
        ws_h = w["ws_sh"][: bx * I * 2].view(torch.bfloat16).view(bx, I)
        w["fork"].record(stream)
        side.wait_event(w["fork"])
        rec(8, side)
        mt.moe_shared_gate_up(w["x"], w["w_gate"], w["w_up_s"], ws_h, weights_static=True, inputs_ready=True,
                              stream=side)
        rec(9, side)
        rec(4, side)
        mt.moe_tail_latent_norm(w["latent"], w["lat_gamma"], w["y"], eps=1e-6, inputs_ready=True, stream=side)
        rec(5, side)
        rec(6, side)
        mt.moe_tail_up_project_shared_down(w["y"], w["w_up"], w["shared"], ws_h, w["w_down"], w["out"],
                                           weights_static=True, stream=side)
        rec(7, side)
        rec(10, side)
        rec(11, side)
        w["join"].record(side)
        ep(stream)
        tp(stream)
        stream.wait_event(w["join"])
        return
    w["fork"].record(stream)
    side.wait_event(w["fork"])
    if comp != "two_branch_one_call":  # the shared expert as its two calls, weights requested before each wait
        bx = w["x"].shape[0]
        ws_h = w["ws_sh"][: bx * I * 2].view(torch.bfloat16).view(bx, I)
        rec(8, side)  # one interval over both calls: an event between them would break their overlap
        mt.moe_shared_gate_up(w["x"], w["w_gate"], w["w_up_s"], ws_h, weights_static=True, stream=side)
        mt.moe_shared_down(ws_h, w["w_down"], w["d_slot"], accumulate=False, weights_static=True, stream=side)
        rec(9, side)
        rec(10, side)
        rec(11, side)
    else:
        shared_expert(side, w["d_slot"], False)
    rec(4, side)
    mt.moe_tail_latent_up_flags(w["latent"], w["lat_gamma"], w["w_up"], w["shared9"], w["out"], w["y"],
                                eps=1e-6, inputs_ready=True, weights_static=True, stream=side)
    rec(5, side)
    rec(6, side)
    rec(7, side)
    w["join"].record(side)
    ep(stream)
    tp(stream)
    stream.wait_event(w["join"])


CALLS = ["ep_finalize", "tp_finalize", "latent_up", "shared_expert"]

# The step's algorithmic bytes whatever its composition: every input read once
# (EP rows, expert-TP partials, latent partials, W_up, shared partials, the
# shared expert's weights and x, indices, weights, gains) and the three outputs
# written once; no intermediate (y, h, d) counted.
STEP_BYTES = (BYTES["ep_finalize"] + BYTES["tp_finalize"] + BYTES["latent_up"] + 3 * I * H * 2 + B * H * 2)


def step_calls(composition: str, side) -> dict:
    """The calls of one step as the composition makes them: for each, the
    (start, end) event pairs around it in an instrumented step, the bytes the
    call itself moves (its inputs read once, its outputs written once,
    intermediates it reads or writes included), its FLOPs and its launches."""
    fin = {"ep_finalize": dict(pairs=[(0, 1)], bytes=BYTES["ep_finalize"], launches=1),
           "tp_finalize": dict(pairs=[(2, 3)], bytes=BYTES["tp_finalize"], launches=1)}
    if side is not None and composition == "two_branch_fused":
        return dict(fin, **{
            "shared_gate_up": dict(pairs=[(8, 9)], bytes=2 * I * H * 2 + B * H * 2 + B * I * 2,
                                   flops=2 * B * 2 * I * H, launches=1),
            "latent_norm": dict(pairs=[(4, 5)], bytes=TP * B * L * 2 + L * 2 + B * L * 2, launches=1),
            "up_project_shared_down": dict(pairs=[(6, 7)],
                                           bytes=H * I * 2 + H * L * 2 + B * I * 2 + B * L * 2 + TP * B * H * 2
                                           + B * H * 2, flops=2 * B * H * (I + L), launches=1)})
    d_slot = side is not None and composition in ("two_branch", "two_branch_one_call")  # d: a shared slot
    return dict(fin, **{
        "latent_up": dict(pairs=[(4, 5), (6, 7)], bytes=BYTES["latent_up"] + (B * H * 2 if d_slot else 0),
                          flops=FLOPS["latent_up"], launches=2),
        "shared_expert": dict(pairs=[(8, 9), (10, 11)],
                              bytes=(3 * I * H * 2 + B * H * 2 + B * H * 2) if d_slot else BYTES["shared_expert"],
                              flops=FLOPS["shared_expert"], launches=2)})


def traffic_record(call: str):
    """ncu DRAM bytes (read + write) of one call of the step, summed over its
    launches, if the committed profile holds it and was taken on the current
    kernel sources (else None).  File lines: 'sources_sha256 <hash>' and
    'traffic <call> <bytes>'."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    if not os.path.exists(path):
        return None
    sha, rec = None, {}
    for line in open(path):
        parts = line.split()
        if len(parts) == 2 and parts[0] == "sources_sha256":
            sha = parts[1]
        elif len(parts) == 3 and parts[0] == "traffic":
            rec[parts[1]] = parts[2]
    if sha != kernel_sources_hash():
        return None
    try:
        return int(rec[call])
    except (KeyError, ValueError):
        return None


# The sources that define the shared-expert call's kernels and their launch
# (plans, tensor maps): a change to any of them invalidates its ncu traffic.
GEMM_SOURCES = ("common.cuh", "decode_gemm.cu", "kernels.h", "moe_tail_api.cu")


def code_only(text: str) -> str:
    """C/CUDA source without its comments, trailing blanks and empty lines:
    what a comment edit leaves unchanged (the sources hold no "//" or "/*"
    inside string literals)."""
    import re

    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_sources_hash() -> str:
    """SHA-256 of the code (comments aside) of the files that define the
    measured GEMM kernels and their launch."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_decode_tail_gb300", "csrc")
    for f in GEMM_SOURCES:
        h.update(code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- CPU oracle

def oracle_token_times(cpu, n_fin: int, n_lat: int, f_lat: float, n_sh: int, f_sh: float):
    """Seconds per token of each call of the step, timed on the oracle (plain
    C, one thread) over a bounded sample: n_fin tokens of each finalize call;
    n_lat tokens of the latent norm and of the up-projection over a fraction
    f_lat of the output features; n_sh tokens of the shared expert over a
    fraction f_sh of the intermediate features (the work per feature is the
    same, so the time scales to the full width)."""
    import oracle

    ep, tp, lat, sh = cpu["ep"], cpu["tp"], cpu["lat"], cpu["sh"]
    res, sample = {}, {}

    def timed(fn):
        t0 = time.perf_counter()
        out = fn()
        return time.perf_counter() - t0, out

    n = max(1, min(B, n_fin))
    t, _ = timed(lambda: oracle.ep_finalize(ep["rows"], ep["rows_per_slot"], ep["idx"][:, :n].contiguous(),
                                            ep["w"][:n].contiguous(), ep["gamma"], 1.0, 1e-6, True, n, TP,
                                            K_ROUTES, P))
    res["ep_finalize"], sample["ep_finalize"] = t / n, f"{n} tokens"
    t, _ = timed(lambda: oracle.tp_finalize(tp["partials"], tp["num_rows"], tp["idx"][:n].contiguous(),
                                            tp["w"][:n].contiguous(), tp["gamma"], 1.0, 1e-6, True, n, TP,
                                            K_ROUTES, P))
    res["tp_finalize"], sample["tp_finalize"] = t / n, f"{n} tokens"
    n = max(1, min(B, n_lat))
    hs = max(8, int(H * min(1.0, f_lat)) // 8 * 8)
    t_norm, y = timed(lambda: oracle.latent_norm(lat["latent"][:, :n].contiguous(), lat["gamma"], 1e-6, n, TP, L))
    t_up, _ = timed(lambda: oracle.latent_up(y, lat["w_up"][:hs].contiguous(),
                                             lat["shared"][:, :n, :hs].contiguous(), TP, n, L, hs))
    res["latent_up"] = (t_norm + t_up * H / hs) / n
    sample["latent_up"] = f"{n} tokens, {hs}/{H} output features"
    n = max(1, min(B, n_sh))
    is_ = max(8, int(I * min(1.0, f_sh)) // 8 * 8)
    t, _ = timed(lambda: oracle.shared_expert(sh["x"][:n], sh["w_gate"][:is_].contiguous(),
                                              sh["w_up"][:is_].contiguous(), sh["w_down"][:, :is_].contiguous(),
                                              n, H, is_, out_in=torch.zeros((n, H), dtype=torch.bfloat16)))
    res["shared_expert"] = t * I / is_ / n
    sample["shared_expert"] = f"{n} tokens, {is_}/{I} intermediate features"
    return res, sample


def oracle_parallel_times(cpu, workers: int, n_tok: int = B):
    """Seconds per token of each call with the oracle run token-parallel on
    `workers` host threads (the oracle is plain C called through ctypes, which
    releases the GIL): each call's n_tok tokens are split into one contiguous
    slice per thread, and the wall time of the whole call is divided by n_tok."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    ep, tp, lat, sh = cpu["ep"], cpu["tp"], cpu["lat"], cpu["sh"]
    n = max(1, min(B, n_tok))
    bounds = [(n * i // workers, n * (i + 1) // workers) for i in range(workers)]
    bounds = [(a, b) for a, b in bounds if b > a]

    def ep_slice(a, b):
        oracle.ep_finalize(ep["rows"], ep["rows_per_slot"], ep["idx"][:, a:b].contiguous(), ep["w"][a:b].contiguous(),
                           ep["gamma"], 1.0, 1e-6, True, b - a, TP, K_ROUTES, P)

    def tp_slice(a, b):
        oracle.tp_finalize(tp["partials"], tp["num_rows"], tp["idx"][a:b].contiguous(), tp["w"][a:b].contiguous(),
                           tp["gamma"], 1.0, 1e-6, True, b - a, TP, K_ROUTES, P)

    def lat_slice(a, b):
        y = oracle.latent_norm(lat["latent"][:, a:b].contiguous(), lat["gamma"], 1e-6, b - a, TP, L)
        oracle.latent_up(y, lat["w_up"], lat["shared"][:, a:b].contiguous(), TP, b - a, L, H)

    def sh_slice(a, b):
        oracle.shared_expert(sh["x"][a:b].contiguous(), sh["w_gate"], sh["w_up"], sh["w_down"], b - a, H, I,
                             out_in=torch.zeros((b - a, H), dtype=torch.bfloat16))

    res = {}
    with ThreadPoolExecutor(max_workers=len(bounds)) as pool:
        for name, fn in (("ep_finalize", ep_slice), ("tp_finalize", tp_slice), ("latent_up", lat_slice),
                         ("shared_expert", sh_slice)):
            t0 = time.perf_counter()
            list(pool.map(lambda ab: fn(*ab), bounds))
            res[name] = (time.perf_counter() - t0) / n
    return res, len(bounds)


def cpu_baseline(cpu):
    """The oracle on the host: token-parallel over all host threads for the
    step's 64 tokens of every call (the reported value), and on one thread over
    a bounded sample (64 tokens of each finalize, 16 of the latent tail, 32 of
    the shared expert, all at full width; about 10 s)."""
    per_tok, sample = oracle_token_times(cpu, 64, 16, 1.0, 32, 1.0)
    sec = sum(per_tok.values())
    cores = max(1, min(64, os.cpu_count() or 1))
    par_tok, used = oracle_parallel_times(cpu, cores)
    par_sec = sum(par_tok.values())
    return {"value": 1.0 / par_sec, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": (f"each call over the step's {B} tokens at full width, token-parallel on {used} host threads "
                       "(plain C oracle through ctypes; wall seconds per token summed over the four calls)"),
            "us_per_token": {k: round(v * 1e6, 1) for k, v in par_tok.items()},
            "single_thread": {"value": 1.0 / sec, "cores": 1,
                              "sample": "; ".join(f"{k}: {v}" for k, v in sample.items()),
                              "us_per_token": {k: round(v * 1e6, 1) for k, v in per_tok.items()}}}


# ----------------------------------------------------------------------------- arms

def reference_arm(args, world, rank):
    """The oracle as the reference implementation, timed on the host cores."""
    if rank != 0:
        return 0
    from moe_decode_tail_gb300 import synth

    cpu = dict(ep=synth.config(2), tp=synth.config(3, b=B), lat=synth.latent_up_inputs(synth.SEED_BASE + 4, b=B),
               sh=synth.config(5))
    total = args.steps + args.warmup
    budget = max(0.005, min(2.0, 150.0 / max(1, total)))  # seconds per step: the run ends in minutes
    # one token through each finalize (a few ms); the GEMM calls over the
    # fraction of their features that fits the rest of the step's budget
    frac = min(1.0, max(0.0, budget - 0.005) / 0.2)
    sample_args = (1, 1, max(8.0 / H, frac), 1, max(8.0 / I, frac))
    for _ in range(args.warmup):
        oracle_token_times(cpu, *sample_args)
    t0 = time.perf_counter()
    acc = {c: 0.0 for c in CALLS}
    sample = None
    for _ in range(args.steps):
        r, sample = oracle_token_times(cpu, *sample_args)
        for c in CALLS:
            acc[c] += r[c]
    elapsed = time.perf_counter() - t0
    sec_per_token = sum(acc.values()) / max(1, args.steps)
    value = 1.0 / sec_per_token
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed * 1e3 / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64",
        "data": "synthetic (seeded splitmix64 + Box-Muller; random-init weights)",
        "config": workload_config(),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "per step: " + "; ".join(f"{k}: {v}" for k, v in sample.items())},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config():
    return {
        "workload": "MoE decode tail step at b=64: EP finalize (tp=8 slots, P=4096, top-8 of 128 experts, 1% x8 "
                    "outlier rows, weight_before_norm) + expert-TP finalize (tp=8 K-partials, P=4096, top-8) + "
                    "latent tail (8 x [64,3584] partials -> RMSNorm -> W_up [7168,3584], + 8 x [64,7168] shared "
                    "partials) + fused shared expert (W_gate/W_up [6144,7168], W_down [7168,6144], accumulate)",
        "b": B, "tp": TP, "P": P, "top_k": K_ROUTES, "experts": E, "L": L, "H": H, "I": I,
        "l2": "no flush: a step reads ~390 MB (3x the 129 MB L2), so each input is cold when read",
    }


def cuda_arm(args, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    from moe_decode_tail_gb300 import build as cuda_build

    if rank == 0 or world == 1:
        cuda_build.build()
    barrier(dist, dev)
    import moe_decode_tail_gb300 as mt

    mt.lib()
    cpu, w = make_workload(dev)
    w["composition"] = args.composition
    # the routed finalize calls (latency-bound) on a high-priority stream, the
    # weight-streaming calls (shared expert, then latent tail) beside them
    stream = torch.cuda.Stream(dev, priority=-1)
    side = None if args.sequential else torch.cuda.Stream(dev, priority=0)
    K, W = args.steps, args.warmup
    G = max(1, min(args.graph_steps, K))

    with torch.cuda.stream(stream):
        for _ in range(3):  # eager warm-up: loads the kernels
            run_step(mt, w, stream, side=side)
    torch.cuda.synchronize()

    def capture(n, with_events):
        # Per-call events (external: recorded as event nodes of the graph, replayed
        # with it) in every tenth step only: an event between two calls keeps the
        # second from being scheduled while the first drains.
        evs = ([[torch.cuda.Event(enable_timing=True, external=True) for _ in range(EVENTS_PER_STEP)] if i % 10 == 0 else None
                for i in range(n)] if with_events else None)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                run_step(mt, w, stream, evs[i] if evs else None, side=side)
        return g, [e for e in evs if e is not None] if evs else None

    # The timed region replays graphs without events only: K // G replays of a
    # G-step graph and one graph of the K % G remaining steps.  A copy of the
    # G-step graph with per-call events replays after the timed region and
    # gives each call's duration.
    clean_g = capture(G, False)[0]
    rest = K % G
    rest_g = capture(rest, False)[0] if rest else None
    inst_g, inst_ev = capture(G, True)
    torch.cuda.synchronize()
    # warm-up: at least W steps from the timed graphs (replay() launches on the current stream)
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-W // G))):
            clean_g.replay()
        if rest_g is not None:
            rest_g.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    barrier(dist, dev)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(K // G):
            clean_g.replay()
        if rest_g is not None:
            rest_g.replay()
        stop.record(stream)
    torch.cuda.synchronize()
    barrier(dist, dev)
    clocks = sampler.stop() if rank == 0 else None
    seconds = start.elapsed_time(stop) / 1e3
    max_s, units = aggregate(seconds, float(B * K), dist, dev)
    # the instrumented copy, outside the timed region
    with torch.cuda.stream(stream):
        inst_g.replay()
    torch.cuda.synchronize()

    # per-call durations over the instrumented steps of that replay
    table = step_calls(args.composition, side)
    per_call = {c: [] for c in table}
    for evs in inst_ev:
        for c, t in table.items():
            per_call[c].append(sum(evs[i].elapsed_time(evs[j]) for i, j in t["pairs"]) * 1e3)  # us
    calls = {}
    hbm, bf16_tf, peak_kind = peaks()
    for c, t in table.items():
        us = statistics.mean(per_call[c])
        gbs = t["bytes"] / (us * 1e-6) / 1e9
        calls[c] = {"us": round(us, 3), "tokens_per_s": B / (us * 1e-6), "algorithmic_bytes": t["bytes"],
                    "achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
                    "hbm_frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4), "launches": t["launches"]}
        if "flops" in t:
            calls[c]["tflops"] = round(t["flops"] / (us * 1e-6) / 1e12, 2)

    # end to end through the public API from pinned host buffers
    e2e = e2e_leg(mt, w, stream, min(args.e2e_steps, K), dist, dev, side)

    if rank != 0:
        return 0
    dom = max(table, key=lambda c: calls[c]["us"])
    roof = {
        "bound": "hbm", "kernel": f"moe_{dom}" if dom.startswith("shared") else f"moe_tail_{dom}",
        "launches": table[dom]["launches"],
        "achieved": calls[dom]["achieved_gbs"], "peak": hbm, "unit": "GB/s",
        "frac": round(calls[dom]["achieved_gbs"] / hbm, 4), "traffic": traffic_record(dom),
        "algorithmic_bytes_per_call": table[dom]["bytes"],
        "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
        "note": "per-call CUDA events on the launch stream, recorded as graph nodes in every tenth step of a "
                "replay made after the timed region (those steps lose the overlap between calls, so the per-call "
                "figures are conservative; the timed replays carry no events)",
    }
    ms = max_s * 1e3 / K
    line = {
        "metric": METRIC, "value": units / max_s, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms, "us_per_layer": ms * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded splitmix64 + Box-Muller; random-init weights)",
        "config": dict(workload_config(), composition=(
            "sequential: EP, TP, latent tail, then the shared expert accumulating into out" if side is None else
            "two branches: on a side stream the shared expert (gate/up, then down, both with static weights) writes "
            "d into an extra shared-partial slot, then the latent tail follows (its norm, then its up-projection), "
            "adding all slots; EP and TP on a high-priority stream beside them"
            if args.composition == "two_branch" else
            "two branches as two_branch, with the shared expert as one moe_shared_expert call"
            if args.composition == "two_branch_one_call" else
            "two branches: on a side stream the shared expert's gate/up (static weights, inputs ready), the "
            "latent norm (inputs ready), then one kernel whose cluster ranks stream the down projection or the "
            "latent up-projection and which adds bf16(d) after the shared partials "
            "(moe_tail_up_project_shared_down, static weights); EP and TP on a high-priority stream beside them"
            if args.composition == "two_branch_fused" else
            "two branches: the shared expert's gate/up on a side stream; EP, TP and the latent tail on a "
            "high-priority stream beside it; then the down projection adds d into the latent tail's output")),
        "roofline": roof, "calls": calls, "e2e": e2e,
        "step_roofline": {
            "algorithmic_bytes": STEP_BYTES,
            "achieved_gbs": round(STEP_BYTES / (max_s / K) / 1e9, 1),
            "peak": hbm, "unit": "GB/s",
            "frac": round(STEP_BYTES / (max_s / K) / 1e9 / hbm, 4),
            "frac_nominal": round(STEP_BYTES / (max_s / K) / 1e9 / NOMINAL_HBM_GBS, 4),
            "note": "the step's algorithmic bytes (every input read once, the outputs written once, no "
                    "intermediate) over the step time: the whole step is an HBM stream",
        },
        "gpu_launches": sum(t["launches"] for t in table.values()) * K, "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cpu)
    if not args.no_configs:
        line["configs_isolated"] = isolated_configs(mt, cpu, w, dev, stream)
        alone = line["configs_isolated"]["results"].get("5_gate_up_b64")
        if alone and dom == "shared_gate_up":  # the same kernel timed alone, for comparison
            roof["alone"] = {"configs_isolated": "5_gate_up_b64", "us": alone["us"], "frac": alone["hbm_frac"]}
        line["step_by_batch"] = dict(step_by_batch(mt, w, dev, stream, side),
                                     b64={"us_per_step": round(ms * 1e3, 2), "tokens_per_s": round(units / max_s, 1)})
    print(json.dumps(line), flush=True)
    return 0


def config_bytes(name: str, d: dict) -> int:
    """Algorithmic bytes (read + write) of one call at a workload's sizes: every
    route row, weight and partial read once, the output written once."""
    if name == "ep":
        b, tp, K, P = d["b"], d["tp"], d["K"], d["P"]
        return b * K * P * 2 + tp * b * K * 4 + b * K * 4 + P * 2 + b * P * 2
    if name == "tp":
        b, tp, K, P = d["b"], d["tp"], d["K"], d["P"]
        return tp * b * K * P * 2 + 2 * b * K * 4 + P * 2 + b * P * 2
    if name == "latent":
        b, tp, tp_s, L_, H_ = d["b"], d["tp"], d["tp_s"], d["L"], d["H"]
        return H_ * L_ * 2 + tp * b * L_ * 2 + tp_s * b * H_ * 2 + L_ * 2 + b * H_ * 2
    b, H_, I_ = d["b"], d["H"], d["I"]  # shared expert added into out: h written + read, out read + written
    return 3 * H_ * I_ * 2 + b * H_ * 2 + 2 * b * I_ * 2 + 2 * b * H_ * 2


def floor_lib():
    """The latency-floor kernels (include/moe_tail_floor.h), built on first use."""
    import ctypes

    from moe_decode_tail_gb300 import build as cuda_build

    L_ = ctypes.CDLL(cuda_build.build(floor=True))
    P_, i32 = ctypes.c_void_p, ctypes.c_int
    L_.moe_tail_floor_empty.argtypes = [i32, i32, i32, i32, P_]
    L_.moe_tail_floor_read.argtypes = [P_, ctypes.c_size_t, i32, i32, i32, i32, P_, P_]
    L_.moe_tail_floor_gather.argtypes = [P_, i32, P_, ctypes.c_int64, i32, i32, i32, i32, P_, P_]
    return L_


def ep_floor(d, dev, timed, copies_for, ep_us) -> dict:
    """Latency floors of the EP finalize call at config 2, on its own grid (two
    column bands of 256 threads per token, clusters of two, b = 64 tokens):
    an empty kernel (launch and dependency wait), one trip reading the call's
    algorithmic bytes, and the two dependent trips of its access pattern (the
    token's route indices, then its 8 local rows' bands).  Each is timed as
    the call is (a graph of back-to-back launches, inputs rotated past L2)."""
    import ctypes

    fl = floor_lib()
    gx, gy, thr, cl = 2, d["b"], 256, 2
    st = torch.cuda.current_stream(dev)
    sptr = lambda: ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    sink = torch.zeros(gx * gy, dtype=torch.int32, device=dev)
    nbytes = config_bytes("ep", d)
    nbytes -= nbytes % 16
    n = copies_for(nbytes)
    bufs = [torch.empty(nbytes, dtype=torch.uint8, device=dev).random_(0, 255) for _ in range(n)]
    # the gather: each token's 8 local routes as (slot, row) -> a row of the [tp * rows_per_slot, P] table
    tp, K, R = d["tp"], d["K"], d["rows_per_slot"]
    idx = d["idx"].numpy()
    flat = []
    for t in range(d["b"]):
        flat.append([s * R + int(j) for s in range(tp) for j in idx[s, t] if 0 <= j < R][:K])
    gidx = torch.tensor(flat, dtype=torch.int32, device=dev)
    rows = [d["rows"].to(dev)] + [None] * (copies_for(d["rows"].numel() * 2) - 1)
    for i in range(1, len(rows)):
        rows[i] = rows[0].clone()

    def call(rc):
        assert rc == 0, rc

    out = {"grid": f"{gx} x {gy} CTAs of {thr} threads, clusters of {cl}"}
    out["empty_us"] = round(timed(lambda i: call(fl.moe_tail_floor_empty(gx, gy, thr, cl, sptr())), 1), 3)
    out["read_us"] = round(timed(lambda i: call(fl.moe_tail_floor_read(
        ctypes.c_void_p(bufs[i].data_ptr()), nbytes, gx, gy, thr, cl, ctypes.c_void_p(sink.data_ptr()), sptr())),
        n), 3)
    out["gather_us"] = round(timed(lambda i: call(fl.moe_tail_floor_gather(
        ctypes.c_void_p(gidx.data_ptr()), K, ctypes.c_void_p(rows[i].data_ptr()), tp * R, gx, gy, thr, cl,
        ctypes.c_void_p(sink.data_ptr()), sptr())), len(rows)), 3)
    out["ep_over_read"] = round(ep_us / out["read_us"], 3)
    out["ep_over_gather"] = round(ep_us / out["gather_us"], 3)
    del bufs, rows, st
    return out


def tp_floor(d, dev, timed, parts, tp_us) -> dict:
    """Memory floor of the expert-TP call at config 3 on its own grid (two
    column bands of 256 threads per token, clusters of two, b = 128 tokens):
    a kernel that only gathers the call's rows -- each token's K routes in all
    tp slots, 16 rows in flight per thread, the depth of the call's 2-stage
    ring -- timed as the call is."""
    import ctypes

    fl = floor_lib()
    gx, gy, thr, cl = 2, d["b"], 256, 2
    sptr = lambda: ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    sink = torch.zeros(gx * gy, dtype=torch.int32, device=dev)
    tp, K, R = d["tp"], d["K"], d["num_rows"]
    idx = d["idx"].numpy()
    gidx = torch.tensor([[s * R + int(idx[t, k]) for k in range(K) for s in range(tp)] for t in range(d["b"])],
                        dtype=torch.int32, device=dev)

    def call(i):
        rc = fl.moe_tail_floor_gather(ctypes.c_void_p(gidx.data_ptr()), K * tp, ctypes.c_void_p(parts[i].data_ptr()),
                                      tp * R, gx, gy, thr, cl, ctypes.c_void_p(sink.data_ptr()), sptr())
        assert rc == 0, rc

    out = {"grid": f"{gx} x {gy} CTAs of {thr} threads, clusters of {cl}"}
    out["gather_us"] = round(timed(call, len(parts)), 3)
    out["tp_over_gather"] = round(tp_us / out["gather_us"], 3)
    return out


def isolated_configs(mt, cpu, w, dev, stream) -> dict:
    """Each workload timed alone: one call per graph node, CUDA events around
    replays of a graph of max(20, copies) calls that cycles over copies of the
    call's large inputs (together more than twice the L2; at most 256 copies,
    so the smallest calls stay L2-resident), median of 7 replays.  Also each
    call at b = 1 and b = 8 (the small-batch decode regime), the latent tail
    also with both promises and in its opt-in one-kernel form."""
    from moe_decode_tail_gb300 import synth

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    hbm, _, kind = peaks()

    def timed(fn, copies, reps=20, replays=7):
        reps = max(reps, copies)  # every replay cycles through all the copies
        with torch.cuda.stream(stream):
            for i in range(copies):
                fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                fn(r % copies)
        ts = []
        with torch.cuda.stream(stream):
            g.replay()
            for _ in range(replays):
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                e.record(stream)
                e.synchronize()
                ts.append(a.elapsed_time(e) * 1e3 / reps)
        return statistics.median(ts)

    def copies_for(nbytes):  # enough copies to exceed twice the L2, at most 256 (tiny calls stay L2-resident)
        return min(256, max(1, -(-2 * l2 // max(1, nbytes)) + 1))

    res = {}

    def report(key, us, nbytes, copies, target):
        gbs = nbytes / (us * 1e-6) / 1e9
        res[key] = {"us": round(us, 3), "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1),
                    "hbm_frac": round(gbs / hbm, 4), "hbm_frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                    "input_copies": copies, "target": target}

    def ep_like(key, d, target, n=None, ready_key=None):
        nb = config_bytes("ep", d)
        n = n or copies_for(nb)
        rows = [d["rows"].to(dev)] + [None] * (n - 1)
        for i in range(1, n):
            rows[i] = rows[0].clone()
        idx, wt, gam = d["idx"].to(dev), d["w"].to(dev), d["gamma"].to(dev)
        out = torch.empty((d["b"], d["P"]), dtype=torch.bfloat16, device=dev)
        us = timed(lambda i: mt.moe_tail_ep_finalize(rows[i], idx, wt, gam, out, gain_center=d["gain_center"],
                                                     eps=d["eps"], weight_before_norm=d["weight_before_norm"],
                                                     stream=stream), n)
        report(key, us, nb, n, target)
        if ready_key:  # the same call with the inputs-ready promise (moe_tail_ep_finalize_flags)
            us = timed(lambda i: mt.moe_tail_ep_finalize_flags(
                rows[i], idx, wt, gam, out, gain_center=d["gain_center"], eps=d["eps"],
                weight_before_norm=d["weight_before_norm"], inputs_ready=True, stream=stream), n)
            report(ready_key, us, nb, n, target)

    ep_like("1_ep_tiny_b4_P512", synth.config(1), "parity; latency-bound (report us; inputs L2-resident)", n=1)
    ep_like("2_ep_b64_P4096", cpu["ep"], ">= 0.70 of HBM (hard at 4.7 MB)", ready_key="2_ep_b64_P4096_ready")
    res["2_ep_b64_P4096"]["floor"] = ep_floor(cpu["ep"], dev, timed, copies_for, res["2_ep_b64_P4096"]["us"])

    d = synth.config(3)
    nb = config_bytes("tp", d)
    n = copies_for(nb)
    parts = [d["partials"].to(dev)]
    parts += [parts[0].clone() for _ in range(n - 1)]
    idx, wt, gam = d["idx"].to(dev), d["w"].to(dev), d["gamma"].to(dev)
    out = torch.empty((d["b"], d["P"]), dtype=torch.bfloat16, device=dev)
    us = timed(lambda i: mt.moe_tail_tp_finalize(parts[i], idx, wt, gam, out, gain_center=d["gain_center"],
                                                 eps=d["eps"], weight_before_norm=d["weight_before_norm"],
                                                 stream=stream), n)
    report("3_tp_b128_P4096", us, nb, n, ">= 0.70 of HBM")
    res["3_tp_b128_P4096"]["floor"] = tp_floor(d, dev, timed, parts, us)
    # ... with the inputs-ready promise (moe_tail_tp_finalize_flags): each call reads its
    # partials while the previous call drains
    us = timed(lambda i: mt.moe_tail_tp_finalize_flags(parts[i], idx, wt, gam, out, gain_center=d["gain_center"],
                                                       eps=d["eps"], weight_before_norm=d["weight_before_norm"],
                                                       inputs_ready=True, stream=stream), n)
    report("3_tp_b128_P4096_ready", us, nb, n, ">= 0.70 of HBM")
    del parts

    d = synth.config(4)
    nb = config_bytes("latent", d)
    n = copies_for(nb)
    wu = [d["w_up"].to(dev)]
    wu += [wu[0].clone() for _ in range(n - 1)]
    lat, gam, sh = d["latent"].to(dev), d["gamma"].to(dev), d["shared"].to(dev)
    out = torch.empty((d["b"], d["H"]), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mt.moe_tail_workspace_bytes(0, d["b"], d["L"]), dtype=torch.uint8, device=dev)
    us = timed(lambda i: mt.moe_tail_latent_up(lat, gam, wu[i], sh, out, ws, eps=d["eps"], stream=stream), n)
    report("4_latent_up_b16", us, nb, n, ">= 0.60 of the weight-stream roofline")
    # the same tail as its two calls with the promises a serving loop can make
    # here (inputs ready, weights static): the norm of call i+1 reads its inputs
    # while the up-projection of call i streams
    y = ws[: d["b"] * d["L"] * 2].view(torch.bfloat16).view(d["b"], d["L"])

    def split_call(i):
        mt.moe_tail_latent_norm(lat, gam, y, eps=d["eps"], inputs_ready=True, stream=stream)
        mt.moe_tail_up_project(y, wu[i], sh, out, weights_static=True, stream=stream)

    us = timed(split_call, n)
    report("4_latent_up_b16_two_calls", us, nb, n, ">= 0.60 of the weight-stream roofline")
    # ... and as one call with the same promises (moe_tail_latent_up_flags)
    us = timed(lambda i: mt.moe_tail_latent_up_flags(lat, gam, wu[i], sh, out, y, eps=d["eps"], inputs_ready=True,
                                                     weights_static=True, stream=stream), n)
    report("4_latent_up_b16_flags", us, nb, n, ">= 0.60 of the weight-stream roofline")
    del wu

    d = dict(b=B, H=H, I=I)
    nb = config_bytes("shared", d)
    n = 2
    ws_ = [(w["w_gate"], w["w_up_s"], w["w_down"])]
    ws_.append(tuple(t.clone() for t in ws_[0]))
    out = torch.zeros((B, H), dtype=torch.bfloat16, device=dev)
    us = timed(lambda i: mt.moe_shared_expert(w["x"], *ws_[i], out, w["ws_sh"], accumulate=True, stream=stream), n)
    report("5_shared_expert_b64", us, nb, n, ">= 0.60 of the weight-stream roofline")
    # ... as its two calls with static weights: each gate/up requests its first
    # weight tiles while the previous call's down projection drains
    h_ = w["ws_sh"][: B * I * 2].view(torch.bfloat16).view(B, I)

    def shared_static(i):
        mt.moe_shared_gate_up(w["x"], ws_[i][0], ws_[i][1], h_, weights_static=True, stream=stream)
        mt.moe_shared_down(h_, ws_[i][2], out, accumulate=True, weights_static=True, stream=stream)

    us = timed(shared_static, n)
    report("5_shared_expert_b64_static", us, nb, n, ">= 0.60 of the weight-stream roofline")
    # its gate/up alone: the decode step's longest call without the step's
    # concurrent finalize calls and down + up stream
    nb_gu = 2 * I * H * 2 + B * H * 2 + B * I * 2
    us = timed(lambda i: mt.moe_shared_gate_up(w["x"], ws_[i][0], ws_[i][1], h_, stream=stream), n)
    report("5_gate_up_b64", us, nb_gu, n, "report (the decode step's longest call, alone)")

    # the shared expert's down projection alone (d written, not accumulated): the
    # split-K GEMM against the page's persistent form on 56, 28 and 14 CTAs (each
    # walking 1, 2 or 4 output tiles with two alternating TMEM accumulators)
    wds = [ws_[0][2], ws_[1][2]] + [ws_[0][2].clone() for _ in range(2)]
    nb_down = H * I * 2 + B * I * 2 + B * H * 2
    us = timed(lambda i: mt.moe_shared_down(h_, wds[i], out, accumulate=False, stream=stream), len(wds))
    report("5_down_b64", us, nb_down, len(wds), "report (the persistent form's comparison)")
    for ctas in (56, 28, 14):
        us = timed(lambda i: mt.moe_shared_down_persistent(h_, wds[i], out, accumulate=False, ctas=ctas,
                                                           stream=stream), len(wds))
        report(f"5_down_persistent_b64_{ctas}ctas", us, nb_down, len(wds), "report (the page's SharedDown form)")
    del wds

    # the composed layer of configs 4 and 5 at b = 64, as the default step's side
    # stream runs it: gate/up, the latent norm, then the down projection and the
    # up-projection in one kernel (algorithmic bytes: no intermediate counted)
    wl = [w["w_up"], w["w_up"].clone()]

    def layer(i):
        mt.moe_shared_gate_up(w["x"], ws_[i][0], ws_[i][1], h_, weights_static=True, inputs_ready=True,
                              stream=stream)
        mt.moe_tail_latent_norm(w["latent"], w["lat_gamma"], w["y"], eps=1e-6, inputs_ready=True, stream=stream)
        mt.moe_tail_up_project_shared_down(w["y"], wl[i], w["shared"], h_, ws_[i][2], w["out"], weights_static=True,
                                           stream=stream)

    nb_layer = 3 * H * I * 2 + B * H * 2 + BYTES["latent_up"]
    us = timed(layer, 2)
    report("4+5_latent_tail_and_shared_expert_b64", us, nb_layer, 2, "composed layer (report)")
    del ws_, wl
    torch.cuda.synchronize()

    # the small-batch decode regime: each call at b = 1 and b = 8 (decode shapes of
    # configs 2, 3, 4 and 5; weights rotate over copies, activations are tiny)
    small = {}
    for bs in (1, 8):
        row = {}
        d = synth.config(2, b=bs)
        nb = config_bytes("ep", d)
        n = copies_for(nb)
        rows = [d["rows"].to(dev)]
        rows += [rows[0].clone() for _ in range(n - 1)]
        idx, wt, gam = d["idx"].to(dev), d["w"].to(dev), d["gamma"].to(dev)
        out = torch.empty((bs, d["P"]), dtype=torch.bfloat16, device=dev)
        row["ep_finalize"] = timed(lambda i: mt.moe_tail_ep_finalize(rows[i], idx, wt, gam, out, stream=stream), n)
        del rows
        d = synth.config(3, b=bs)
        nb = config_bytes("tp", d)
        n = copies_for(nb)
        parts = [d["partials"].to(dev)]
        parts += [parts[0].clone() for _ in range(n - 1)]
        idx, wt, gam = d["idx"].to(dev), d["w"].to(dev), d["gamma"].to(dev)
        out = torch.empty((bs, d["P"]), dtype=torch.bfloat16, device=dev)
        row["tp_finalize"] = timed(lambda i: mt.moe_tail_tp_finalize(parts[i], idx, wt, gam, out, stream=stream), n)
        del parts
        lat = w["latent"][:, :bs].contiguous()
        sh = w["shared"][:, :bs].contiguous()
        wu = [w["w_up"], w["w_up"].clone(), w["w_up"].clone(), w["w_up"].clone(), w["w_up"].clone(),
              w["w_up"].clone()]
        out = torch.empty((bs, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(mt.moe_tail_workspace_bytes(0, bs, L), dtype=torch.uint8, device=dev)
        row["latent_up"] = timed(lambda i: mt.moe_tail_latent_up(lat, w["lat_gamma"], wu[i], sh, out, ws,
                                                                 stream=stream), len(wu))
        # the same through moe_tail_latent_up_flags with both promises, and both
        # ways in the opt-in one-kernel form
        yb = torch.empty((bs, L), dtype=torch.bfloat16, device=dev)

        def flags_call(i, promises):
            mt.moe_tail_latent_up_flags(lat, w["lat_gamma"], wu[i], sh, out, yb, inputs_ready=promises,
                                        weights_static=promises, stream=stream)

        row["latent_up_promises"] = timed(lambda i: flags_call(i, True), len(wu))
        with mt.kernel_form(mt.FORM_LATENT, mt.FORM_LATENT_ONE_KERNEL):
            row["latent_up_one_kernel"] = timed(lambda i: flags_call(i, False), len(wu))
            row["latent_up_promises_one_kernel"] = timed(lambda i: flags_call(i, True), len(wu))
        del wu
        x = w["x"][:bs].contiguous()
        sw = [(w["w_gate"], w["w_up_s"], w["w_down"])]
        sw.append(tuple(t.clone() for t in sw[0]))
        wss = torch.empty(mt.moe_tail_workspace_bytes(1, bs, I), dtype=torch.uint8, device=dev)
        out = torch.zeros((bs, H), dtype=torch.bfloat16, device=dev)
        row["shared_expert"] = timed(lambda i: mt.moe_shared_expert(x, *sw[i], out, wss, accumulate=True,
                                                                    stream=stream), 2)
        del sw
        small[f"b{bs}"] = {k: round(v, 3) for k, v in row.items()}
    torch.cuda.synchronize()
    return {"peak_gbs": hbm, "peak_source": f"{kind} hbm_gbs (MEASURED_PEAKS.json)", "l2_bytes": l2,
            "method": ("each call alone: a graph of max(20, copies) calls cycling over copies of the call's large "
                       "inputs (together > 2x L2, at most 256 copies), median of 7 replays"),
            "results": res, "small_batch_us": small}


def step_by_batch(mt, w, dev, stream, side, sizes=(1, 8, 32, 128)) -> dict:
    """The same composed step at other batch sizes (fresh seeded activations,
    the b = 64 workload's resident weights): graphs of 20 steps, median of 7
    replays, per-step time and tokens/s."""
    res = {}
    for b in sizes:
        _, wb = make_workload(dev, b, weights=w)
        wb["composition"] = w.get("composition", "two_branch_fused")
        with torch.cuda.stream(stream):
            for _ in range(3):
                run_step(mt, wb, stream, side=side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(20):
                run_step(mt, wb, stream, side=side)
        ts = []
        with torch.cuda.stream(stream):
            g.replay()
            for _ in range(7):
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                e.record(stream)
                e.synchronize()
                ts.append(a.elapsed_time(e) * 1e3 / 20)
        us = statistics.median(ts)
        res[f"b{b}"] = {"us_per_step": round(us, 2), "tokens_per_s": round(b / (us * 1e-6), 1)}
        del wb, g
    torch.cuda.synchronize()
    return res


def packed_layout(named):
    """Byte offsets of tensors packed one after another in one buffer, each
    256-byte aligned (the calls want 16), and the buffer's size: named is a
    list of (name, tensor)."""
    offs, off = {}, 0
    for k, t in named:
        offs[k] = off
        off = (off + t.numel() * t.element_size() + 255) // 256 * 256
    return offs, off


def e2e_leg(mt, w, stream, steps, dist, dev, side=None):
    """The same step through the public API with host buffers: every step
    copies its activations from pinned host memory and reads its outputs back
    (weights stay resident, as in serving).  A step's activations sit in one
    pinned host buffer and, on the device, in one buffer whose tensors the
    calls take as views (256-byte aligned), so a step moves them with one
    host-to-device copy; its three outputs come back the same way, in one copy.
    Two sets of device buffers alternate, so step i+1's host-to-device copy
    (on its own stream) runs while step i computes, and step i's outputs are
    read back on a third stream; every step still moves all of its inputs and
    outputs."""
    inputs = ["ep_rows", "ep_idx", "ep_w", "tp_part", "tp_idx", "tp_w", "latent", "x"]
    outputs = ["out_ep", "out_tp", "out"]

    def view(buf, offs, k, like):
        n = like.numel() * like.element_size()
        return buf[offs[k]: offs[k] + n].view(like.dtype).view(like.shape)

    # inputs, then the latent tail's shared-partial slots with the shared expert's
    # slot last: the copy covers every input and stops before that slot
    in_offs, in_total = packed_layout([(k, w[k]) for k in inputs] + [("shared9", w["shared9"])])
    h2d = in_offs["shared9"] + w["shared"].numel() * w["shared"].element_size()
    host_in = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    for k in inputs:
        view(host_in, in_offs, k, w[k]).copy_(w[k].cpu())
    view(host_in, in_offs, "shared9", w["shared"]).copy_(w["shared"].cpu())
    out_offs, out_total = packed_layout([(k, w[k]) for k in outputs])
    host_out = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d2h = out_total
    sets = []
    for _ in range(2):
        s = dict(w)  # weights, workspaces and events shared: the steps run in stream order
        s["packed_in"] = torch.empty(in_total, dtype=torch.uint8, device=dev)
        s["packed_out"] = torch.empty(out_total, dtype=torch.uint8, device=dev)
        for k in inputs:
            s[k] = view(s["packed_in"], in_offs, k, w[k])
        s["shared9"] = view(s["packed_in"], in_offs, "shared9", w["shared9"])
        s["shared"], s["d_slot"] = s["shared9"][:TP], s["shared9"][TP]
        for k in outputs:
            s[k] = view(s["packed_out"], out_offs, k, w[k])
        sets.append(s)
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    computed, read_back = [ev(), ev()], [ev(), ev()]
    issued = [0]

    def one():
        i = issued[0]
        s, buf = sets[i % 2], i % 2
        ready = ev()
        if i >= 2:
            h2d_stream.wait_event(computed[buf])  # step i-2 is done with these inputs
        with torch.cuda.stream(h2d_stream):
            s["packed_in"][:h2d].copy_(host_in, non_blocking=True)
            ready.record(h2d_stream)
        stream.wait_event(ready)
        if i >= 2:
            stream.wait_event(read_back[buf])  # step i-2's outputs have been read back
        run_step(mt, s, stream, side=side)
        computed[buf].record(stream)
        d2h_stream.wait_event(computed[buf])
        with torch.cuda.stream(d2h_stream):
            host_out[buf].copy_(s["packed_out"], non_blocking=True)
            read_back[buf].record(d2h_stream)
        issued[0] += 1

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        barrier(dist, dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d_stream.wait_event(a)
        for _ in range(steps):
            one()
        for e in read_back:
            stream.wait_event(e)
        b.record(stream)
        torch.cuda.synchronize()
    s, units = aggregate(a.elapsed_time(b) / 1e3, float(B * steps), dist, dev)
    link = link_rates(sets[0]["packed_in"][:h2d], host_in, sets[0]["packed_out"], host_out[0], h2d_stream)
    step_s = s / steps
    return {"value": units / s, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": step_s * 1e3,
            "h2d_gbs": round(h2d / step_s / 1e9, 1),
            "link_peak_gbs": link,
            "h2d_frac_of_link": round(h2d / step_s / 1e9 / link["h2d"], 4),
            "pipelining": "double-buffered activations: step i+1's host-to-device copy overlaps step i's compute; "
                          "one copy each way per step (activations and outputs packed in one buffer)"}


def link_rates(dev_in, host_in, dev_out, host_out, stream, reps=10) -> dict:
    """GB/s of plain pinned copies of the e2e step's own buffers, alone on one
    stream (host to device: the step's packed inputs; device to host: its packed
    outputs): the link rate the e2e figure is bounded by."""
    res = {}
    for name, dst, src in (("h2d", dev_in, host_in), ("d2h", host_out, dev_out)):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                dst.copy_(src, non_blocking=True)
            b.record(stream)
        b.synchronize()
        res[name] = round(reps * src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    return res


def only_config(args) -> int:
    """One workload's call, eagerly, --calls times on cuda:0 (for ncu): configs
    1-2 EP finalize, 3 expert-TP finalize, 4 the latent tail (moe_tail_latent_up
    and then moe_tail_latent_up_flags with both promises), 5 the shared expert
    added into out, 6 the default step's side-stream calls at b = 64, 7 config 5's
    down projection, K-split and persistent."""
    import moe_decode_tail_gb300 as mt
    from moe_decode_tail_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = args.only_config
    d = synth.config(n) if n <= 5 else None
    g = lambda t: t.to(dev)
    if n in (1, 2):
        rows, idx, wt, gam = g(d["rows"]), g(d["idx"]), g(d["w"]), g(d["gamma"])
        out = torch.empty((d["b"], d["P"]), dtype=torch.bfloat16, device=dev)
        calls = [lambda: mt.moe_tail_ep_finalize(rows, idx, wt, gam, out, gain_center=d["gain_center"], eps=d["eps"],
                                                 weight_before_norm=d["weight_before_norm"])]
    elif n == 3:
        parts, idx, wt, gam = g(d["partials"]), g(d["idx"]), g(d["w"]), g(d["gamma"])
        out = torch.empty((d["b"], d["P"]), dtype=torch.bfloat16, device=dev)
        calls = [lambda: mt.moe_tail_tp_finalize(parts, idx, wt, gam, out, gain_center=d["gain_center"], eps=d["eps"],
                                                 weight_before_norm=d["weight_before_norm"])]
    elif n == 4:
        lat, gam, wu, sh = g(d["latent"]), g(d["gamma"]), g(d["w_up"]), g(d["shared"])
        out = torch.empty((d["b"], d["H"]), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(mt.moe_tail_workspace_bytes(0, d["b"], d["L"]), dtype=torch.uint8, device=dev)
        y = ws[: d["b"] * d["L"] * 2].view(torch.bfloat16).view(d["b"], d["L"])
        calls = [lambda: mt.moe_tail_latent_up(lat, gam, wu, sh, out, ws, eps=d["eps"]),
                 lambda: mt.moe_tail_latent_up_flags(lat, gam, wu, sh, out, y, eps=d["eps"], inputs_ready=True,
                                                     weights_static=True)]
    elif n == 5:
        x, wg, wu, wd = g(d["x"]), g(d["w_gate"]), g(d["w_up"]), g(d["w_down"])
        out = torch.zeros((d["b"], d["H"]), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(mt.moe_tail_workspace_bytes(1, d["b"], d["I"]), dtype=torch.uint8, device=dev)
        calls = [lambda: mt.moe_shared_expert(x, wg, wu, wd, out, ws, accumulate=True)]
    elif n == 7:  # config 5's down projection: the K-split GEMM, then the persistent form on 56 CTAs
        s = synth.shared_expert_inputs(0x5EED0007, b=B, H=H, I=I)
        hh, wd = g(s["x"][:, :I].contiguous()), g(s["w_down"])
        out = torch.zeros((B, H), dtype=torch.bfloat16, device=dev)
        calls = [lambda: mt.moe_shared_down(hh, wd, out, accumulate=False),
                 lambda: mt.moe_shared_down_persistent(hh, wd, out, accumulate=False, ctas=56)]
    else:  # the default step's side stream at b = 64
        _, w = make_workload(dev)
        h = torch.empty((B, I), dtype=torch.bfloat16, device=dev)

        def side_calls():
            mt.moe_shared_gate_up(w["x"], w["w_gate"], w["w_up_s"], h, weights_static=True, inputs_ready=True)
            mt.moe_tail_latent_norm(w["latent"], w["lat_gamma"], w["y"], eps=1e-6, inputs_ready=True)
            mt.moe_tail_up_project_shared_down(w["y"], w["w_up"], w["shared"], h, w["w_down"], w["out"],
                                               weights_static=True)
        calls = [side_calls]
    for call in calls:
        for _ in range(args.calls):
            call()
    torch.cuda.synchronize()
    print(json.dumps({"only_config": n, "calls_each": args.calls, "forms": len(calls),
                      "device_error": mt.moe_tail_take_device_error()}), flush=True)
    return 0


def trace_run(args) -> int:
    """Per-CTA timeline from the trace build (libmoetail_trace.so, loaded
    through MOE_TAIL_LIBRARY before the first library call).  "step": ten
    decode steps as one graph replay, as the timed region runs them, and the
    launches of two steps in its middle; "latent": the latent tail's opt-in
    one-kernel form (pinned with moe_tail_set_kernel_form) at b = 1, 4, 16, each call alone,
    without and with both promises."""
    from moe_decode_tail_gb300 import build as cuda_build

    os.environ["MOE_TAIL_LIBRARY"] = cuda_build.build(trace=True)
    import moe_decode_tail_gb300 as mt
    from moe_decode_tail_gb300.trace import Tracer, describe, launches

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.trace == "latent":
        g = torch.Generator(device=dev).manual_seed(7)
        wc = [(0.02 * torch.randn(H, L, device=dev, generator=g)).to(torch.bfloat16) for _ in range(6)]
        gamma = (1 + 0.05 * torch.randn(L, device=dev, generator=g)).to(torch.bfloat16)
        tracer = Tracer(mt)
        mt.moe_tail_set_kernel_form(mt.FORM_LATENT, mt.FORM_LATENT_ONE_KERNEL)
        for b in (1, 4, 16):
            lat = (0.5 * torch.randn(TP, b, L, device=dev, generator=g)).to(torch.bfloat16)
            sh = (0.5 * torch.randn(TP + 1, b, H, device=dev, generator=g)).to(torch.bfloat16)
            y = torch.empty((b, L), dtype=torch.bfloat16, device=dev)
            out = torch.empty((b, H), dtype=torch.bfloat16, device=dev)
            for promises in (False, True):
                def call(i):
                    mt.moe_tail_latent_up_flags(lat, gamma, wc[i % len(wc)], sh, out, y, inputs_ready=promises,
                                                weights_static=promises)
                for i in range(6):  # warm-up
                    call(i)
                torch.cuda.synchronize()
                tracer.attach()
                for i in range(6):
                    call(i)
                    torch.cuda.synchronize()
                print(f"-- b = {b}, promises {promises}")
                for kid, i, rs in launches(tracer.records())[1:3]:
                    print("  " + describe([(kid, i, rs)])[0])
    else:
        _, w = make_workload(dev)
        w["composition"] = args.composition
        stream = torch.cuda.Stream(dev, priority=-1)
        side = torch.cuda.Stream(dev, priority=0)
        tracer = Tracer(mt)
        with torch.cuda.stream(stream):
            for _ in range(3):
                run_step(mt, w, stream, side=side)
        torch.cuda.synchronize()
        steps = 10
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(steps):
                run_step(mt, w, stream, side=side)
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
    return 0


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, world, rank)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA arm has no CPU fallback)")
    if args.only_config is not None:
        return only_config(args)
    if args.trace is not None:
        return trace_run(args)
    return cuda_arm(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
