"""The composed decode step exactly as bench.py times it (two branches: the
shared expert -- as its two calls, or as one -- then the latent tail on a
side stream, EP and expert-TP finalize beside them, or on the side stream
the shared expert's gate/up, the latent norm and then the down projection
with the up-projection in one kernel; and the sequential
composition, where the shared
expert accumulates into the latent tail's output; and latent_main, where the
latent tail runs beside the shared expert's gate/up and the down projection
then accumulates into its output), checked against the oracle on sampled
tokens:
EP and expert-TP outputs and the latent norm's y bit for bit; in the two
branch compositions, the step's output against the oracle's up-projection of
the GPU's y with the shared expert's BF16 output d as one more shared partial
(GEMM bound), and d against the oracle's down projection of the GPU's h (GEMM
bound); where d is added into the latent tail's output instead, each term at
the GEMM bound and the add bit for bit, given the GPU's own terms."""
import importlib.util
import os

import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOKENS = (0, 1, 29, 63)


def close(got, ref, what):
    g, r = got.float(), ref.float()
    ulp = torch.exp2(torch.floor(torch.log2(r.abs().clamp_min(2.0 ** -126))) - 7)
    bad = (g - r).abs() > 2 * ulp + 1e-3
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} of {bad.numel()} out of tolerance"


@pytest.fixture(scope="module", params=["two_branch", "two_branch_one_call", "sequential", "latent_main",
                                        "two_branch_fused"])
def step(request):
    from moe_decode_tail_gb300 import build as cuda_build

    cuda_build.build()
    import moe_decode_tail_gb300 as mt

    mt.lib()
    spec = importlib.util.spec_from_file_location("bench_step", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dev = torch.device("cuda", 0)
    cpu, w = bench.make_workload(dev)
    stream = torch.cuda.Stream(dev, priority=-1)
    side = None if request.param == "sequential" else torch.cuda.Stream(dev, priority=0)
    if side is not None:
        w["composition"] = request.param
    for k in ("out_ep", "out_tp", "out", "y"):
        w[k].fill_(float("nan"))
    w["d_slot"].fill_(float("nan"))
    if request.param == "sequential":  # the shared expert adds into the latent tail's output (after it)
        w["out"].zero_()
    with torch.cuda.stream(stream):
        bench.run_step(mt, w, stream, side=side)
    torch.cuda.synchronize()
    assert mt.moe_tail_take_device_error() == 0
    got = {k: w[k].cpu() for k in ("out_ep", "out_tp", "out", "shared9")}
    got["y"] = w["ws_lat"][: bench.B * bench.L * 2].view(torch.bfloat16).view(bench.B, bench.L).cpu()
    if request.param in ("sequential", "latent_main"):
        # the two terms of the step's last add, recomputed alone from the same
        # inputs (both calls are deterministic): the latent tail's own output,
        # and d = bf16(down(h)) of the step's h
        B, I = bench.B, bench.I
        ws = torch.empty_like(w["ws_lat"])
        tail = torch.full_like(w["out"], float("nan"))
        mt.moe_tail_latent_up(w["latent"], w["lat_gamma"], w["w_up"], w["shared"], tail, ws, eps=1e-6)
        d = torch.full_like(w["out"], float("nan"))
        mt.moe_shared_down(w["ws_sh"][: B * I * 2].view(torch.bfloat16).view(B, I), w["w_down"], d, accumulate=False)
        torch.cuda.synchronize()
        got["tail"], got["d"] = tail.cpu(), d.cpu()
    if request.param == "two_branch_fused":
        # the fused call again, with its optional d output: the same out, and d
        B, I = bench.B, bench.I
        again = torch.full_like(w["out"], float("nan"))
        d = torch.full_like(w["out"], float("nan"))
        mt.moe_tail_up_project_shared_down(w["y"], w["w_up"], w["shared"],
                                           w["ws_sh"][: B * I * 2].view(torch.bfloat16).view(B, I), w["w_down"],
                                           again, d)
        torch.cuda.synchronize()
        got["out_again"], got["d"] = again.cpu(), d.cpu()
    return bench, cpu, got, w["ws_sh"].cpu(), request.param


def test_step_finalize_outputs(step):
    bench, cpu, got, _, _ = step
    ep, tp = cpu["ep"], cpu["tp"]
    for t in TOKENS:
        ref = oracle.ep_finalize(ep["rows"], ep["rows_per_slot"], ep["idx"][:, t:t + 1].contiguous(),
                                 ep["w"][t:t + 1].contiguous(), ep["gamma"], 1.0, 1e-6, True, 1, bench.TP,
                                 bench.K_ROUTES, bench.P)
        assert torch.equal(got["out_ep"][t:t + 1].view(torch.int16), ref.view(torch.int16)), f"EP token {t}"
        ref = oracle.tp_finalize(tp["partials"], tp["num_rows"], tp["idx"][t:t + 1].contiguous(),
                                 tp["w"][t:t + 1].contiguous(), tp["gamma"], 1.0, 1e-6, True, 1, bench.TP,
                                 bench.K_ROUTES, bench.P)
        assert torch.equal(got["out_tp"][t:t + 1].view(torch.int16), ref.view(torch.int16)), f"TP token {t}"


def test_step_latent_tail_and_shared_expert(step):
    bench, cpu, got, ws_sh, mode = step
    lat, sh = cpu["lat"], cpu["sh"]
    B, L, H, I, TP = bench.B, bench.L, bench.H, bench.I, bench.TP
    h_gpu = ws_sh[: B * I * 2].view(torch.bfloat16).view(B, I)
    for t in TOKENS:
        y_ref = oracle.latent_norm(lat["latent"][:, t:t + 1].contiguous(), lat["gamma"], 1e-6, 1, TP, L)
        assert torch.equal(got["y"][t:t + 1].view(torch.int16), y_ref.view(torch.int16)), f"y token {t}"
        if mode == "two_branch_fused":
            # d: a valid down projection of the GPU's h; out: the up-projection of y
            # plus the eight shared partials and d, d last
            d_ref = oracle.shared_down(h_gpu[t:t + 1].contiguous(), sh["w_down"], 1, H, I, accumulate=False)
            close(got["d"][t:t + 1], d_ref, f"d token {t}")
            sh9 = torch.cat([got["shared9"][:TP, t:t + 1], got["d"][None, t:t + 1]]).contiguous()
            close(got["out"][t:t + 1], oracle.latent_up(got["y"][t:t + 1].contiguous(), lat["w_up"], sh9, TP + 1, 1,
                                                        L, H), f"out token {t}")
        elif mode.startswith("two_branch"):
            # d: a valid down projection of the GPU's h; out: the up-projection of y
            # plus all nine partials (d included)
            d_gpu = got["shared9"][TP]
            d_ref = oracle.shared_down(h_gpu[t:t + 1].contiguous(), sh["w_down"], 1, H, I, accumulate=False)
            close(d_gpu[t:t + 1], d_ref, f"d token {t}")
            out_ref = oracle.latent_up(got["y"][t:t + 1].contiguous(), lat["w_up"],
                                       got["shared9"][:, t:t + 1].contiguous(), TP + 1, 1, L, H)
            close(got["out"][t:t + 1], out_ref, f"out token {t}")
        else:
            # out = bf16(latent tail + bf16(down(h))): each term against the oracle
            # (the tail from the GPU's y, d from the GPU's h) at the GEMM bound ...
            tail_ref = oracle.latent_up(got["y"][t:t + 1].contiguous(), lat["w_up"],
                                        got["shared9"][:TP, t:t + 1].contiguous(), TP, 1, L, H)
            close(got["tail"][t:t + 1], tail_ref, f"latent tail token {t}")
            d_ref = oracle.shared_down(h_gpu[t:t + 1].contiguous(), sh["w_down"], 1, H, I, accumulate=False)
            close(got["d"][t:t + 1], d_ref, f"d token {t}")
    if mode == "two_branch_fused":
        assert torch.equal(got["out_again"].view(torch.int16), got["out"].view(torch.int16)), "fused call repeats"
    if not mode.startswith("two_branch"):
        # ... and the add itself bit for bit, every token: pz(bf16(f32(tail) + f32(d)))
        s = got["tail"].float() + got["d"].float()
        ref = s.to(torch.bfloat16).view(torch.int16)
        ref = torch.where(ref == -32768, torch.zeros_like(ref), ref)
        assert torch.equal(got["out"].view(torch.int16), ref), f"{mode}: out != bf16(tail + d)"
