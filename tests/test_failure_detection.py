"""Failure detection without a GPU fault: a kernel wait that expires is
reported through the device error word and the context stays usable.  The
expiry is produced two ways, and nothing traps and nothing hangs: a barrier
that nothing arrives at, with a 20 ms limit (the self-test kernel); and the
product kernels' own operand-stage waits cut to 1 ns, so that a GEMM and the
staged expert-TP finalize take their abort paths (stop issuing, wait for
their copies and tensor-core work in flight with the full limit, free tensor
memory, return) -- after which the next normal call must be bit-exact."""
import pytest
import torch

import oracle
from moe_decode_tail_gb300 import synth


@pytest.fixture(scope="module")
def mt():
    from moe_decode_tail_gb300 import build as cuda_build

    cuda_build.build()
    import moe_decode_tail_gb300

    moe_decode_tail_gb300.lib()
    return moe_decode_tail_gb300


def test_selftest_rejects_limits_out_of_range(mt):
    # host-side checks only: nothing is launched
    assert mt.lib().moe_tail_selftest_wait_timeout(0, None) == mt.EINVAL
    assert mt.lib().moe_tail_selftest_wait_timeout(1000001, None) == mt.EINVAL


@pytest.mark.skipif(torch.cuda.is_available(), reason="with a GPU a valid limit launches the self-test")
def test_selftest_accepts_the_limits_at_the_ends_of_its_range(mt):
    # 1 us and 1 s pass the host checks; with no GPU visible the call then
    # fails at its first CUDA call instead of being refused
    assert mt.lib().moe_tail_selftest_wait_timeout(1, None) == mt.ECUDA
    assert mt.lib().moe_tail_selftest_wait_timeout(1000000, None) == mt.ECUDA


@pytest.mark.gpu
def test_expired_wait_is_reported_and_the_device_stays_usable(mt):
    assert mt.moe_tail_take_device_error() == 0
    mt.moe_tail_selftest_wait_timeout(20000)
    torch.cuda.synchronize()
    assert mt.moe_tail_take_device_error() & 1
    assert mt.moe_tail_take_device_error() == 0  # read clears it
    # a normal call afterwards still computes the right result
    d = synth.config(1)
    ref = oracle.ep_finalize(d["rows"], d["rows_per_slot"], d["idx"], d["w"], d["gamma"], d["gain_center"],
                             d["eps"], d["weight_before_norm"], d["b"], d["tp"], d["K"], d["P"])
    out = torch.full((d["b"], d["P"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    mt.moe_tail_ep_finalize(d["rows"].cuda(), d["idx"].cuda(), d["w"].cuda(), d["gamma"].cuda(), out,
                            gain_center=d["gain_center"], eps=d["eps"], weight_before_norm=d["weight_before_norm"])
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().view(torch.int16), ref.view(torch.int16))
    assert mt.moe_tail_take_device_error() == 0


def test_stage_wait_limit_above_a_second_is_refused(mt):
    # host-side checks only: nothing is launched
    assert mt.lib().moe_tail_set_stage_wait_limit(1_000_000_001) == mt.EINVAL
    assert mt.lib().moe_tail_set_stage_wait_limit(0) == mt.OK


def _short_stage_wait_then_normal(mt, call):
    """Run call() once with a 1 ns operand-stage wait (no stage of weights or
    rows can land that fast, so the kernels abort), then with the default
    limit; returns (error bits after the first run, the second run's output)."""
    assert mt.moe_tail_take_device_error() == 0
    mt.moe_tail_set_stage_wait_limit(1)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        mt.moe_tail_set_stage_wait_limit(0)
    bits = mt.moe_tail_take_device_error()
    out = call()
    torch.cuda.synchronize()
    return bits, out


@pytest.mark.gpu
def test_gemm_abort_path_raises_and_the_next_call_is_exact(mt):
    # the up-projection GEMM (clusters of 8 CTAs splitting K): the tensor-core
    # issuer's stage wait runs out, the CTA stops issuing, waits for its copies
    # in flight and its issued work, frees its tensor memory and returns
    b, L, H = 8, 1024, 1024
    d = synth.latent_up_inputs(0xAB0, b=b, tp=2, tp_s=2, L=L, H=H)
    y = d["latent"][0].contiguous().cuda()
    w, sh = d["w_up"].cuda(), d["shared"].cuda()

    def call():
        out = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        mt.moe_tail_up_project(y, w, sh, out)
        return out

    ref = call()
    torch.cuda.synchronize()
    bits, out = _short_stage_wait_then_normal(mt, call)
    assert bits & 1, bits
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["gate_up", "down", "down_up", "persistent_down", "latent_one_kernel"])
def test_every_gemm_mode_aborts_cleanly_and_the_next_call_is_exact(mt, pin, mode):
    # each other decode-GEMM kernel the same way: its operand-stage wait runs
    # out, it raises bit 1, drains what it started and returns; the next call
    # with the default limit gives the bits of a call made before
    b, H, I, L = 8, 1024, 768, 512
    s = synth.shared_expert_inputs(0xAB1, b=b, H=H, I=I)
    x, wg, wu, wd = (s[k].cuda() for k in ("x", "w_gate", "w_up", "w_down"))
    h = synth.bf16(synth.normal(0xAB2, 1, b * I, std=0.5), (b, I)).cuda()
    d = synth.latent_up_inputs(0xAB3, b=b, tp=2, tp_s=2, L=L, H=H)
    lat, gam, wl, sh = d["latent"].cuda(), d["gamma"].cuda(), d["w_up"].cuda(), d["shared"].cuda()
    y = d["latent"][0].contiguous().cuda()
    if mode == "latent_one_kernel":
        pin(mt.FORM_LATENT, mt.FORM_LATENT_ONE_KERNEL)

    def call():
        if mode == "gate_up":
            out = torch.full((b, I), float("nan"), dtype=torch.bfloat16, device="cuda")
            mt.moe_shared_gate_up(x, wg, wu, out)
        elif mode == "latent_one_kernel":
            out = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device="cuda")
            yy = torch.empty((b, L), dtype=torch.bfloat16, device="cuda")
            mt.moe_tail_latent_up_flags(lat, gam, wl, sh, out, yy, eps=d["eps"])
        else:
            out = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device="cuda")
            if mode == "down":
                mt.moe_shared_down(h, wd, out, accumulate=False)
            elif mode == "persistent_down":
                mt.moe_shared_down_persistent(h, wd, out, accumulate=False, ctas=3)
            else:
                mt.moe_tail_up_project_shared_down(y, wl, sh, h, wd, out)
        return out

    ref = call()
    torch.cuda.synchronize()
    bits, out = _short_stage_wait_then_normal(mt, call)
    assert bits & 1, bits
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.gpu
def test_staged_finalize_abort_path_raises_and_the_next_call_is_exact(mt, pin):
    # the staged expert-TP finalize: its threads' stage wait runs out, nothing
    # more is copied, and the copies in flight land before the CTA ends
    pin(mt.FORM_TP, 1)
    d = synth.config(3, b=64)
    args = [d[k].cuda() for k in ("partials", "idx", "w", "gamma")]

    def call():
        out = torch.full((d["b"], d["P"]), float("nan"), dtype=torch.bfloat16, device="cuda")
        mt.moe_tail_tp_finalize(*args, out, gain_center=d["gain_center"], eps=d["eps"],
                                weight_before_norm=d["weight_before_norm"])
        return out

    ref = call()
    torch.cuda.synchronize()
    bits, out = _short_stage_wait_then_normal(mt, call)
    assert bits & 1, bits
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert mt.moe_tail_take_device_error() == 0
