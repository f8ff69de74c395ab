"""Failure detection without a GPU fault: a kernel wait that expires is
reported through the device error word and the context stays usable.  The
expiry is produced by a barrier that nothing arrives at, with a 20 ms limit;
nothing traps and nothing hangs."""
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
