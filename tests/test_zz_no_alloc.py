"""moe_tail_latent_up_noalloc: the latent tail for callers that cannot
allocate device memory (a plugin handed only its input and output buffers, a
host whose device memory is all held by its own pool, a hot path that must not
call cudaMalloc).  It keeps y in a fixed array inside the library instead of a
caller workspace; its output must match moe_tail_latent_up's on the same
inputs, call after call, since every call reuses that one array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone."""
import ctypes

import pytest
import torch

from moe_decode_tail_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    from moe_decode_tail_gb300 import build as cuda_build

    cuda_build.build()
    import moe_decode_tail_gb300

    moe_decode_tail_gb300.lib()
    return moe_decode_tail_gb300


def close(got, ref):
    """|got - ref| <= 2 BF16 ulp(|ref|) + 1e-3, the GEMM tolerance of the tests."""
    g, r = got.float().cpu(), ref.float().cpu()
    ulp = torch.exp2(torch.floor(torch.log2(r.abs().clamp_min(2.0 ** -126))) - 7)
    return bool(((g - r).abs() <= 2 * ulp + 1e-3).all())


def inputs(seed, b, L=3584, H=7168, tp=8, tp_s=8):
    d = synth.latent_up_inputs(seed, b=b, tp=tp, L=L, H=H, tp_s=tp_s)
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def with_workspace(mt, d):
    b, L, H = d["b"], d["L"], d["H"]
    ws = torch.empty(mt.moe_tail_workspace_bytes(0, b, L), dtype=torch.uint8, device="cuda")
    out = torch.empty((b, H), dtype=torch.bfloat16, device="cuda")
    mt.moe_tail_latent_up(d["latent"], d["gamma"], d["w_up"], d["shared"], out, ws, eps=d["eps"])
    return out


def without_workspace(mt, d):
    out = torch.full((d["b"], d["H"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    mt.moe_tail_latent_up_noalloc(d["latent"], d["gamma"], d["w_up"], d["shared"], out, eps=d["eps"])
    return out


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row(mt):
    # two different problems back to back: the second call reuses the array
    # the first one filled, so stale contents would show up here
    first = inputs(0x5EED0004, b=16)
    second = inputs(0x5EED0044, b=64, tp_s=0)
    a1 = without_workspace(mt, first)
    a2 = without_workspace(mt, second)
    torch.cuda.synchronize()
    assert close(a1, with_workspace(mt, first))
    assert close(a2, with_workspace(mt, second))
    # and the first problem again, after the larger one
    a3 = without_workspace(mt, first)
    assert close(a3, with_workspace(mt, first))
    assert mt.moe_tail_take_device_error() == 0


def test_noalloc_refuses_a_problem_larger_than_its_array(mt):
    b, L = 147, 3584  # y = 147 * 3584 * 2 bytes > 1 MiB
    d = inputs(7, b=b, L=L, H=256, tp=1, tp_s=0)
    out = torch.zeros((b, 256), dtype=torch.bfloat16, device="cuda")
    rc = mt.lib().moe_tail_latent_up_noalloc(
        ctypes.c_void_p(d["latent"].data_ptr()), ctypes.c_void_p(d["gamma"].data_ptr()), d["eps"],
        ctypes.c_void_p(d["w_up"].data_ptr()), None, 0, b, 1, L, 256, ctypes.c_void_p(out.data_ptr()), None)
    assert rc == mt.EINVAL
    with pytest.raises(ValueError, match="scratch"):
        mt.moe_tail_latent_up_noalloc(d["latent"], d["gamma"], d["w_up"], None, out)
    torch.cuda.synchronize()
    assert bool((out.float() == 0).all())  # nothing ran


def test_noalloc_in_the_one_kernel_form(mt, pin):
    # with the latent tail's one-kernel form pinned, the call keeps y on chip and
    # passes the kernel no y pointer at all; at a batch that form takes (b = 8)
    # its output must still match the workspace entry point's, and no bounded
    # wait may have expired
    pin(mt.FORM_LATENT, mt.FORM_LATENT_ONE_KERNEL)
    d = inputs(0x5EED0048, b=8)
    got = without_workspace(mt, d)
    torch.cuda.synchronize()
    assert mt.moe_tail_take_device_error() == 0
    pin(mt.FORM_LATENT, 2)  # the reference: the workspace entry point as its two kernels
    ref = with_workspace(mt, d)
    torch.cuda.synchronize()
    assert close(got, ref)
    assert mt.moe_tail_take_device_error() == 0
