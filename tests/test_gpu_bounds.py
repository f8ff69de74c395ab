"""Every entry point writes only inside its outputs and workspace.

compute-sanitizer is closed on this machine, so out-of-range writes are caught
with canaries: each output and workspace is carved out of a larger buffer
whose 4 KB before and after hold a sentinel byte, the call runs at ragged
sizes (widths not multiples of a tile, odd token counts, more than one K
split, both finalize kernels, both latent-tail forms, the up-projection with
the shared down projection, the persistent down projection), and the sentinel bytes
must be unchanged afterwards.  The values themselves are checked by the
parity tests."""
import math

import pytest
import torch

from moe_decode_tail_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
PAD = 4096
SENTINEL = 0x5A


@pytest.fixture(scope="module")
def mt():
    from moe_decode_tail_gb300 import build as cuda_build

    cuda_build.build()
    import moe_decode_tail_gb300

    moe_decode_tail_gb300.lib()
    return moe_decode_tail_gb300


class Guarded:
    """A tensor (or a byte workspace) inside a sentinel-filled buffer."""

    def __init__(self, shape, dtype=torch.bfloat16, nbytes=None):
        self.n = nbytes if nbytes is not None else math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((PAD + self.n + PAD,), SENTINEL, dtype=torch.uint8, device=DEV)
        inner = self.buf[PAD: PAD + self.n]
        self.t = inner if nbytes is not None else inner.view(dtype).view(shape)
        if nbytes is None and dtype == torch.bfloat16:
            self.t.fill_(float("nan"))

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[:PAD] == SENTINEL).all()) and bool((self.buf[PAD + self.n:] == SENTINEL).all())


def dev(d, *keys):
    return [d[k].to(DEV) for k in keys]


@pytest.mark.parametrize("kw", [dict(b=5, tp=3, P=264, K=3, num_experts=9), dict(b=33, tp=8, P=1000, K=8, num_experts=32)])
def test_ep_finalize(mt, kw):
    d = synth.ep_finalize_inputs(0xB0 + kw["b"], **kw)
    out = Guarded((d["b"], d["P"]))
    rows, idx, w, gam = dev(d, "rows", "idx", "w", "gamma")
    mt.moe_tail_ep_finalize(rows, idx, w, gam, out.t, gain_center=d["gain_center"], eps=d["eps"],
                            weight_before_norm=True)
    out2 = Guarded((d["b"], d["P"]))
    mt.moe_tail_ep_finalize_flags(rows, idx, w, gam, out2.t, gain_center=d["gain_center"], eps=d["eps"],
                                  weight_before_norm=True, inputs_ready=True)
    assert out.intact() and out2.intact()
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.parametrize("staged", ["0", "1"])
@pytest.mark.parametrize("kw", [dict(b=9, tp=3, P=264, K=5), dict(b=70, tp=2, P=1000, K=8)])
def test_tp_finalize(mt, pin, staged, kw):
    pin(mt.FORM_TP, 1 if staged == "1" else 2)
    d = synth.tp_finalize_inputs(0xB1 + kw["b"], num_experts=16, **kw)
    out = Guarded((d["b"], d["P"]))
    parts, idx, w, gam = dev(d, "partials", "idx", "w", "gamma")
    mt.moe_tail_tp_finalize(parts, idx, w, gam, out.t, gain_center=d["gain_center"], eps=d["eps"],
                            weight_before_norm=False)
    out2 = Guarded((d["b"], d["P"]))
    mt.moe_tail_tp_finalize_flags(parts, idx, w, gam, out2.t, gain_center=d["gain_center"], eps=d["eps"],
                                  weight_before_norm=False, inputs_ready=True)
    assert out.intact() and out2.intact()
    assert mt.moe_tail_take_device_error() == 0


LATENT = [dict(b=5, tp=3, tp_s=2, L=264, H=200), dict(b=17, tp=2, tp_s=1, L=1000, H=520),
          dict(b=33, tp=4, tp_s=0, L=512, H=136)]


@pytest.mark.parametrize("kw", LATENT)
def test_latent_tail_calls(mt, pin, kw):
    d = synth.latent_up_inputs(0xB2 + kw["b"], **kw)
    b, L, H = d["b"], d["L"], d["H"]
    lat, gam, wu = dev(d, "latent", "gamma", "w_up")
    sh = None if d["shared"] is None else d["shared"].to(DEV)
    guards = []
    # one call, with its workspace exactly as large as required
    out, ws = Guarded((b, H)), Guarded(None, nbytes=mt.moe_tail_workspace_bytes(0, b, L))
    mt.moe_tail_latent_up(lat, gam, wu, sh, out.t, ws.t, eps=d["eps"])
    guards += [out, ws]
    # the two steps as split calls
    y, out2 = Guarded((b, L)), Guarded((b, H))
    mt.moe_tail_latent_norm(lat, gam, y.t, eps=d["eps"], inputs_ready=True)
    mt.moe_tail_up_project(y.t, wu, sh, out2.t, weights_static=True)
    guards += [y, out2]
    # the flags call in both forms, and the call without a workspace
    for one_kernel in ("0", "1"):
        pin(mt.FORM_LATENT, 1 if one_kernel == "1" else 2)
        y3, out3 = Guarded((b, L)), Guarded((b, H))
        mt.moe_tail_latent_up_flags(lat, gam, wu, sh, out3.t, y3.t, eps=d["eps"], inputs_ready=True,
                                    weights_static=True)
        out4 = Guarded((b, H))
        mt.moe_tail_latent_up_noalloc(lat, gam, wu, sh, out4.t, eps=d["eps"])
        guards += [y3, out3, out4]
    assert all(g.intact() for g in guards)
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.parametrize("kw", [dict(b=3, H=520, I=200), dict(b=65, H=264, I=392)])
def test_shared_expert_calls(mt, kw):
    s = synth.shared_expert_inputs(0xB3 + kw["b"], **kw)
    b, H, I = s["b"], s["H"], s["I"]
    x, wg, wu, wd = dev(s, "x", "w_gate", "w_up", "w_down")
    out, ws = Guarded((b, H)), Guarded(None, nbytes=mt.moe_tail_workspace_bytes(1, b, I))
    out.t.zero_()
    mt.moe_shared_expert(x, wg, wu, wd, out.t, ws.t, accumulate=True)
    h, out2 = Guarded((b, I)), Guarded((b, H))
    mt.moe_shared_gate_up(x, wg, wu, h.t, weights_static=True)
    mt.moe_shared_down(h.t, wd, out2.t, accumulate=False, weights_static=True)
    out3, out4 = Guarded((b, H)), Guarded((b, H))
    out4.t.zero_()
    mt.moe_shared_down_persistent(h.t, wd, out3.t, accumulate=False, ctas=3)
    mt.moe_shared_down_persistent(h.t, wd, out4.t, accumulate=True)
    assert all(g.intact() for g in (out, ws, h, out2, out3, out4))
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.parametrize("kw", [dict(b=37, L=264, I=200, H=136, tp_s=3), dict(b=5, L=1000, I=520, H=392, tp_s=0)])
def test_up_project_shared_down(mt, kw):
    b, L, I, H, tp_s = kw["b"], kw["L"], kw["I"], kw["H"], kw["tp_s"]
    g = lambda *shape: (0.5 * torch.randn(*shape, device=DEV)).to(torch.bfloat16)
    y, w_up, h, w_down = g(b, L), g(H, L), g(b, I), g(H, I)
    shared = g(tp_s, b, H) if tp_s else None
    out, d = Guarded((b, H)), Guarded((b, H))
    mt.moe_tail_up_project_shared_down(y, w_up, shared, h, w_down, out.t, d.t, weights_static=True)
    out2 = Guarded((b, H))
    mt.moe_tail_up_project_shared_down(y, w_up, shared, h, w_down, out2.t)
    assert out.intact() and d.intact() and out2.intact()
    assert mt.moe_tail_take_device_error() == 0
