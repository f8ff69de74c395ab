"""The Python binding's argument checks, on the CPU.

The C entry points take bare pointers and read every layout from the sizes,
so the binding must refuse a tensor whose type or shape differs from the one
the sizes imply (a transposed weight, FP32 where BF16 is read, an index
tensor of another width) instead of handing it over to be misread.  Each
call here gets CPU tensors: with every type and shape right, the call must
get as far as the last check (tensors must be CUDA tensors) -- so the new
checks accept the shapes the GPU tests and the bench pass -- and with one
argument wrong it must name that argument."""
import numpy as np
import pytest
import torch

import moe_decode_tail_gb300 as mt
from moe_decode_tail_gb300 import synth

BF = torch.bfloat16
REACHED_CUDA_CHECK = "contiguous CUDA tensors"


def ep_args(b=4, tp=2, P=512, K=4):
    d = synth.ep_finalize_inputs(0xC0, b=b, tp=tp, P=P, K=K, num_experts=8)
    return [d["rows"], d["idx"], d["w"], d["gamma"], torch.empty((b, P), dtype=BF)]


def tp_args(b=6, tp=3, P=264, K=3):
    d = synth.tp_finalize_inputs(0xC1, b=b, tp=tp, P=P, K=K, num_experts=16)
    return [d["partials"], d["idx"], d["w"], d["gamma"], torch.empty((b, P), dtype=BF)]


def latent_args(b=3, tp=2, tp_s=2, L=264, H=200):
    d = synth.latent_up_inputs(0xC2, b=b, tp=tp, tp_s=tp_s, L=L, H=H)
    return [d["latent"], d["gamma"], d["w_up"], d["shared"], torch.empty((b, H), dtype=BF),
            torch.empty((b, L), dtype=BF)]


def shared_args(b=3, H=200, I=136):
    s = synth.shared_expert_inputs(0xC3, b=b, H=H, I=I)
    return [s["x"], s["w_gate"], s["w_up"], s["w_down"], torch.empty((b, H), dtype=BF),
            torch.empty(64, dtype=torch.uint8)]


def reaches_cuda_check(fn, *args, **kw):
    with pytest.raises(ValueError, match=REACHED_CUDA_CHECK):
        fn(*args, **kw)


FIN = [mt.moe_tail_ep_finalize, mt.moe_tail_ep_finalize_flags]
TPFIN = [mt.moe_tail_tp_finalize, mt.moe_tail_tp_finalize_flags]


@pytest.mark.parametrize("fn", FIN)
@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16])
def test_ep_finalize_accepts_its_shapes(fn, wdtype):
    rows, idx, w, gam, out = ep_args()
    reaches_cuda_check(fn, rows, idx, w.to(wdtype), gam, out)
    # no tokens: empty index and weights, an empty slice of a larger output
    big = torch.empty((4, 512), dtype=BF)
    reaches_cuda_check(fn, rows, idx[:, :0].contiguous(), w[:0].contiguous(), gam, big[:0])


@pytest.mark.parametrize("fn", TPFIN)
def test_tp_finalize_accepts_its_shapes(fn):
    parts, idx, w, gam, out = tp_args()
    reaches_cuda_check(fn, parts, idx, w, gam, out)
    # an earlier output read back as a one-slot partial tensor of b rows
    b2, K2 = 5, 2
    idx2 = torch.from_numpy((synth.u64(1, 1, b2 * K2) % 6).astype(np.int32).reshape(b2, K2))
    reaches_cuda_check(fn, out.view(1, 6, 264), idx2, synth.softmax_weights(1, 2, b2, K2), gam,
                       torch.empty((b2, 264), dtype=BF))


@pytest.mark.parametrize("fn", FIN + TPFIN)
@pytest.mark.parametrize("which,bad,name", [
    (0, lambda t: t.float(), "rows|partials"),                     # FP32 rows
    (0, lambda t: t[0], "rows|partials"),                          # a slot, not [tp, rows, P]
    (1, lambda t: t.long(), "permuted_idx"),                       # int64 indices
    (1, lambda t: t.reshape(-1), "permuted_idx"),                  # flattened indices
    (2, lambda t: t.double(), "route weights"),                    # FP64 weights
    (2, lambda t: t.reshape(-1), "route_weights"),                 # 1-D weights
    (3, lambda t: t.float(), "gamma"),                             # FP32 gamma
    (3, lambda t: t[:-8].contiguous(), "gamma"),                   # short gamma
    (4, lambda t: t.float(), "out"),                               # FP32 output
    (4, lambda t: t.t().contiguous(), "out"),                      # transposed output
])
def test_finalize_refuses_a_wrong_argument(fn, which, bad, name):
    args = ep_args() if fn in FIN else tp_args()
    args[which] = bad(args[which])
    with pytest.raises(ValueError, match=rf"^({name}) "):
        fn(*args)


@pytest.mark.parametrize("tp_s", [0, 2, 9])
def test_latent_calls_accept_their_shapes(tp_s):
    lat, gam, wu, sh, out, y = latent_args(tp_s=tp_s)
    ws = torch.empty(4096, dtype=torch.uint8)
    reaches_cuda_check(mt.moe_tail_latent_up, lat, gam, wu, sh, out, ws)
    reaches_cuda_check(mt.moe_tail_latent_up_flags, lat, gam, wu, sh, out, y, inputs_ready=True,
                       weights_static=True)
    reaches_cuda_check(mt.moe_tail_latent_up_noalloc, lat, gam, wu, sh, out)
    reaches_cuda_check(mt.moe_tail_latent_norm, lat, gam, y)
    reaches_cuda_check(mt.moe_tail_up_project, y, wu, sh, out)
    # y as the bench and the one-call form hold it: a view of a byte workspace
    yv = ws[: 3 * 264 * 2].view(BF).view(3, 264)
    reaches_cuda_check(mt.moe_tail_latent_norm, lat, gam, yv)


LATENT_BAD = [
    (0, lambda t: t.float(), "latent"),
    (0, lambda t: t.sum(0), "latent"),                         # slots already summed: 2-D
    (1, lambda t: t.float(), "gamma"),
    (1, lambda t: t[:-1].contiguous(), "gamma"),
    (2, lambda t: t.t().contiguous(), "w_up"),                 # [L, H] instead of [H, L]
    (2, lambda t: t.float(), "w_up"),
    (3, lambda t: t[:, :-1].contiguous(), "shared"),           # fewer tokens than the latent
    (3, lambda t: t.float(), "shared"),
    (3, lambda t: t[0], "shared"),                             # one slot, not [tp_s, b, H]
    (4, lambda t: t[:, :-2].contiguous(), "out"),
    (4, lambda t: t.float(), "out"),
]


@pytest.mark.parametrize("which,bad,name", LATENT_BAD)
def test_latent_calls_refuse_a_wrong_argument(which, bad, name):
    args = latent_args()
    args[which] = bad(args[which])
    lat, gam, wu, sh, out, y = args
    with pytest.raises(ValueError, match=rf"^({name}) "):
        mt.moe_tail_latent_up(lat, gam, wu, sh, out, torch.empty(4096, dtype=torch.uint8))
    with pytest.raises(ValueError, match=rf"^({name}) "):
        mt.moe_tail_latent_up_flags(lat, gam, wu, sh, out, y)
    with pytest.raises(ValueError, match=rf"^({name}) "):
        mt.moe_tail_latent_up_noalloc(lat, gam, wu, sh, out)


@pytest.mark.parametrize("bad", [lambda t: t.float(), lambda t: t.t().contiguous(), lambda t: t[:-1].contiguous()])
def test_latent_split_calls_refuse_a_wrong_y(bad):
    lat, gam, wu, sh, out, y = latent_args()
    with pytest.raises(ValueError, match="^y "):
        mt.moe_tail_latent_up_flags(lat, gam, wu, sh, out, bad(y))
    with pytest.raises(ValueError, match="^y "):
        mt.moe_tail_latent_norm(lat, gam, bad(y))
    with pytest.raises(ValueError, match="^(y|w_up|shared|out) "):
        mt.moe_tail_up_project(bad(y), wu, sh, out)


def test_up_project_refuses_mismatched_weights_and_partials():
    lat, gam, wu, sh, out, y = latent_args()
    with pytest.raises(ValueError, match="^w_up "):
        mt.moe_tail_up_project(y, wu.t().contiguous(), sh, out)
    with pytest.raises(ValueError, match="^shared "):
        mt.moe_tail_up_project(y, wu, sh[:, :-1].contiguous(), out)
    with pytest.raises(ValueError, match="^out "):
        mt.moe_tail_up_project(y, wu, sh, out.float())


def test_shared_expert_calls_accept_their_shapes():
    x, wg, wu, wd, out, ws = shared_args()
    h = torch.empty((3, 136), dtype=BF)
    reaches_cuda_check(mt.moe_shared_expert, x, wg, wu, wd, out, ws)
    reaches_cuda_check(mt.moe_shared_gate_up, x, wg, wu, h)
    reaches_cuda_check(mt.moe_shared_down, h, wd, out, accumulate=False)
    # the down projection into one slot of a [slots, b, H] partial tensor
    slots = torch.empty((9, 3, 200), dtype=BF)
    reaches_cuda_check(mt.moe_shared_down, h, wd, slots[8], accumulate=False)


@pytest.mark.parametrize("which,bad,name", [
    (0, lambda t: t.float(), "x"),
    (0, lambda t: t[:, :-1].contiguous(), "x|w_gate"),
    (1, lambda t: t.t().contiguous(), "w_gate"),
    (2, lambda t: t.t().contiguous(), "w_up"),
    (2, lambda t: t.float(), "w_up"),
    (3, lambda t: t.t().contiguous(), "w_down"),
    (4, lambda t: t[:-1].contiguous(), "out"),
])
def test_shared_expert_calls_refuse_a_wrong_argument(which, bad, name):
    args = shared_args()
    args[which] = bad(args[which])
    x, wg, wu, wd, out, ws = args
    with pytest.raises(ValueError, match=rf"^({name}) "):
        mt.moe_shared_expert(x, wg, wu, wd, out, ws)
    h = torch.empty((3, 136), dtype=BF)
    if which <= 2:
        with pytest.raises(ValueError, match=rf"^({name}) "):
            mt.moe_shared_gate_up(x, wg, wu, h)
    if which >= 3:
        with pytest.raises(ValueError, match=rf"^({name}) "):
            mt.moe_shared_down(h, wd, out)


def test_shared_split_calls_refuse_a_wrong_h():
    x, wg, wu, wd, out, ws = shared_args()
    for bad in (torch.empty((3, 136)), torch.empty((3, 135), dtype=BF), torch.empty((4, 136), dtype=BF)):
        with pytest.raises(ValueError, match="^h "):
            mt.moe_shared_gate_up(x, wg, wu, bad)
    with pytest.raises(ValueError, match="^h "):
        mt.moe_shared_down(torch.empty((3, 136)), wd, out)
    with pytest.raises(ValueError, match="^(w_down|out) "):
        mt.moe_shared_down(torch.empty((3, 135), dtype=BF), wd, out)


def test_missing_library_fails_loudly():
    # no CPU path: without the CUDA library every call that reaches it raises
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import moe_decode_tail_gb300 as mt\n"
            "try:\n"
            "    mt.moe_tail_workspace_bytes(0, 4, 512)\n"
            "except RuntimeError as e:\n"
            "    print('refused:', e)\n")
    env = dict(os.environ, MOE_TAIL_LIBRARY=os.path.join(root, "no_such_libmoetail.so"), PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=root, timeout=300)
    assert r.returncode == 0 and "refused:" in r.stdout and "is missing" in r.stdout, r.stdout + r.stderr
