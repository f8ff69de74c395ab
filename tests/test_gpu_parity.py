"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Finalize outputs and the latent norm's y must be bit-exact BF16; the GEMM
paths (latent up-projection, shared expert h and output) must satisfy
|gpu - oracle| <= 2 ulp_bf16(|oracle|) + 1e-3 element by element.  Inputs are
the seeded decode workloads (full sizes where the oracle finishes in seconds,
sampled tokens otherwise) plus ragged, degenerate and crafted-rounding cases.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_tail_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def mt():
    from moe_decode_tail_gb300 import build as cuda_build

    cuda_build.build()
    oracle.build()
    import moe_decode_tail_gb300

    moe_decode_tail_gb300.lib()
    yield moe_decode_tail_gb300
    assert moe_decode_tail_gb300.moe_tail_take_device_error() == 0


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def assert_bitexact(got, ref, what=""):
    g, r = bits(got), bits(ref)
    if not np.array_equal(g, r):
        bad = np.argwhere(g != r)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {g.size} differ; first at {i}: "
                             f"gpu {got.float().cpu()[i].item()!r} oracle {ref.float()[i].item()!r}")


def assert_gemm_close(got, ref, what=""):
    g = got.detach().float().cpu()
    r = ref.float()
    ulp = torch.exp2(torch.floor(torch.log2(r.abs().clamp_min(2.0 ** -126))) - 7)
    err = (g - r).abs()
    ok = err <= 2 * ulp + 1e-3
    if not bool(ok.all()):
        i = tuple(torch.nonzero(~ok)[0].tolist())
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.numel()} out of tolerance; first at {i}: "
                             f"gpu {g[i].item()!r} oracle {r[i].item()!r}")


def accumulated(out_in, d):
    """pz(bf16(f32(out_in) + f32(d))): the accumulate step's one rounding, in
    FP32 on the host (d is the BF16 down output the GPU wrote)."""
    s = out_in.detach().float().cpu() + d.detach().float().cpu()  # one IEEE binary32 add per element
    b = s.to(torch.bfloat16).view(torch.int16)  # round to nearest even
    return torch.where(b == -32768, torch.zeros_like(b), b).view(torch.bfloat16)


def assert_accumulated_exact(got, out_in, d, what=""):
    """out = bf16(out_in + bf16(d)) bit for bit, given the GPU's own bf16(d):
    once d is known nothing in the accumulate step is left to tolerance."""
    assert_bitexact(got, accumulated(out_in, d), what)


# ------------------------------------------------------------------ EP finalize

def run_ep(mt, d, out=None, **kw):
    a = dict(d)
    a.update(kw)
    if out is None:
        out = torch.full((a["b"], a["P"]), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_ep_finalize(a["rows"].to(DEV), a["idx"].to(DEV), a["w"].to(DEV), a["gamma"].to(DEV), out,
                            gain_center=a["gain_center"], eps=a["eps"], weight_before_norm=a["weight_before_norm"])
    torch.cuda.synchronize()
    return out


def ref_ep(d, **kw):
    a = dict(d)
    a.update(kw)
    return oracle.ep_finalize(a["rows"], a["rows_per_slot"], a["idx"], a["w"], a["gamma"], a["gain_center"],
                              a["eps"], a["weight_before_norm"], a["b"], a["tp"], a["K"], a["P"])


def bf16_bits_pz(x32):
    """BF16 bits (round to nearest even, -0 made +0) of float32 values."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    b = t.view(torch.int16).numpy().astype(np.uint16)
    b[b == 0x8000] = 0
    return b


def fp32_inv_rms(ss, P, eps=1e-6):
    """1 / sqrt(ss * (float)(1/P) + eps), each step one FP32 operation."""
    f = np.float32
    return f(1.0) / np.sqrt(f(f(ss) * f(1.0 / P)) + f(eps))


@pytest.mark.parametrize("wbn", [True, False])
@pytest.mark.parametrize("wdtype", [torch.float32, torch.bfloat16])
def test_ep_routing_marker_rows(mt, wbn, wdtype):
    # Every route row is a marker: 1.0 at column s*R + j (slot s, row j), zeros
    # elsewhere; route k has weight 2^-k and the gains are 1.  Token t's output
    # then holds bf16(inv * 2^-k) at column s*R + j for each local route (s, k)
    # with idx[s][t][k] = j -- inv = 1/sqrt(1/P + eps) in FP32 -- and zeros
    # elsewhere.  The expected output is written here from the routing table
    # alone (no oracle): a wrong slot, row, route weight or locality test shows
    # up as a lit or dark column.
    b, tp, R, K, P = 16, 4, 8, 4, 512
    rng = np.random.default_rng(0x3A7)
    idx = np.empty((tp, b, K), dtype=np.int32)
    for s in range(tp):
        for t in range(b):  # distinct per (slot, token): -3..-1 and R..R+2 are not local
            idx[s, t] = rng.choice(np.arange(-3, R + 3), size=K, replace=False)
    rows = torch.zeros((tp, R, P))
    for s in range(tp):
        for j in range(R):
            rows[s, j, s * R + j] = 1.0
    w = torch.tensor([[2.0 ** -k for k in range(K)]] * b, dtype=torch.float32).to(wdtype)
    d = dict(rows=rows.to(torch.bfloat16), rows_per_slot=R, idx=torch.from_numpy(idx), w=w,
             gamma=torch.zeros(P, dtype=torch.bfloat16), gain_center=1.0, eps=1e-6, weight_before_norm=wbn,
             b=b, tp=tp, K=K, P=P)
    inv = fp32_inv_rms(1.0, P)
    expect = np.zeros((b, P), dtype=np.float32)
    for s in range(tp):
        for t in range(b):
            for k in range(K):
                j = idx[s, t, k]
                if 0 <= j < R:
                    expect[t, s * R + j] = inv * np.float32(2.0 ** -k)
    out = run_ep(mt, d)
    got = bits(out).astype(np.uint16)
    assert np.array_equal(got, bf16_bits_pz(expect)), "EP marker rows: routing"
    assert_bitexact(out, ref_ep(d), "EP marker rows vs oracle")


@pytest.mark.parametrize("wbn", [True, False])
def test_tp_routing_marker_rows(mt, wbn):
    # Every slot's K-partial of row j holds 1.0 at column j, and slot s adds a
    # slot marker 2^-s at column 256 + s; route k has weight 2^-k, gains 1.
    # So x_j = tp at column j and 2^-s at 256 + s, ss = tp^2 + sum_s 4^-s
    # exactly, and token t's output is bf16(tp * inv * 2^-k) at column
    # idx[t][k] for each valid route, the route-ordered FP32 sum of
    # (2^-s * inv) * 2^-k over the valid routes at column 256 + s (every slot
    # must have been summed), and zeros elsewhere -- written out here from the
    # routing table, without the oracle.
    b, tp, K, P, rows_n = 16, 4, 4, 512, 32
    rng = np.random.default_rng(0x3A8)
    idx = np.stack([rng.choice(np.arange(-2, rows_n + 2), size=K, replace=False) for _ in range(b)])
    idx = idx.astype(np.int32)
    q = torch.zeros((tp, rows_n, P))
    for s in range(tp):
        for j in range(rows_n):
            q[s, j, j] = 1.0
            q[s, j, 256 + s] = 2.0 ** -s
    d = dict(partials=q.to(torch.bfloat16), num_rows=rows_n, idx=torch.from_numpy(idx),
             w=torch.tensor([[2.0 ** -k for k in range(K)]] * b, dtype=torch.float32),
             gamma=torch.zeros(P, dtype=torch.bfloat16), gain_center=1.0, eps=1e-6, weight_before_norm=wbn,
             b=b, tp=tp, K=K, P=P)
    f = np.float32
    ss = f(f(0.0) + f(tp * tp))  # chunk 0: the route column
    marker_sq = f(0.0)
    for s in range(tp):  # chunk 1: lane 0 squares columns 256.. in order
        marker_sq = f(marker_sq + f(f(2.0 ** -s) * f(2.0 ** -s)))
    ss = f(ss + marker_sq)
    inv = fp32_inv_rms(ss, P)
    expect = np.zeros((b, P), dtype=np.float32)
    for t in range(b):
        acc = np.zeros(tp, dtype=np.float32)
        for k in range(K):
            j = idx[t, k]
            if 0 <= j < rows_n:
                expect[t, j] = f(f(tp) * inv) * f(2.0 ** -k)
                for s in range(tp):
                    acc[s] = f(acc[s] + f(f(f(2.0 ** -s) * inv) * f(2.0 ** -k)))
        expect[t, 256:256 + tp] = acc
    out = run_tp(mt, d)
    got = bits(out).astype(np.uint16)
    assert np.array_equal(got, bf16_bits_pz(expect)), "TP marker rows: routing and slot sum"
    assert_bitexact(out, ref_tp(d), "TP marker rows vs oracle")


@pytest.mark.parametrize("wbn", [True, False])
def test_ep_tiny(mt, wbn):
    d = synth.config(1, weight_before_norm=wbn)
    assert_bitexact(run_ep(mt, d), ref_ep(d), "EP b=4 tp=2 P=512")


@pytest.mark.parametrize("wbn", [True, False])
def test_ep_decode_full(mt, wbn):
    d = synth.config(2, weight_before_norm=wbn)
    assert_bitexact(run_ep(mt, d), ref_ep(d), "EP b=64 tp=8 P=4096 K=8")


def test_ep_bf16_route_weights(mt):
    d = synth.config(2)
    d["w"] = d["w"].to(torch.bfloat16)
    assert_bitexact(run_ep(mt, d), ref_ep(d), "EP bf16 weights")


@pytest.mark.parametrize("kw", [
    dict(b=1, tp=1, P=8, K=1, num_experts=1),             # smallest
    dict(b=5, tp=3, P=264, K=3, num_experts=9),           # ragged last chunk
    dict(b=7, tp=4, P=1000, K=5, num_experts=16),         # P not a multiple of 256
    dict(b=3, tp=32, P=512, K=32, num_experts=64),        # widest slots and routes
    dict(b=2, tp=8, P=32768, K=8, num_experts=64),        # widest row
    dict(b=130, tp=2, P=2048, K=8, num_experts=32),       # many tokens
])
def test_ep_shapes(mt, kw):
    d = synth.ep_finalize_inputs(0xE9 + kw["P"], **kw)
    assert_bitexact(run_ep(mt, d), ref_ep(d), f"EP {kw}")


def test_ep_non_local_and_out_of_range_indices(mt):
    d = synth.config(2, b=16)
    idx = d["idx"].clone()
    idx[:, 3, :] = -1                       # token 3: nothing local anywhere
    idx[2, 5, :] = d["rows_per_slot"] + 3    # out of range on the high side
    idx[0, 6, :] = -100
    d["idx"] = idx
    out = run_ep(mt, d)
    assert_bitexact(out, ref_ep(d), "EP non-local")
    assert np.all(bits(out)[3] == 0)


def test_ep_many_local_routes_per_slot(mt):
    # every route of every token local to every slot: tp * K = 64 rows per token
    b, tp, K, P, R = 4, 8, 8, 1024, 16
    rows = synth.bf16(synth.normal(77, 1, tp * R * P), (tp, R, P))
    idx = torch.from_numpy((synth.u64(77, 2, tp * b * K) % R).astype(np.int32).reshape(tp, b, K))
    d = dict(rows=rows, rows_per_slot=R, idx=idx, w=synth.softmax_weights(77, 3, b, K),
             gamma=synth.bf16(synth.normal(77, 4, P, std=0.1), (P,)), gain_center=1.0, eps=1e-6,
             weight_before_norm=True, b=b, tp=tp, K=K, P=P)
    assert_bitexact(run_ep(mt, d), ref_ep(d), "EP 64 local rows")


@pytest.mark.parametrize("regs", ["0", "1"])
def test_ep_both_kernels(mt, pin, regs):
    # the register-resident EP kernel (default) and the route-parallel one
    # (kernel form 2) on the decode shape and on one token with more
    # local routes than a pass holds
    pin(mt.FORM_EP, 1 if regs == "1" else 2)
    d = synth.config(2, weight_before_norm=False)
    assert_bitexact(run_ep(mt, d), ref_ep(d), f"EP b=64 kernel regs={regs}")
    d = synth.ep_finalize_inputs(0xE11, b=9, tp=4, P=2048, K=24, num_experts=24)
    assert_bitexact(run_ep(mt, d), ref_ep(d), f"EP K=24 kernel regs={regs}")


def test_ep_b_zero_leaves_out_untouched(mt):
    d = synth.config(1)
    out = torch.full((4, 512), 3.0, dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_ep_finalize(d["rows"].to(DEV), d["idx"][:, :0].contiguous().to(DEV), d["w"][:0].contiguous().to(DEV),
                            d["gamma"].to(DEV), out[:0])
    torch.cuda.synchronize()
    assert bool((out.float() == 3.0).all())


def _const_ep(weights_per_slot, P=256, row_value=1.0, gamma=0.0, gc=1.0, eps=0.0, wbn=True):
    tp = len(weights_per_slot)
    K = sum(len(ws) for ws in weights_per_slot)
    R = max(1, max(len(ws) for ws in weights_per_slot))
    idx = np.full((tp, 1, K), -1, dtype=np.int32)
    w = np.zeros((1, K), dtype=np.float32)
    k = 0
    for s, ws in enumerate(weights_per_slot):
        for r, wv in enumerate(ws):
            idx[s, 0, k] = r
            w[0, k] = wv
            k += 1
    return dict(rows=torch.full((tp, R, P), row_value).to(torch.bfloat16), rows_per_slot=R,
                idx=torch.from_numpy(idx), w=torch.from_numpy(w), gamma=torch.full((P,), gamma).to(torch.bfloat16),
                gain_center=gc, eps=eps, weight_before_norm=wbn, b=1, tp=tp, K=K, P=P)


@pytest.mark.parametrize("case,expect", [
    (dict(weights_per_slot=[[1.0 + 2.0 ** -8 + 2.0 ** -20], [2.0 ** -8]]), 1.015625),   # per-slot rounding
    (dict(weights_per_slot=[[1.0], [2.0 ** -8], [2.0 ** -24], [2.0 ** -24]]), 1.0),       # slot order
    (dict(weights_per_slot=[[1.0 + 2.0 ** -8, 2.0 ** -24, 2.0 ** -24]]), 1.0),            # route order
    (dict(weights_per_slot=[[1.0]], row_value=1.75 * 2.0 ** -75, gamma=1.625 * 2.0 ** -73, gc=0.0,
          eps=2.0 ** -100, wbn=True), 1.5 * 2.0 ** -97),                                  # subnormals kept,
    (dict(weights_per_slot=[[1.0]], row_value=1.75 * 2.0 ** -75, gamma=1.625 * 2.0 ** -73, gc=0.0,
          eps=2.0 ** -100, wbn=False), 1.421875 * 2.0 ** -97),                            # product order
])
def test_ep_crafted_rounding_cases(mt, case, expect):
    # the oracle pins' hand-derived cases, on the GPU
    d = _const_ep(**case)
    out = run_ep(mt, d)
    assert bool((out.float().cpu() == expect).all()), out.float().cpu()[0, :4]


@pytest.mark.parametrize("pattern", ["lane", "butterfly", "chunks"])
def test_ep_sum_of_squares_tree(mt, pattern):
    # one route, w = 1, gains 1, eps 0: out = bf16(x / sqrt(ss / P)).  The rows
    # are the oracle pins' tree cases, whose ss differ by tree shape; the GPU
    # must give the oracle's bits for P = 4096 split over a cluster.
    P = 4096
    v = torch.zeros(P)
    if pattern == "lane":
        v[0], v[1:8] = 4096.0, 1.0
    elif pattern == "butterfly":
        v[0], v[8:256:8] = 4096.0, 1.0
    else:
        v[0], v[256::256] = 4096.0, 1.0
    d = _const_ep([[1.0]], P=P)
    d["rows"] = v.to(torch.bfloat16).reshape(1, 1, P)
    assert_bitexact(run_ep(mt, d), ref_ep(d), f"SS tree {pattern}")


# ------------------------------------------------------------------ expert-TP finalize

def run_tp(mt, d, **kw):
    a = dict(d)
    a.update(kw)
    out = torch.full((a["b"], a["P"]), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_tp_finalize(a["partials"].to(DEV), a["idx"].to(DEV), a["w"].to(DEV), a["gamma"].to(DEV), out,
                            gain_center=a["gain_center"], eps=a["eps"], weight_before_norm=a["weight_before_norm"])
    torch.cuda.synchronize()
    return out


def ref_tp(d, **kw):
    a = dict(d)
    a.update(kw)
    return oracle.tp_finalize(a["partials"], a["num_rows"], a["idx"], a["w"], a["gamma"], a["gain_center"],
                              a["eps"], a["weight_before_norm"], a["b"], a["tp"], a["K"], a["P"])


@pytest.mark.parametrize("wbn", [True, False])
def test_tp_decode_full(mt, wbn):
    d = synth.config(3, weight_before_norm=wbn)
    assert_bitexact(run_tp(mt, d), ref_tp(d), "TP b=128 tp=8 P=4096 K=8")


def test_tp_bf16_weights_and_bad_indices(mt):
    d = synth.config(3, b=32)
    d["w"] = d["w"].to(torch.bfloat16)
    idx = d["idx"].clone()
    idx[4, 2] = -1
    idx[9, :] = d["num_rows"]
    d["idx"] = idx
    out = run_tp(mt, d)
    assert_bitexact(out, ref_tp(d), "TP bf16 weights, bad indices")
    assert np.all(bits(out)[9] == 0)


@pytest.mark.parametrize("kw", [
    dict(b=1, tp=1, P=8, K=1), dict(b=9, tp=3, P=264, K=5), dict(b=4, tp=32, P=512, K=32),
    dict(b=3, tp=2, P=32768, K=2), dict(b=300, tp=2, P=768, K=3),
])
def test_tp_shapes(mt, kw):
    d = synth.tp_finalize_inputs(0x7B + kw["P"], num_experts=64, **kw)
    assert_bitexact(run_tp(mt, d), ref_tp(d), f"TP {kw}")


@pytest.mark.parametrize("staged", ["0", "1"])
@pytest.mark.parametrize("b", [3, 64])
def test_tp_both_kernels(mt, pin, staged, b):
    # the staged kernel (chosen from b * K >= 512) and the route-parallel one
    # (chosen below), each forced on a batch the other would take
    pin(mt.FORM_TP, 1 if staged == "1" else 2)
    d = synth.config(3, b=b, weight_before_norm=(b == 3))
    assert_bitexact(run_tp(mt, d), ref_tp(d), f"TP b={b} staged={staged}")


@pytest.mark.parametrize("kind", ["ep", "tp_staged", "tp_route_parallel"])
def test_finalize_flags_call_matches_plain_call(mt, pin, kind):
    # the calls with MOE_TAIL_INPUTS_READY give the plain calls' bits
    if kind == "ep":
        d = synth.config(2)
        plain = run_ep(mt, d)
        out = torch.full_like(plain, float("nan"))
        mt.moe_tail_ep_finalize_flags(d["rows"].to(DEV), d["idx"].to(DEV), d["w"].to(DEV), d["gamma"].to(DEV), out,
                                      gain_center=d["gain_center"], eps=d["eps"],
                                      weight_before_norm=d["weight_before_norm"], inputs_ready=True)
        ref = ref_ep(d)
    else:
        pin(mt.FORM_TP, 1 if kind == "tp_staged" else 2)
        d = synth.config(3, b=64)
        plain = run_tp(mt, d)
        out = torch.full_like(plain, float("nan"))
        mt.moe_tail_tp_finalize_flags(d["partials"].to(DEV), d["idx"].to(DEV), d["w"].to(DEV), d["gamma"].to(DEV),
                                      out, gain_center=d["gain_center"], eps=d["eps"],
                                      weight_before_norm=d["weight_before_norm"], inputs_ready=True)
        ref = ref_tp(d)
    torch.cuda.synchronize()
    assert_bitexact(out, plain, f"{kind} flags call vs plain call")
    assert_bitexact(out, ref, f"{kind} flags call vs oracle")
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.parametrize("staged", ["0", "1"])
def test_tp_flags_inputs_ready_waits_before_writing_out(mt, pin, staged):
    # on one stream: TP(Q1) -> X; TP reading X as its partials -> Y; then TP with
    # inputs_ready from Q3 into X.  The last call may start while the second
    # still reads X, so it writes X only after that call ends: Y is the
    # finalize of TP(Q1), X that of Q3.
    pin(mt.FORM_TP, 1 if staged == "1" else 2)
    b, tp, K, P = 64, 8, 8, 4096
    d1 = synth.tp_finalize_inputs(0xC1, b=b, tp=tp, P=P, K=K)
    d3 = synth.tp_finalize_inputs(0xC3, b=b, tp=tp, P=P, K=K)
    b2, K2 = 16, 4
    idx2 = torch.from_numpy((synth.u64(0xC2, 1, b2 * K2) % b).astype(np.int32).reshape(b2, K2))
    w2 = synth.softmax_weights(0xC2, 2, b2, K2)
    x1_ref = ref_tp(d1)
    d2 = dict(partials=x1_ref.reshape(1, b, P), num_rows=b, idx=idx2, w=w2, gamma=d1["gamma"], gain_center=1.0,
              eps=1e-6, weight_before_norm=True, b=b2, tp=1, K=K2, P=P)
    y_ref = ref_tp(d2)
    x3_ref = ref_tp(d3)
    X = torch.empty((b, P), dtype=torch.bfloat16, device=DEV)
    Y = torch.full((b2, P), float("nan"), dtype=torch.bfloat16, device=DEV)
    q1, q3 = d1["partials"].to(DEV), d3["partials"].to(DEV)
    idx1, idx3, i2 = d1["idx"].to(DEV), d3["idx"].to(DEV), idx2.to(DEV)
    w1, w3, ww2, gam = d1["w"].to(DEV), d3["w"].to(DEV), w2.to(DEV), d1["gamma"].to(DEV)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    mt.moe_tail_tp_finalize(q1, idx1, w1, gam, X, stream=st)
    mt.moe_tail_tp_finalize(X.view(1, b, P), i2, ww2, gam, Y, stream=st)
    mt.moe_tail_tp_finalize_flags(q3, idx3, w3, d3["gamma"].to(DEV), X, inputs_ready=True, stream=st)
    torch.cuda.synchronize()
    assert_bitexact(Y, y_ref, "the call reading X saw the first X")
    assert_bitexact(X, x3_ref, "X is the last call's output")
    assert mt.moe_tail_take_device_error() == 0


# ------------------------------------------------------------------ latent tail

def run_latent(mt, d):
    b, L, H = d["b"], d["L"], d["H"]
    ws = torch.full((mt.moe_tail_workspace_bytes(0, b, L),), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    sh = None if d["shared"] is None else d["shared"].to(DEV)
    mt.moe_tail_latent_up(d["latent"].to(DEV), d["gamma"].to(DEV), d["w_up"].to(DEV), sh, out, ws, eps=d["eps"])
    torch.cuda.synchronize()
    y = ws[: b * L * 2].view(torch.bfloat16).view(b, L)
    return y, out


def test_latent_up_full(mt):
    d = synth.config(4)
    y_ref, out_ref = oracle.latent_tail(d["latent"], d["gamma"], d["eps"], d["w_up"], d["shared"], d["tp_s"],
                                        d["b"], d["tp"], d["L"], d["H"])
    y, out = run_latent(mt, d)
    assert_bitexact(y, y_ref, "latent y b=16")
    assert_gemm_close(out, out_ref, "latent out b=16 [7168]")


@pytest.mark.parametrize("kw", [
    dict(b=1, tp=1, tp_s=0, L=3584, H=7168),
    dict(b=5, tp=3, tp_s=2, L=264, H=200),        # ragged K tail and M tail
    dict(b=33, tp=8, tp_s=8, L=1024, H=384),       # N tile 64
    dict(b=64, tp=8, tp_s=8, L=3584, H=1024),      # the shared-expert batch
    dict(b=100, tp=2, tp_s=1, L=512, H=256),       # N tile 128
    dict(b=130, tp=2, tp_s=1, L=512, H=256),       # two token tiles
])
def test_latent_up_shapes(mt, kw):
    d = synth.latent_up_inputs(0x1A7 + kw["b"], **kw)
    y_ref, out_ref = oracle.latent_tail(d["latent"], d["gamma"], d["eps"], d["w_up"], d["shared"], d["tp_s"],
                                        d["b"], d["tp"], d["L"], d["H"])
    y, out = run_latent(mt, d)
    assert_bitexact(y, y_ref, f"latent y {kw}")
    assert_gemm_close(out, out_ref, f"latent out {kw}")


def test_latent_up_identity_weight(mt):
    # W_up = [I; 0]: out[:, :L] = bf16(y + sum shared) exactly equals the oracle
    b, tp, L, H = 4, 2, 256, 512
    d = synth.latent_up_inputs(0x1D, b=b, tp=tp, L=L, H=H, tp_s=0)
    w = torch.zeros((H, L))
    w[:L, :L] = torch.eye(L)
    d["w_up"] = w.to(torch.bfloat16)
    y, out = run_latent(mt, d)
    assert_bitexact(out[:, :L], y, "identity up-projection")
    assert np.all(bits(out)[:, L:] == 0)


@pytest.mark.parametrize("kw", [
    dict(b=16, tp=8, tp_s=8, L=3584, H=7168),
    dict(b=5, tp=3, tp_s=2, L=264, H=200),
    dict(b=64, tp=8, tp_s=9, L=3584, H=1024),
    dict(b=3, tp=1, tp_s=0, L=512, H=256),
])
@pytest.mark.parametrize("static", [False, True])
def test_latent_steps_as_separate_calls(mt, kw, static):
    # moe_tail_latent_norm then moe_tail_up_project, on two streams joined by an
    # event as a scheduler would run them: y bit-exact against the oracle's
    # norm, out within the GEMM bound of the oracle's up-projection of that y,
    # and both bit-identical to the one-call latent tail
    d = synth.latent_up_inputs(0x5E9 + kw["b"] + kw["tp_s"], **kw)
    b, L, H = d["b"], d["L"], d["H"]
    y_ref, out_ref = oracle.latent_tail(d["latent"], d["gamma"], d["eps"], d["w_up"], d["shared"], d["tp_s"],
                                        b, d["tp"], L, H)
    y = torch.full((b, L), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    sh = None if d["shared"] is None else d["shared"].to(DEV)
    lat, gam, w = d["latent"].to(DEV), d["gamma"].to(DEV), d["w_up"].to(DEV)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    ready = torch.cuda.Event()
    mt.moe_tail_latent_norm(lat, gam, y, eps=d["eps"], inputs_ready=static, stream=s1)
    ready.record(s1)
    s2.wait_event(ready)
    mt.moe_tail_up_project(y, w, sh, out, weights_static=static, stream=s2)
    torch.cuda.synchronize()
    assert_bitexact(y, y_ref, f"latent norm {kw}")
    assert_gemm_close(out, out_ref, f"up-projection {kw}")
    y1, out1 = run_latent(mt, d)
    assert np.array_equal(bits(y1), bits(y)) and np.array_equal(bits(out1), bits(out))
    assert mt.moe_tail_take_device_error() == 0


def test_latent_norm_inputs_ready_waits_before_writing_y(mt):
    # norm(A) -> up-projection reading y -> norm(B) with inputs_ready on one
    # stream: the second norm may start while the GEMM still reads y, so it
    # must not write y before the GEMM is done; outA must be A's up-projection
    kw = dict(b=64, tp=8, tp_s=8, L=3584, H=7168)
    A = synth.latent_up_inputs(0xA11, **kw)
    B = synth.latent_up_inputs(0xB22, **kw)
    _, out_ref = oracle.latent_tail(A["latent"], A["gamma"], A["eps"], A["w_up"], A["shared"], A["tp_s"],
                                    64, 8, 3584, 7168)
    yB_ref = oracle.latent_norm(B["latent"], B["gamma"], B["eps"], 64, 8, 3584)
    y = torch.empty((64, 3584), dtype=torch.bfloat16, device=DEV)
    out = torch.full((64, 7168), float("nan"), dtype=torch.bfloat16, device=DEV)
    latA, latB, gam = A["latent"].to(DEV), B["latent"].to(DEV), A["gamma"].to(DEV)
    gamB, w, sh = B["gamma"].to(DEV), A["w_up"].to(DEV), A["shared"].to(DEV)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    mt.moe_tail_latent_norm(latA, gam, y, eps=A["eps"], stream=st)
    mt.moe_tail_up_project(y, w, sh, out, weights_static=True, stream=st)
    mt.moe_tail_latent_norm(latB, gamB, y, eps=B["eps"], inputs_ready=True, stream=st)
    torch.cuda.synchronize()
    assert_gemm_close(out, out_ref, "up-projection of the first y")
    assert_bitexact(y, yB_ref, "second y")
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.parametrize("kw", [
    dict(b=1, tp=8, tp_s=9, L=3584, H=7168),     # the decode shape: K split over 8-CTA clusters, 3 CTAs per SM
    dict(b=16, tp=8, tp_s=8, L=3584, H=7168),
    dict(b=5, tp=3, tp_s=0, L=1000, H=520),      # split 8, ragged last chunk, M tail
    dict(b=17, tp=2, tp_s=1, L=8192, H=264),     # N tile 32, 32 chunks, two ring stages
    dict(b=32, tp=9, tp_s=2, L=256, H=136),      # one chunk shared by all four CTAs of a cluster
    dict(b=8, tp=32, tp_s=32, L=8, H=8),         # one K block, no cluster
    dict(b=12, tp=1, tp_s=0, L=8200, H=64),      # 33 chunks: the two-kernel form
])
@pytest.mark.parametrize("flags", [0, 1, 2, 3])
def test_latent_one_kernel_matches_split_calls(mt, pin, kw, flags):
    # moe_tail_latent_up_flags with its one-kernel form taken wherever it fits
    # (up to 32 tokens): y and out bit for bit those of moe_tail_latent_norm +
    # moe_tail_up_project, y bit-exact against the oracle's norm and out within
    # the GEMM bound of the oracle's up-projection
    d = synth.latent_up_inputs(0xF05E + kw["b"] + kw["L"], **kw)
    b, L, H = d["b"], d["L"], d["H"]
    lat, gam, w = d["latent"].to(DEV), d["gamma"].to(DEV), d["w_up"].to(DEV)
    sh = None if d["shared"] is None else d["shared"].to(DEV)
    y1 = torch.full((b, L), float("nan"), dtype=torch.bfloat16, device=DEV)
    out1 = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_latent_norm(lat, gam, y1, eps=d["eps"])
    mt.moe_tail_up_project(y1, w, sh, out1)
    pin(mt.FORM_LATENT, 1)
    y2 = torch.full((b, L), float("nan"), dtype=torch.bfloat16, device=DEV)
    out2 = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_latent_up_flags(lat, gam, w, sh, out2, y2, eps=d["eps"], inputs_ready=bool(flags & 2),
                                weights_static=bool(flags & 1))
    torch.cuda.synchronize()
    assert mt.moe_tail_take_device_error() == 0
    assert np.array_equal(bits(y2), bits(y1)), f"y one kernel vs split {kw}"
    assert np.array_equal(bits(out2), bits(out1)), f"out one kernel vs split {kw}"
    y_ref, out_ref = oracle.latent_tail(d["latent"], d["gamma"], d["eps"], d["w_up"], d["shared"], d["tp_s"],
                                        b, d["tp"], L, H)
    assert_bitexact(y2, y_ref, f"latent y {kw}")
    assert_gemm_close(out2, out_ref, f"latent out {kw}")


@pytest.mark.parametrize("choice", ["0", "1"])
def test_latent_up_and_noalloc_take_either_form(mt, pin, choice):
    # moe_tail_latent_up and the workspace-free call at b = 4, with the one-kernel
    # form switched off and on: the same bits either way
    pin(mt.FORM_LATENT, 1 if choice == "1" else 2)
    d = synth.latent_up_inputs(0x0F4, b=4, tp=8, tp_s=9, L=3584, H=7168)
    y, out = run_latent(mt, d)
    out_na = torch.full((4, 7168), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_latent_up_noalloc(d["latent"].to(DEV), d["gamma"].to(DEV), d["w_up"].to(DEV),
                                  d["shared"].to(DEV), out_na, eps=d["eps"])
    torch.cuda.synchronize()
    y_ref, out_ref = oracle.latent_tail(d["latent"], d["gamma"], d["eps"], d["w_up"], d["shared"], 9, 4, 8, 3584,
                                        7168)
    assert_bitexact(y, y_ref, "latent y b=4")
    assert_gemm_close(out, out_ref, "latent out b=4")
    assert np.array_equal(bits(out_na), bits(out))
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.parametrize("one_kernel", ["0", "1"])
def test_latent_up_flags_inputs_ready_waits_before_writing_y(mt, pin, one_kernel):
    # norm(A) -> up-projection reading y -> the flags call for B with
    # inputs_ready into the same y, on one stream (both forms): B's first
    # kernel may start while the up-projection still reads y, so y is written
    # only after that kernel ends; outA must be A's up-projection and y, outB B's
    pin(mt.FORM_LATENT, 1 if one_kernel == "1" else 2)
    kw = dict(b=16, tp=8, tp_s=8, L=3584, H=7168)
    A = synth.latent_up_inputs(0xA13, **kw)
    B = synth.latent_up_inputs(0xB24, **kw)
    yA_ref, outA_ref = oracle.latent_tail(A["latent"], A["gamma"], A["eps"], A["w_up"], A["shared"], 8, 16, 8,
                                          3584, 7168)
    yB_ref, outB_ref = oracle.latent_tail(B["latent"], B["gamma"], B["eps"], A["w_up"], B["shared"], 8, 16, 8,
                                          3584, 7168)
    y = torch.empty((16, 3584), dtype=torch.bfloat16, device=DEV)
    outA = torch.full((16, 7168), float("nan"), dtype=torch.bfloat16, device=DEV)
    outB = torch.full((16, 7168), float("nan"), dtype=torch.bfloat16, device=DEV)
    w = A["w_up"].to(DEV)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    mt.moe_tail_latent_norm(A["latent"].to(DEV), A["gamma"].to(DEV), y, eps=A["eps"], stream=st)
    mt.moe_tail_up_project(y, w, A["shared"].to(DEV), outA, weights_static=True, stream=st)
    mt.moe_tail_latent_up_flags(B["latent"].to(DEV), B["gamma"].to(DEV), w, B["shared"].to(DEV), outB, y,
                                eps=B["eps"], inputs_ready=True, weights_static=True, stream=st)
    torch.cuda.synchronize()
    assert_gemm_close(outA, outA_ref, "up-projection of the first y")
    assert_bitexact(y, yB_ref, "second y")
    assert_gemm_close(outB, outB_ref, "latent tail of B")
    assert mt.moe_tail_take_device_error() == 0


# ------------------------------------------------------------------ the header's limits

@pytest.mark.parametrize("case", ["ep_b_max", "tp_b_max", "ep_all_max", "tp_all_max", "latent_b_max",
                                  "latent_L_max"])
def test_maximum_sizes(mt, case):
    # b = 65535 (one CTA row of the finalize grids per token: the grid's y
    # limit), tp = K = 32 with P = 32768 together, and the latent tail at its
    # largest b and L; finalize outputs and y bit-exact, out within the GEMM bound
    if case == "ep_b_max":
        d = synth.ep_finalize_inputs(0x3A1, b=65535, tp=1, P=8, K=1, num_experts=1)
        assert_bitexact(run_ep(mt, d), ref_ep(d), case)
    elif case == "tp_b_max":
        d = synth.tp_finalize_inputs(0x3A2, b=65535, tp=1, P=8, K=1, num_experts=1)
        assert_bitexact(run_tp(mt, d), ref_tp(d), case)
    elif case == "ep_all_max":
        d = synth.ep_finalize_inputs(0x3A3, b=2, tp=32, P=32768, K=32, num_experts=64)
        assert_bitexact(run_ep(mt, d), ref_ep(d), case)
    elif case == "tp_all_max":
        d = synth.tp_finalize_inputs(0x3A4, b=2, tp=32, P=32768, K=32, num_experts=64)
        assert_bitexact(run_tp(mt, d), ref_tp(d), case)
    else:
        kw = dict(b=65535, tp=1, tp_s=1, L=8, H=8) if case == "latent_b_max" else \
            dict(b=2, tp=2, tp_s=32, L=32768, H=64)
        d = synth.latent_up_inputs(0x3A5 + kw["L"], **kw)
        y_ref, out_ref = oracle.latent_tail(d["latent"], d["gamma"], d["eps"], d["w_up"], d["shared"], d["tp_s"],
                                            d["b"], d["tp"], d["L"], d["H"])
        y, out = run_latent(mt, d)
        assert_bitexact(y, y_ref, f"{case} y")
        assert_gemm_close(out, out_ref, f"{case} out")
    assert mt.moe_tail_take_device_error() == 0


@pytest.mark.parametrize("ctas", [2, 0])
def test_down_projections_at_the_token_limit(mt, ctas):
    # b = 65535 (512 token tiles of 128): the persistent down projection walks
    # 512 tiles over 2 CTAs (each accumulator reused 128 times) or over one CTA
    # per SM, and the down + up kernel runs 512 token tiles of its clusters;
    # d against the oracle on sampled tokens and against moe_shared_down on
    # every element, out against the oracle with the GPU's d as a shared slot
    b, H, I, L = 65535, 8, 64, 64
    h = synth.bf16(synth.normal(0x3B0, 1, b * I, std=0.5), (b, I))
    wd = synth.bf16(synth.normal(0x3B0, 2, H * I, std=0.05), (H, I))
    y = synth.bf16(synth.normal(0x3B0, 3, b * L, std=0.5), (b, L))
    wu = synth.bf16(synth.normal(0x3B0, 4, H * L, std=0.05), (H, L))
    hg, wdg = h.to(DEV), wd.to(DEV)
    d = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_shared_down_persistent(hg, wdg, d, accumulate=False, ctas=ctas)
    d2 = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_shared_down(hg, wdg, d2, accumulate=False)
    out = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    d3 = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_up_project_shared_down(y.to(DEV), wu.to(DEV), None, hg, wdg, out, d3)
    torch.cuda.synchronize()
    assert mt.moe_tail_take_device_error() == 0
    d_c, d3_c, out_c = d.cpu(), d3.cpu(), out.cpu()
    for t in (0, 127, 128, 40000, b - 1):
        sl = slice(t, t + 1)
        d_ref = oracle.shared_down(h[sl], wd, 1, H, I, accumulate=False)
        assert_gemm_close(d_c[sl], d_ref, f"persistent d token {t}")
        assert_gemm_close(d3_c[sl], d_ref, f"down + up d token {t}")
        assert_gemm_close(out_c[sl], oracle.latent_up(y[sl], wu, d3_c[None, sl].contiguous(), 1, 1, L, H),
                          f"down + up out token {t}")
    assert_gemm_close(d_c, d2.cpu(), "persistent d vs the split-K call, every element")


# ------------------------------------------------------------------ shared expert
#
# gate and up are FP32 sums whose order the pages leave open, so bf16(gate),
# bf16(up) and h may differ from the double oracle by an ulp in a few elements
# per token: several h are correct.  The unique parts are compared with the
# oracle on oracle-only inputs -- h itself, and the down stage on an h both
# sides compute exactly -- and the GPU's d is checked to be a valid down
# projection of the GPU's own h.

def run_shared(mt, s, out_in, accumulate=True):
    b, H, I = s["b"], s["H"], s["I"]
    ws = torch.full((mt.moe_tail_workspace_bytes(1, b, I),), 0xFF, dtype=torch.uint8, device=DEV)
    out = out_in.to(DEV).clone()
    mt.moe_shared_expert(s["x"].to(DEV), s["w_gate"].to(DEV), s["w_up"].to(DEV), s["w_down"].to(DEV), out, ws,
                         accumulate=accumulate)
    torch.cuda.synchronize()
    return ws[: b * I * 2].view(torch.bfloat16).view(b, I).cpu(), out.cpu()


def check_shared(mt, s, out_in, tokens=None, what=""):
    b, H, I = s["b"], s["H"], s["I"]
    h, out = run_shared(mt, s, out_in, accumulate=True)
    h2, d = run_shared(mt, s, torch.zeros((b, H), dtype=torch.bfloat16), accumulate=False)
    assert_bitexact(h2, h, f"{what} h is deterministic")
    for t in (range(b) if tokens is None else tokens):
        sl = slice(t, t + 1)
        h_ref, _ = oracle.shared_expert(s["x"][sl], s["w_gate"], s["w_up"], s["w_down"], 1, H, I, accumulate=False)
        assert_gemm_close(h[sl], h_ref, f"{what} h token {t}")
        d_valid = oracle.shared_down(h[sl], s["w_down"], 1, H, I, accumulate=False)
        assert_gemm_close(d[sl], d_valid, f"{what} d token {t} (down projection of the GPU's h)")
    assert_accumulated_exact(out, out_in, d, f"{what} out, every token")


@pytest.mark.parametrize("kw", [
    dict(b=1, H=512, I=256), dict(b=3, H=520, I=200), dict(b=17, H=1024, I=768), dict(b=64, H=768, I=512),
    dict(b=100, H=256, I=384), dict(b=129, H=256, I=128),
])
def test_shared_expert_shapes(mt, kw):
    s = synth.shared_expert_inputs(0x5E + kw["b"], **kw)
    out_in = synth.bf16(synth.normal(0x5E, 99, kw["b"] * kw["H"]), (kw["b"], kw["H"]))
    check_shared(mt, s, out_in, what=str(kw))


def test_shared_expert_full_size_b128_sampled_tokens(mt):
    # H = 7168, I = 6144 at b = 128: 128-token tiles, gate/up's 4-way K split
    # with 2-stage rings and the down projection's 3-stage rings; the oracle
    # recomputes 4 tokens (both ends of the tile and its middle), and every
    # token's accumulated output is checked bit for bit against the GPU's d
    s = synth.shared_expert_inputs(0x5EED0128, b=128, H=7168, I=6144)
    out_in = synth.bf16(synth.normal(0x5E, 128, 128 * 7168), (128, 7168))
    check_shared(mt, s, out_in, tokens=(0, 63, 64, 127), what="b=128 H=7168 I=6144")


def test_shared_expert_full_size_sampled_tokens(mt):
    # the full decode layer: latent tail at b = 64, then the shared expert
    # added into its output; the oracle recomputes 6 sampled tokens
    b = 64
    lat = synth.latent_up_inputs(0x5EED0004, b=b)
    s = synth.config(5)
    _, out = run_latent(mt, lat)
    latent_out = out.cpu().clone()
    for t in (0, 1, 17, 31, 50, 63):
        _, lat_ref = oracle.latent_tail(lat["latent"][:, t:t + 1].contiguous(), lat["gamma"], lat["eps"],
                                        lat["w_up"], lat["shared"][:, t:t + 1].contiguous(), 8, 1, 8, 3584, 7168)
        assert_gemm_close(latent_out[t:t + 1], lat_ref, f"latent out token {t}")
    check_shared(mt, s, latent_out, tokens=(0, 1, 17, 31, 50, 63), what="b=64 H=7168 I=6144")


def test_shared_expert_down_stage_full_size_exact_h(mt):
    # x is one-hot (column c_t for token t) and W_gate is 32 on those columns,
    # so gate = 32 and up = W_up[:, c_t] exactly in FP32 and in double, and
    # silu(32) * up = 32 * up on both sides (exp(-32) vanishes next to 1 in
    # FP32 and moves the double product by far less than half a BF16 ulp):
    # h is one exact value.  The down projection is then compared with the
    # oracle's at the GEMM tolerance, at full size.
    b, H, I = 64, 7168, 6144
    s = synth.config(5, with_weights=False)
    cols = [(t * 97 + 5) % H for t in range(b)]
    x = torch.zeros((b, H))
    wg = torch.zeros((I, H))
    for t, c in enumerate(cols):
        x[t, c] = 1.0
        wg[:, c] = 32.0
    s["x"], s["w_gate"] = x.to(torch.bfloat16), wg.to(torch.bfloat16)
    s["w_up"] = synth.bf16(synth.normal(0x5EED0005, 22, I * H, std=0.02), (I, H))
    s["w_down"] = synth.bf16(synth.normal(0x5EED0005, 23, H * I, std=0.02), (H, I))
    out_in = synth.bf16(synth.normal(0x5EED0005, 30, b * H), (b, H))
    h, out = run_shared(mt, s, out_in, accumulate=True)
    _, d = run_shared(mt, s, torch.zeros((b, H), dtype=torch.bfloat16), accumulate=False)
    for t in (0, 9, 33, 63):
        sl = slice(t, t + 1)
        h_ref, d_ref = oracle.shared_expert(s["x"][sl], s["w_gate"], s["w_up"], s["w_down"], 1, H, I,
                                            accumulate=False)
        assert_bitexact(h[sl], h_ref, f"exact h token {t}")
        assert_gemm_close(d[sl], d_ref, f"down projection token {t}")
    assert_accumulated_exact(out, out_in, d, "accumulated output, every token")


@pytest.mark.parametrize("kw", [dict(b=64, H=7168, I=6144), dict(b=5, H=264, I=200), dict(b=130, H=256, I=128)])
@pytest.mark.parametrize("static,ready", [(False, False), (True, False), (True, True), (False, True)])
def test_shared_expert_as_two_calls(mt, kw, static, ready):
    # moe_shared_gate_up (with or without the promises) then moe_shared_down on
    # two streams joined by an event, with the latent-tail-like addend in out:
    # bit-identical to the one call
    s = synth.shared_expert_inputs(0x2C + kw["b"], **kw)
    b, H, I = s["b"], s["H"], s["I"]
    out_in = synth.bf16(synth.normal(0x2C, 5, b * H), (b, H))
    h1, out1 = run_shared(mt, s, out_in, accumulate=True)
    x, wg, wu, wd = (s[k].to(DEV) for k in ("x", "w_gate", "w_up", "w_down"))
    h = torch.full((b, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = out_in.to(DEV).clone()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    mt.moe_shared_gate_up(x, wg, wu, h, weights_static=static, inputs_ready=ready, stream=s1)
    joined = torch.cuda.Event()
    joined.record(s1)
    s2.wait_event(joined)
    mt.moe_shared_down(h, wd, out, accumulate=True, weights_static=static, stream=s2)
    torch.cuda.synchronize()
    assert_bitexact(h, h1, f"h {kw}")
    assert_bitexact(out, out1, f"out {kw}")
    d = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_shared_down(h, wd, d, accumulate=False)
    torch.cuda.synchronize()
    t = min(3, b - 1)
    assert_gemm_close(d[t:t + 1], oracle.shared_down(h[t:t + 1].cpu(), s["w_down"], 1, H, I, accumulate=False),
                      f"d token {t} {kw}")
    assert mt.moe_tail_take_device_error() == 0


def test_gate_up_inputs_ready_waits_before_writing_h(mt):
    # on one stream: gate/up(x1) -> h; the down projection reading h -> d1;
    # gate/up(x2) with both promises -> h.  The last call may run its K loop
    # while the down projection still reads h, so it writes h only after that
    # call ends: d1 is the down projection of h(x1), h is h(x2) -- each bit for
    # bit the result of the same call made alone
    s1 = synth.shared_expert_inputs(0x6A1, b=64, H=7168, I=6144)
    s2 = synth.shared_expert_inputs(0x6A2, b=64, H=7168, I=6144)
    b, H, I = 64, 7168, 6144
    x1, x2 = s1["x"].to(DEV), s2["x"].to(DEV)
    wg, wu, wd = (s1[k].to(DEV) for k in ("w_gate", "w_up", "w_down"))
    h_a = torch.empty((b, I), dtype=torch.bfloat16, device=DEV)
    h_b = torch.empty((b, I), dtype=torch.bfloat16, device=DEV)
    d_ref = torch.empty((b, H), dtype=torch.bfloat16, device=DEV)
    mt.moe_shared_gate_up(x1, wg, wu, h_a)
    mt.moe_shared_gate_up(x2, wg, wu, h_b)
    mt.moe_shared_down(h_a, wd, d_ref, accumulate=False)
    torch.cuda.synchronize()
    h = torch.empty((b, I), dtype=torch.bfloat16, device=DEV)
    d1 = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    mt.moe_shared_gate_up(x1, wg, wu, h, stream=st)
    mt.moe_shared_down(h, wd, d1, accumulate=False, weights_static=True, stream=st)
    mt.moe_shared_gate_up(x2, wg, wu, h, weights_static=True, inputs_ready=True, stream=st)
    torch.cuda.synchronize()
    assert_bitexact(d1, d_ref, "the down projection saw the first h")
    assert_bitexact(h, h_b, "h is the last call's output")
    assert mt.moe_tail_take_device_error() == 0


def test_shared_expert_zero_input_leaves_out(mt):
    s = synth.shared_expert_inputs(3, b=5, H=256, I=128)
    s["x"] = torch.zeros_like(s["x"])
    out_in = synth.bf16(synth.normal(3, 9, 5 * 256), (5, 256))
    _, out = run_shared(mt, s, out_in)
    assert_bitexact(out, out_in, "x = 0")


def test_no_device_error_raised(mt):
    assert mt.moe_tail_take_device_error() == 0


# ------------------------------------------ the persistent down projection

@pytest.mark.parametrize("kw", [
    dict(b=64, H=7168, I=6144, ctas=0), dict(b=64, H=7168, I=6144, ctas=28),   # 56 tiles: 1 or 2 per CTA
    dict(b=1, H=7168, I=6144, ctas=14), dict(b=16, H=1024, I=768, ctas=3),      # 4 tiles per CTA
    dict(b=130, H=264, I=200, ctas=2),   # two token tiles, ragged M and K
    dict(b=37, H=136, I=136, ctas=1),    # one CTA walks every tile
    dict(b=5, H=520, I=1000, ctas=200),  # more CTAs asked for than there are tiles
])
def test_persistent_down(mt, kw):
    # d against the oracle's down projection of h (GEMM bound) on sampled tokens,
    # against moe_shared_down (K split over a cluster) on every element (the same
    # bits almost everywhere, within the GEMM bound), and the accumulating call
    # bit for bit bf16(out_in + d) given the GPU's d
    b, H, I, ctas = kw["b"], kw["H"], kw["I"], kw["ctas"]
    seed = 0xE0 + b + H
    h = synth.bf16(synth.normal(seed, 1, b * I, std=0.5), (b, I))
    wd = synth.bf16(synth.normal(seed, 2, H * I, std=0.02), (H, I))
    out_in = synth.bf16(synth.normal(seed, 3, b * H), (b, H))
    hg, wg = h.to(DEV), wd.to(DEV)
    d = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_shared_down_persistent(hg, wg, d, accumulate=False, ctas=ctas)
    d2 = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_shared_down(hg, wg, d2, accumulate=False)
    out = out_in.to(DEV)
    mt.moe_shared_down_persistent(hg, wg, out, accumulate=True, ctas=ctas, weights_static=True)
    torch.cuda.synchronize()
    assert mt.moe_tail_take_device_error() == 0
    d_c = d.cpu()
    for t in sorted({0, b // 2, b - 1}):
        sl = slice(t, t + 1)
        assert_gemm_close(d_c[sl], oracle.shared_down(h[sl], wd, 1, H, I, accumulate=False), f"d token {t} {kw}")
    same = bits(d) == bits(d2)
    assert same.mean() > 0.99, f"d differs from the split-K call in {1 - same.mean():.4f} of elements {kw}"
    assert_gemm_close(d_c, d2.cpu(), f"d vs the split-K call, every element {kw}")
    assert_accumulated_exact(out, out_in, d_c, f"accumulated out, every token {kw}")


# ------------------------------------------ up-projection + shared down projection in one kernel

@pytest.mark.parametrize("kw", [
    dict(b=64, L=3584, I=6144, H=7168, tp_s=8), dict(b=16, L=3584, I=6144, H=7168, tp_s=8),
    dict(b=1, L=3584, I=6144, H=7168, tp_s=0), dict(b=37, L=264, I=200, H=136, tp_s=3),
    dict(b=130, L=512, I=384, H=256, tp_s=1),
    # one K block each (a cluster of two, one rank per projection); ten down
    # blocks against one up block (five ranks of two down blocks, one rank for
    # the up-projection)
    dict(b=5, L=64, I=64, H=128, tp_s=2), dict(b=3, L=64, I=640, H=128, tp_s=1),
])
def test_up_project_shared_down(mt, kw):
    # out = bf16(u + (sum_s shared[s] + bf16(d))): d against the oracle's down
    # projection of h, out against the oracle's up-projection of y with the
    # GPU's bf16(d) as one more shared slot (GEMM bound), on sampled tokens;
    # and every element against the two-call form (moe_shared_down writing d
    # into a slot, then moe_tail_up_project), which sums d and u over other K
    # splits: the same bits almost everywhere, and within the GEMM bound
    # wherever the two d agree
    b, L, I, H, tp_s = kw["b"], kw["L"], kw["I"], kw["H"], kw["tp_s"]
    seed = 0xD0 + b + L
    y = synth.bf16(synth.normal(seed, 1, b * L, std=1.0), (b, L))
    w_up = synth.bf16(synth.normal(seed, 2, H * L, std=0.02), (H, L))
    h = synth.bf16(synth.normal(seed, 3, b * I, std=0.5), (b, I))
    w_down = synth.bf16(synth.normal(seed, 4, H * I, std=0.02), (H, I))
    shared = synth.bf16(synth.normal(seed, 5, tp_s * b * H, std=0.5), (tp_s, b, H)) if tp_s else None
    g = lambda t: None if t is None else t.to(DEV)
    out = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    d = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_up_project_shared_down(g(y), g(w_up), g(shared), g(h), g(w_down), out, d)
    # the two-call form
    slots = torch.empty((tp_s + 1, b, H), dtype=torch.bfloat16, device=DEV)
    if tp_s:
        slots[:tp_s].copy_(g(shared))
    mt.moe_shared_down(g(h), g(w_down), slots[tp_s], accumulate=False)
    out2 = torch.full((b, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mt.moe_tail_up_project(g(y), g(w_up), slots, out2)
    torch.cuda.synchronize()
    assert mt.moe_tail_take_device_error() == 0
    out_c, d_c = out.cpu(), d.cpu()
    for t in sorted({0, b // 2, b - 1}):
        sl = slice(t, t + 1)
        assert_gemm_close(d_c[sl], oracle.shared_down(h[sl], w_down, 1, H, I, accumulate=False), f"d token {t} {kw}")
        sh9 = torch.cat([shared[:, sl] if tp_s else torch.empty((0, 1, H), dtype=torch.bfloat16), d_c[None, sl]])
        ref = oracle.latent_up(y[sl], w_up, sh9.contiguous(), tp_s + 1, 1, L, H)
        assert_gemm_close(out_c[sl], ref, f"out token {t} {kw}")
    same_d = bits(d) == bits(slots[tp_s])
    assert same_d.mean() > 0.99, f"the two d differ in {1 - same_d.mean():.4f} of elements {kw}"
    same_out = bits(out) == bits(out2)
    assert same_out.mean() > 0.99, f"out differs from the two-call form in {1 - same_out.mean():.4f} of elements {kw}"
    mask = torch.from_numpy(same_d)  # where the two d agree, out differs only through u's K split
    assert_gemm_close(out_c[mask], out2.cpu()[mask], f"out vs the two-call form where d agrees {kw}")
