"""Pins of the CPU oracle to facts outside itself.

Each test fixes the oracle against something the pages or mathematics decide:
closed forms derived by hand (values written below, not recomputed), crafted
inputs whose result depends on the order of FP32 additions (each expected value
is derived in the test's comment), invariants the method states (b = 0 does
nothing, non-local routes contribute nothing, production order is irrelevant,
gains of one make weight_before_norm moot), the identity between the EP and
expert-TP formulas, library routines (torch's BF16 rounding, numpy matmul) on
the special cases that reduce to them, and brute-force double recomputation on
tiny inputs.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from moe_decode_tail_gb300 import synth


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.uint16)).view(np.int16)).view(torch.bfloat16)


def bf(values, shape=None) -> torch.Tensor:
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.reshape(shape) if shape is not None else t


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def ep_call(d, **kw):
    a = dict(d)
    a.update(kw)
    return oracle.ep_finalize(a["rows"], a["rows_per_slot"], a["idx"], a["w"], a["gamma"], a["gain_center"],
                              a["eps"], a["weight_before_norm"], a["b"], a["tp"], a["K"], a["P"])


def tp_call(d, **kw):
    a = dict(d)
    a.update(kw)
    return oracle.tp_finalize(a["partials"], a["num_rows"], a["idx"], a["w"], a["gamma"], a["gain_center"],
                              a["eps"], a["weight_before_norm"], a["b"], a["tp"], a["K"], a["P"])


def constant_ep(weights_per_slot, P=256, row_value=1.0, gamma=0.0, gc=1.0, eps=0.0, wbn=True):
    """One token; slot s holds one route row per entry of weights_per_slot[s],
    every row the constant row_value; route weights FP32 as given."""
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


# --------------------------------------------------------------------------- BF16

def test_bf16_from_f32_matches_torch_rounding():
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # ties, just-above/below ties, subnormals, zeros, infinities
    special = np.array([0x3F808000, 0x3F818000, 0x3F808001, 0x3F807FFF, 0x00008000, 0x00018000,
                        0x80000000, 0x00000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x00000001],
                       dtype=np.uint32)
    u = np.concatenate([u, special])
    f = u.view(np.float32)
    ref = bits(torch.from_numpy(f.copy()).to(torch.bfloat16))
    got = np.array([oracle.bf16_from_f32(float(x)) for x in f], dtype=np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x7F) != 0)


def _nearest_bf16_exact(d: float) -> int:
    """Brute force: the BF16 pattern nearest to d in exact rational arithmetic,
    ties to the even significand."""
    f32 = np.float32(d)
    base = int(np.array([f32], dtype=np.float32).view(np.uint32)[0] >> 16)
    target = Fraction(d)
    best = None
    for cand in range(max(0, (base & 0x7FFF) - 2) | (base & 0x8000), ((base & 0x7FFF) + 3) | (base & 0x8000)):
        v = np.array([cand << 16], dtype=np.uint32).view(np.float32)[0]
        if not np.isfinite(v):
            continue
        dist = abs(Fraction(float(v)) - target)
        key = (dist, cand & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return best[1]


def test_bf16_from_f64_is_correctly_rounded():
    rng = np.random.default_rng(11)
    ds = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000))
    # double-rounding traps: just above a BF16 tie by less than half a binary32 ulp
    ds += [1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -8 - 2.0 ** -30, -(3.0 + 2.0 ** -7 + 2.0 ** -40),
           1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]
    for d in ds:
        assert oracle.bf16_from_f64(float(d)) == _nearest_bf16_exact(float(d)), d
    # 1 + 2^-8 + 2^-30 rounds up; going through binary32 first would give 1.0
    assert oracle.bf16_from_f64(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81


# ------------------------------------------------------------- sum of squares

@pytest.mark.parametrize("P", [256, 4096, 3584, 264, 1000, 8])
def test_sum_of_squares_exact_on_small_integers(P):
    # every partial sum is an integer below 2^24, so any complete tree gives the
    # exact sum of squares: a dropped or doubled column cannot hide
    rng = np.random.default_rng(P)
    v = rng.integers(-16, 17, size=P).astype(np.float32)
    assert oracle.sum_of_squares(v) == float(np.sum(v.astype(np.int64) ** 2))


def test_sum_of_squares_rounds_each_square_before_adding():
    # v = (1, 1 + 2^-12 + 2^-23, 0, ...): the second square is
    # 1 + 2^-11 + 2^-22 + 2^-24 + 2^-34 + 2^-46, rounded to binary32 it is
    # 1 + 2^-11 + 3 * 2^-23.  Added to 1 that is 2 + 2^-11 + 1.5 ulp (ulp 2^-22
    # at 2): a tie, to even, 2 + 2^-11 + 2^-21.  Squaring and adding in one
    # rounding (a fused multiply-add) would give 2 + 2^-11 + 2^-22.
    v = np.zeros(8, dtype=np.float32)
    v[0], v[1] = 1.0, 1.0 + 2.0 ** -12 + 2.0 ** -23
    assert oracle.sum_of_squares(v) == 2.0 + 2.0 ** -11 + 2.0 ** -21


def test_sum_of_squares_lane_adds_columns_in_order():
    # lane 0: 4096^2 = 2^24 then seven 1s.  In column order each +1 is a tie
    # that rounds back to 2^24 (even), so the total is 2^24.  Any other order
    # that adds the ones first gives 2^24 + 7 -> 2^24 + 8.
    v = np.zeros(256, dtype=np.float32)
    v[0] = 4096.0
    v[1:8] = 1.0
    assert oracle.sum_of_squares(v) == 16777216.0


def test_sum_of_squares_lanes_combine_by_butterfly():
    # lane 0 holds 2^24, lanes 1..31 hold 1.  Butterfly levels at lane 0:
    # 2^24+1 -> 2^24 (tie, even); +2 -> 2^24+2; +4 -> 2^24+6; +8 -> 2^24+14;
    # +16 -> 2^24+30, all exact.  A sequential fold over lanes would stay 2^24.
    v = np.zeros(256, dtype=np.float32)
    v[0] = 4096.0
    v[8::8] = 1.0
    assert oracle.sum_of_squares(v) == 16777216.0 + 30.0


def test_sum_of_squares_butterfly_pairs_adjacent_lanes_first():
    # lane 0 holds 2^24, lanes 1 and 17 hold 1.  Offsets 1, 2, 4, 8, 16: lane 0
    # meets lane 1 first (2^24 + 1 is a tie back to 2^24) and lanes 16-31 later
    # bring 1 (again back to 2^24): the total stays 2^24.  Offsets 16 first would
    # pair lanes 1 and 17 (1 + 1 = 2) and end at 2^24 + 2.
    v = np.zeros(256, dtype=np.float32)
    v[0] = 4096.0
    v[8] = 1.0
    v[136] = 1.0
    assert oracle.sum_of_squares(v) == 16777216.0


@pytest.mark.parametrize("ss,expect,other", [
    # ss * (float)(1/3584), then 1/sqrt: 45.38468933105469; the mean as ss / 3584
    # (one rounding instead of two) gives 45.38469314575195
    (1.74, 45.38468933105469, 45.38469314575195),
    # 1 / sqrt(mean): 41.21381378173828; sqrt(1 / mean) gives 41.213809967041016
    (2.11, 41.21381378173828, 41.213809967041016),
])
def test_inverse_rms_rounding_steps(ss, expect, other):
    # the values were found with numpy's IEEE float32 operations; each step of
    # the definition is one rounding, and the neighbouring formulas differ
    f = np.float32
    got = oracle.inverse_rms(float(f(ss)), 3584, 0.0)
    assert got == expect and got != other
    mean = f(f(ss) * f(1.0 / 3584))
    assert float(f(1.0) / np.sqrt(mean)) == expect


def test_sum_of_squares_chunks_fold_in_order():
    # chunk 0 holds 2^24, chunks 1..15 hold 1 each.  Folding chunks in order
    # from +0: every +1 is a tie back to 2^24.  A pairwise fold would give
    # 2^24 + 16 (ones first).
    v = np.zeros(4096, dtype=np.float32)
    v[0] = 4096.0
    v[256::256] = 1.0
    assert oracle.sum_of_squares(v) == 16777216.0


# ------------------------------------------------------------- EP finalize

def test_ep_constant_rows_closed_form():
    # constant rows of 1, gains 1, eps 0: ss = P, mean = 1, inv = 1, every
    # normalised value is 1, so out = bf16(sum of route weights) = 0.875 exactly
    d = constant_ep([[0.5, 0.25], [0.125]])
    out = ep_call(d)
    assert torch.equal(out.float(), torch.full((1, 256), 0.875))


def test_ep_slot_partials_are_rounded_to_bf16_before_the_slot_sum():
    # slot 0 partial 1 + 2^-8 + 2^-20 -> bf16 1 + 2^-7; slot 1 partial 2^-8.
    # Sum 1 + 3*2^-8 is a BF16 tie -> even -> 1 + 2^-6 = 1.015625.  Without the
    # per-slot rounding the sum 1 + 2^-7 + 2^-20 would round to 1.0078125.
    d = constant_ep([[1.0 + 2.0 ** -8 + 2.0 ** -20], [2.0 ** -8]])
    assert torch.equal(ep_call(d).float(), torch.full((1, 256), 1.015625))


def test_ep_slot_sum_stays_in_binary32():
    # three slots with one route each on rows of 1 (n = 1): partials 1,
    # 3 * 2^-10, 3 * 2^-10, all exact in BF16.  Summed in binary32 they give
    # 1 + 1.5 * 2^-8, above the BF16 tie 1 + 2^-8, so out = 1 + 2^-7 (0x3F81).
    # Rounding the running sum to BF16 after each slot would drop each
    # 3 * 2^-10 (below the tie) and give 1.0.
    d = constant_ep([[1.0], [3 * 2.0 ** -10], [3 * 2.0 ** -10]])
    assert np.all(bits(ep_call(d)) == 0x3F81)


def test_ep_slots_sum_in_rank_order():
    # partials 1, 2^-8, 2^-24, 2^-24 in rank order: 1 + 2^-8 exact, then each
    # 2^-24 is a tie back to 1 + 2^-8 (even); BF16 tie -> 1.0.  Summing in
    # reverse would reach 1 + 2^-8 + 2^-23 -> 1.0078125.
    d = constant_ep([[1.0], [2.0 ** -8], [2.0 ** -24], [2.0 ** -24]])
    assert torch.equal(ep_call(d).float(), torch.full((1, 256), 1.0))


def test_ep_routes_sum_in_route_order():
    # one slot, routes 1 + 2^-8, 2^-24, 2^-24: in order each 2^-24 is a tie
    # back to 1 + 2^-8 -> bf16 1.0.  Reverse order: 1 + 2^-8 + 2^-23 -> 1.0078125.
    d = constant_ep([[1.0 + 2.0 ** -8, 2.0 ** -24, 2.0 ** -24]])
    assert torch.equal(ep_call(d).float(), torch.full((1, 256), 1.0))


def test_ep_gain_placement_weight_before_norm():
    # rows 1, gamma 1, gain center 1 -> g = 2, eps 0.  Gain before the norm:
    # v = 2, ss = 4P, inv = 1/2, n = 1 -> out = w.  After the norm: inv = 1,
    # n = 2 -> out = 2w.
    on = ep_call(constant_ep([[0.75]], gamma=1.0, wbn=True))
    off = ep_call(constant_ep([[0.75]], gamma=1.0, wbn=False))
    assert torch.equal(on.float(), torch.full((1, 256), 0.75))
    assert torch.equal(off.float(), torch.full((1, 256), 1.5))


def test_ep_normalisation_product_order_with_subnormals():
    # Rows x = 1.75*2^-75, gamma = 1.625*2^-73 with gain center 0 (g = gamma),
    # eps = 2^-100, one route of weight 1.  x*g = 5.6875*2^-149 is subnormal
    # and rounds to 6*2^-149, so the order of the products shows:
    #  gain before the norm: v = 6*2^-149, v*v underflows to 0, inv = 1/sqrt(2^-100)
    #    = 2^50, n = v*inv = 1.5*2^-97;
    #  gain after the norm: x*x = 1.53125*2^-149 -> 2^-148, ss = 256*2^-148 = 2^-140,
    #    mean = 2^-148, + eps -> 2^-100, inv = 2^50, n = (x*inv)*g = 1.421875*2^-97.
    # Multiplying in the other order in either branch gives the other value;
    # flushing subnormals to zero changes both.
    x, gamma = 1.75 * 2.0 ** -75, 1.625 * 2.0 ** -73
    on = ep_call(constant_ep([[1.0]], row_value=x, gamma=gamma, gc=0.0, eps=2.0 ** -100, wbn=True))
    off = ep_call(constant_ep([[1.0]], row_value=x, gamma=gamma, gc=0.0, eps=2.0 ** -100, wbn=False))
    assert torch.equal(on.float(), torch.full((1, 256), 1.5 * 2.0 ** -97))
    assert torch.equal(off.float(), torch.full((1, 256), 1.421875 * 2.0 ** -97))


def test_ep_product_order_after_the_norm_at_a_bf16_boundary():
    # P = 8, one route of weight 1, row (2.3125, 0.8125, 0, ...), gamma[0] = 2.828125,
    # gain center 0, eps 0, gain after the norm: ss = 2.3125^2 + 0.8125^2 = 6.0078125
    # and inv = 1/sqrt(ss/8) = 1.1539495 in FP32.  (x*inv)*g = 7.546875 rounds to the
    # BF16 0x40F2; x*(inv*g) = 7.5468745 would round to 0x40F1.
    row = torch.tensor([2.3125, 0.8125, 0, 0, 0, 0, 0, 0]).to(torch.bfloat16).reshape(1, 1, 8)
    gamma = torch.tensor([2.828125, 1, 1, 1, 1, 1, 1, 1]).to(torch.bfloat16)
    d = dict(rows=row, rows_per_slot=1, idx=torch.zeros((1, 1, 1), dtype=torch.int32),
             w=torch.ones((1, 1)), gamma=gamma, gain_center=0.0, eps=0.0, weight_before_norm=False,
             b=1, tp=1, K=1, P=8)
    assert int(bits(ep_call(d))[0, 0]) == 0x40F2


def test_ep_inverse_rms_uses_eps():
    # rows 0.5, gains 1, eps 0.75: mean 0.25 + 0.75 = 1 -> inv 1 -> n = 0.5
    d = constant_ep([[1.0]], row_value=0.5, eps=0.75)
    assert torch.equal(ep_call(d).float(), torch.full((1, 256), 0.5))


def test_ep_gains_of_one_make_weight_before_norm_moot():
    d = synth.config(1)
    d["gamma"] = torch.zeros_like(d["gamma"])  # g = 0 + 1 = 1 exactly
    assert np.array_equal(bits(ep_call(d, weight_before_norm=True)), bits(ep_call(d, weight_before_norm=False)))


def test_ep_power_of_two_weight_scales_exactly():
    d = synth.config(1)
    base = ep_call(d).float()
    scaled = ep_call(d, w=d["w"] * 4.0).float()
    assert torch.equal(scaled, base * 4.0)


def test_ep_non_local_route_equals_dropping_it():
    d = synth.config(1)
    drop_k = 2
    idx = d["idx"].clone()
    idx[:, :, drop_k] = torch.where(idx[:, :, drop_k] >= 0, torch.full_like(idx[:, :, drop_k], -7),
                                    idx[:, :, drop_k])
    idx[0, 1, drop_k] = d["rows_per_slot"]  # out of range on the high side too
    idx[1, 1, drop_k] = -1
    keep = [k for k in range(d["K"]) if k != drop_k]
    dropped = ep_call(d, idx=d["idx"][:, :, keep].contiguous(), w=d["w"][:, keep].contiguous(), K=d["K"] - 1)
    assert np.array_equal(bits(ep_call(d, idx=idx)), bits(dropped))


def test_ep_token_without_local_routes_is_positive_zero():
    d = synth.config(1)
    idx = d["idx"].clone()
    idx[:, 2, :] = -1
    out = bits(ep_call(d, idx=idx))
    assert np.all(out[2] == 0)  # +0, never -0


def test_ep_no_output_has_negative_zero():
    d = synth.config(1)
    d["rows"] = torch.where(d["rows"].float().abs() < 0.5, torch.tensor(-0.0), d["rows"].float()).to(torch.bfloat16)
    assert not np.any(bits(ep_call(d)) == 0x8000)


def test_ep_row_placement_within_a_slot_is_irrelevant():
    d = synth.config(2, b=8, P=512)
    perm_idx = d["idx"].clone()
    rows = d["rows"].clone()
    g = torch.Generator().manual_seed(3)
    for s in range(d["tp"]):
        perm = torch.randperm(d["rows_per_slot"], generator=g)
        inv = torch.empty_like(perm)
        inv[perm] = torch.arange(len(perm))
        rows[s] = d["rows"][s][perm]
        m = perm_idx[s] >= 0
        perm_idx[s][m] = inv[perm_idx[s][m].long()].to(torch.int32)
    assert np.array_equal(bits(ep_call(d)), bits(ep_call(d, rows=rows, idx=perm_idx)))


def test_ep_b_zero_does_nothing():
    d = synth.config(1)
    out = ep_call(d, b=0, idx=d["idx"][:, :0].contiguous(), w=d["w"][:0].contiguous())
    assert out.shape == (0, d["P"])


def test_ep_bf16_route_weights_widen_exactly():
    d = synth.config(1)
    wb = d["w"].to(torch.bfloat16)
    assert np.array_equal(bits(ep_call(d, w=wb)), bits(ep_call(d, w=wb.float())))


def _ep_double(d):
    """Brute force in double: the formula with the BF16 partial rounding."""
    rows = d["rows"].double().numpy()
    idx = d["idx"].numpy()
    w = d["w"].double().numpy()
    g = d["gamma"].double().numpy() + d["gain_center"]
    out = np.zeros((d["b"], d["P"]))
    parts = np.zeros((d["tp"], d["b"], d["P"]))
    for t in range(d["b"]):
        for s in range(d["tp"]):
            part = np.zeros(d["P"])
            for k in range(d["K"]):
                j = idx[s, t, k]
                if not 0 <= j < d["rows_per_slot"]:
                    continue
                x = rows[s, j]
                v = x * g if d["weight_before_norm"] else x
                n = v / np.sqrt(np.mean(v * v) + d["eps"])
                if not d["weight_before_norm"]:
                    n = n * g
                part += w[t, k] * n
            parts[s, t] = torch.from_numpy(part).to(torch.bfloat16).double().numpy()
            out[t] += parts[s, t]
    return out, parts


@pytest.mark.parametrize("wbn", [True, False])
def test_ep_brute_force_double(wbn):
    d = synth.config(1, weight_before_norm=wbn)
    ref, parts = _ep_double(d)
    got = ep_call(d).double().numpy()
    tol = ulp_bf16(ref) + ulp_bf16(np.abs(parts).max(axis=0))
    assert np.all(np.abs(got - ref) <= tol)


# ------------------------------------------------------------- expert-TP finalize

@pytest.mark.parametrize("wbn", [True, False])
def test_tp_brute_force_double(wbn):
    # The expert-TP formula recomputed on tiny inputs: each route row's slot sum
    # in binary32 from +0 in slot order, rounded to BF16 (the method fixes both),
    # then the norm, the gains and the weighted route sum in double.  The
    # oracle's binary32 steps must land within one BF16 ulp of it, plus the
    # binary32 rounding of a route sum that cancels.
    d = synth.config(3, b=4, P=264, tp=3, K=3, weight_before_norm=wbn)
    idx = d["idx"].clone()
    idx[1, 2] = -1  # one route without a row
    Q = d["partials"].float().numpy()
    g = d["gamma"].double().numpy() + d["gain_center"]
    w = d["w"].double().numpy()
    ref = np.zeros((d["b"], d["P"]))
    mag = np.zeros((d["b"], d["P"]))
    for t in range(d["b"]):
        for k in range(d["K"]):
            j = int(idx[t, k])
            if not 0 <= j < d["num_rows"]:
                continue
            xs = np.zeros(d["P"], dtype=np.float32)
            for s in range(d["tp"]):
                xs = (xs + Q[s, j]).astype(np.float32)
            x = torch.from_numpy(xs).to(torch.bfloat16).double().numpy()
            v = x * g if wbn else x
            n = v / np.sqrt(np.mean(v * v) + d["eps"])
            if not wbn:
                n = n * g
            ref[t] += w[t, k] * n
            mag[t] += np.abs(w[t, k] * n)
    got = tp_call(d, idx=idx).double().numpy()
    assert np.all(np.abs(got - ref) <= ulp_bf16(ref) + 2.0 ** -20 * mag)


@pytest.mark.parametrize("kind", ["ep", "tp"])
def test_single_route_is_textbook_rmsnorm(kind):
    # One route per token, w = 1, tp = 1, gamma = 0 with gain center 1: the
    # finalize is a plain RMS norm of the route row, x / sqrt(mean(x^2) + eps),
    # computed here in double.  The oracle's FP32 steps round far below a BF16
    # ulp, so every output is within one BF16 ulp of it (and nearly all equal
    # its BF16 rounding).
    P, b, eps = 512, 6, 1e-6
    x = synth.bf16(synth.normal(0x7E, 1, b * P), (b, P))
    common = dict(w=torch.ones((b, 1)), gamma=torch.zeros(P).to(torch.bfloat16), gain_center=1.0, eps=eps,
                  weight_before_norm=True, b=b, tp=1, K=1, P=P)
    if kind == "ep":  # token t's route is row t of the only slot
        out = ep_call(dict(common, rows=x.reshape(1, b, P), rows_per_slot=b,
                           idx=torch.arange(b, dtype=torch.int32).reshape(1, b, 1)))
    else:
        out = tp_call(dict(common, partials=x.reshape(1, b, P), num_rows=b,
                           idx=torch.arange(b, dtype=torch.int32).reshape(b, 1)))
    xd = x.double().numpy()
    ref = xd / np.sqrt(np.mean(xd * xd, axis=1, keepdims=True) + eps)
    got = out.double().numpy()
    assert np.all(np.abs(got - ref) <= ulp_bf16(ref))
    exact = bits(torch.from_numpy(ref).float().to(torch.bfloat16)) == bits(out)
    assert exact.mean() > 0.99


@pytest.mark.parametrize("wbn", [True, False])
def test_tp_equals_ep_on_slot_summed_rows(wbn):
    # x_r = bf16(sum_s Q_s), then the EP formula on one slot with every route
    # local: the two statements of the method must agree bit for bit, with the
    # gains before the norm or after it (gamma is random, so the two differ).
    d = synth.config(3, b=6, P=512, tp=4, weight_before_norm=wbn)
    acc = torch.zeros(d["partials"].shape[1:], dtype=torch.float32)
    for s in range(d["tp"]):  # slot order, one FP32 add per slot
        acc = acc + d["partials"][s].float()
    rows = acc.to(torch.bfloat16).unsqueeze(0)
    ep = oracle.ep_finalize(rows, d["num_rows"], d["idx"].unsqueeze(0).contiguous(), d["w"], d["gamma"],
                            d["gain_center"], d["eps"], d["weight_before_norm"], d["b"], 1, d["K"], d["P"])
    assert np.array_equal(bits(tp_call(d)), bits(ep))


def test_tp_k_partials_sum_in_slot_order_before_rounding():
    # columns 0..127 carry partials 1, 2^-8, 2^-24, 2^-24 in slots 0..3: in slot
    # order x = 1 + 2^-8 (each 2^-24 is a tie back to even) -> bf16 tie -> 1.0.
    # Columns 128..255 carry 1 in slot 0 only -> x = 1.  So x is a row of ones:
    # gains 1, eps 0 -> inv 1 -> out = w = 1 everywhere.  Reverse order would
    # give x = 1.0078125 on half the row and out != 1.
    P = 256
    Q = torch.zeros((4, 1, P))
    for s, v in enumerate([1.0, 2.0 ** -8, 2.0 ** -24, 2.0 ** -24]):
        Q[s, 0, :128] = v
    Q[0, 0, 128:] = 1.0
    d = dict(partials=Q.to(torch.bfloat16), num_rows=1, idx=torch.zeros((1, 1), dtype=torch.int32),
             w=torch.ones((1, 1)), gamma=torch.zeros(P).to(torch.bfloat16), gain_center=1.0, eps=0.0,
             weight_before_norm=True, b=1, tp=4, K=1, P=P)
    assert torch.equal(tp_call(d).float(), torch.ones((1, P)))


def test_tp_non_local_route_contributes_nothing():
    d = synth.config(3, b=4, P=512, tp=2)
    idx = d["idx"].clone()
    idx[1, 3] = -1
    idx[2, 0] = d["num_rows"] + 5
    idx[0, 1] = d["num_rows"]  # one past the last row
    keep_rows = []
    a = tp_call(d, idx=idx)
    for t in range(d["b"]):
        keep = [k for k in range(d["K"]) if 0 <= idx[t, k] < d["num_rows"]]
        keep_rows.append(tp_call(d, idx=idx[t:t + 1, keep].contiguous(), w=d["w"][t:t + 1, keep].contiguous(),
                                 b=1, K=len(keep)))
    assert np.array_equal(bits(a), bits(torch.cat(keep_rows)))


def test_tp_tiny_negative_output_is_positive_zero():
    # one route of weight -2^-140, rows of 1, gains 1, eps 0: n = 1, the route
    # sum is -2^-140, below half the smallest BF16 subnormal (2^-133), so it
    # rounds to -0, which is written as +0
    d = dict(partials=torch.ones((1, 1, 256)).to(torch.bfloat16), num_rows=1,
             idx=torch.zeros((1, 1), dtype=torch.int32), w=torch.full((1, 1), -2.0 ** -140),
             gamma=torch.zeros(256).to(torch.bfloat16), gain_center=1.0, eps=0.0, weight_before_norm=True,
             b=1, tp=1, K=1, P=256)
    assert np.all(bits(tp_call(d)) == 0)


def test_tp_routes_sum_in_route_order():
    # three routes over constant rows of 1 (n = 1), weights 1 + 2^-8, 2^-24,
    # 2^-24 -> 1.0 in route order (see the EP case)
    P = 256
    Q = torch.ones((1, 3, P)).to(torch.bfloat16)
    d = dict(partials=Q, num_rows=3, idx=torch.tensor([[0, 1, 2]], dtype=torch.int32),
             w=torch.tensor([[1.0 + 2.0 ** -8, 2.0 ** -24, 2.0 ** -24]]), gamma=torch.zeros(P).to(torch.bfloat16),
             gain_center=1.0, eps=0.0, weight_before_norm=False, b=1, tp=1, K=3, P=P)
    assert torch.equal(tp_call(d).float(), torch.full((1, P), 1.0))


# ------------------------------------------------------------- latent tail

def test_latent_norm_constant_rows():
    # tp = 2 slots of 1 each -> x = 2; gamma 1, eps 0: inv = 1/2 (up to the
    # rounding of 1/3584, far below BF16) -> y = 1 exactly after BF16 rounding
    L = 3584
    lat = torch.ones((2, 3, L)).to(torch.bfloat16)
    y = oracle.latent_norm(lat, torch.ones(L).to(torch.bfloat16), 0.0, 3, 2, L)
    assert torch.equal(y.float(), torch.ones((3, L)))


def test_latent_norm_matches_textbook_rmsnorm():
    d = synth.config(4, b=3, tp=1, L=512, H=256, tp_s=0, with_weight=False)
    y = oracle.latent_norm(d["latent"], d["gamma"], d["eps"], 3, 1, 512).double().numpy()
    x = d["latent"][0].double().numpy()
    ref = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + d["eps"]) * d["gamma"].double().numpy()
    assert np.all(np.abs(y - ref) <= ulp_bf16(ref))


def _latent_pair(col0_slots, col1, gamma0):
    lat = torch.zeros((2, 1, 8))
    lat[0, 0, 0], lat[1, 0, 0], lat[0, 0, 1] = col0_slots[0], col0_slots[1], col1
    gamma = torch.ones(8)
    gamma[0] = gamma0
    return lat.to(torch.bfloat16), gamma.to(torch.bfloat16)


def test_latent_norm_uses_eps():
    # tp = 2 slots of 1 -> x = 2 over L = 8 columns: ss = 32, mean = 32 * 0.125
    # = 4; eps = 12 makes the denominator 16, inv = 1/4 and y = 2 * 1/4 * 1 =
    # 0.5 exactly (without eps, y would be 1)
    lat = torch.ones((2, 1, 8)).to(torch.bfloat16)
    y = oracle.latent_norm(lat, torch.ones(8).to(torch.bfloat16), 12.0, 1, 2, 8)
    assert torch.equal(y.float(), torch.full((1, 8), 0.5))


def test_latent_norm_brute_force_double():
    # The latent norm recomputed on tiny inputs (ragged chunk: L = 264): the
    # slot sum in binary32 from +0 in slot order, rounded to BF16 (as the
    # method fixes), then x / sqrt(mean(x^2) + eps) * gamma in double.  The
    # oracle's y must be within one BF16 ulp of it.
    b, tp, L = 3, 3, 264
    d = synth.latent_up_inputs(0x1B, b=b, tp=tp, L=L, H=8, tp_s=0)
    lat = d["latent"].float().numpy()
    gamma = d["gamma"].double().numpy()
    ref = np.zeros((b, L))
    for t in range(b):
        xs = np.zeros(L, dtype=np.float32)
        for s in range(tp):
            xs = (xs + lat[s, t]).astype(np.float32)
        x = torch.from_numpy(xs).to(torch.bfloat16).double().numpy()
        ref[t] = x / np.sqrt(np.mean(x * x) + d["eps"]) * gamma
    got = oracle.latent_norm(d["latent"], d["gamma"], d["eps"], b, tp, L).double().numpy()
    assert np.all(np.abs(got - ref) <= ulp_bf16(ref))


def test_latent_norm_rounds_the_slot_sum_to_bf16():
    # column 0 holds 2.578125 and -0.00640869140625 in the two slots, column 1
    # holds 3.546875, gamma[0] = 1.2734375, eps 0.  The slot sum rounded to BF16
    # (2.5625) gives y[0] = 0x4008; the unrounded sum (2.57171...) would give
    # 0x4007.  (Found with numpy float32, each step one rounding.)
    lat, gamma = _latent_pair((2.578125, -0.00640869140625), 3.546875, 1.2734375)
    y = oracle.latent_norm(lat, gamma, 0.0, 1, 2, 8)
    assert int(bits(y)[0, 0]) == 0x4008


def test_latent_norm_product_order():
    # slots (3.609375, -0.041015625) in column 0, 0.55859375 in column 1,
    # gamma[0] = 1.3671875, eps 0: (x * inv) * gamma rounds to 0x4074 and
    # x * (inv * gamma) would round to 0x4075
    lat, gamma = _latent_pair((3.609375, -0.041015625), 0.55859375, 1.3671875)
    y = oracle.latent_norm(lat, gamma, 0.0, 1, 2, 8)
    assert int(bits(y)[0, 0]) == 0x4074


def test_latent_norm_zero_column_with_negative_gamma_is_positive_zero():
    # column 0's slots cancel (1 and -1: x = +0) and gamma[0] = -1.5, so
    # (x * inv) * gamma = +0 * -1.5 = -0, which y (a BF16 output) stores as +0.
    # Column 1 (x = 1) gives ss = 1, inv = sqrt(8), y[1] = bf16(2.828...) = 0x4035.
    lat, gamma = _latent_pair((1.0, -1.0), 1.0, -1.5)
    y = bits(oracle.latent_norm(lat, gamma, 0.0, 1, 2, 8))
    assert int(y[0, 0]) == 0x0000 and int(y[0, 1]) == 0x4035


def test_latent_up_rounds_the_double_sum_straight_to_bf16():
    # y = (1, 2^-8, 2^-30, 0, ...), one output row of ones: the sum is exactly
    # 1 + 2^-8 + 2^-30 in double, above the tie between 1 and 1 + 2^-7, so it
    # rounds up to 0x3F81.  Through binary32 it would first become the tie
    # 1 + 2^-8 and then round to even, 0x3F80.
    y = torch.tensor([[1.0, 2.0 ** -8, 2.0 ** -30, 0, 0, 0, 0, 0]]).to(torch.bfloat16)
    w = torch.ones((1, 8)).to(torch.bfloat16)
    out = oracle.latent_up(y, w, None, 0, 1, 8, 1)
    assert int(bits(out)[0, 0]) == 0x3F81


def test_latent_up_adds_the_shared_slots_in_double():
    # y = (1, 2^-8, 0, ...) against a row of ones gives exactly 1 + 2^-8 (the
    # BF16 tie between 1 and 1 + 2^-7); one shared slot of 2^-30 moves the
    # double sum above the tie, so out rounds up to 0x3F81.  Accumulated in
    # binary32, 1 + 2^-8 + 2^-30 would fall back onto the tie and give 0x3F80.
    y = torch.tensor([[1.0, 2.0 ** -8, 0, 0, 0, 0, 0, 0]]).to(torch.bfloat16)
    shared = torch.full((1, 1, 1), 2.0 ** -30).to(torch.bfloat16)
    out = oracle.latent_up(y, torch.ones((1, 8)).to(torch.bfloat16), shared, 1, 1, 8, 1)
    assert int(bits(out)[0, 0]) == 0x3F81


def test_latent_up_tiny_negative_is_positive_zero():
    # y[0] = 2^-70 times a weight -2^-70: the sum -2^-140 is below half the
    # smallest BF16 subnormal (2^-133), rounds to -0 and is written as +0
    y = torch.zeros((1, 8))
    y[0, 0] = 2.0 ** -70
    w = torch.zeros((1, 8))
    w[0, 0] = -2.0 ** -70
    out = oracle.latent_up(y.to(torch.bfloat16), w.to(torch.bfloat16), None, 0, 1, 8, 1)
    assert int(bits(out)[0, 0]) == 0x0000


def test_latent_up_identity_weight_reproduces_y():
    L, H, b = 256, 512, 3
    y = synth.bf16(synth.normal(1, 1, b * L), (b, L))
    w = torch.zeros((H, L))
    w[:L, :L] = torch.eye(L)
    out = oracle.latent_up(y, w.to(torch.bfloat16), None, 0, b, L, H)
    assert np.array_equal(bits(out[:, :L]), bits(y))
    assert np.all(bits(out[:, L:]) == 0)


def test_latent_up_zero_weight_sums_shared_slots_exactly():
    L, H, b, tp_s = 64, 128, 2, 8
    sh = synth.bf16(synth.normal(2, 1, tp_s * b * H, std=0.5), (tp_s, b, H))
    out = oracle.latent_up(torch.zeros((b, L)).to(torch.bfloat16), torch.zeros((H, L)).to(torch.bfloat16),
                           sh, tp_s, b, L, H)
    exact = [[sum(Fraction(float(sh[s, t, n])) for s in range(tp_s)) for n in range(H)] for t in range(b)]
    for t in range(b):
        for n in range(H):
            assert int(bits(out)[t, n]) == (_nearest_bf16_exact(float(exact[t][n])) if exact[t][n] != 0 else 0)


def test_latent_up_matches_library_matmul():
    d = synth.config(4, b=4, L=256, H=384, tp=2, tp_s=3)
    y = oracle.latent_norm(d["latent"], d["gamma"], d["eps"], 4, 2, 256)
    out = oracle.latent_up(y, d["w_up"], d["shared"], 3, 4, 256, 384)
    ref = y.double().numpy() @ d["w_up"].double().numpy().T + d["shared"].double().numpy().sum(axis=0)
    assert np.array_equal(bits(out), bits(torch.from_numpy(ref).float().to(torch.bfloat16)))


# ------------------------------------------------------------- shared expert

def _onehot_shared(gates, ups, H=16, I=None, down=None):
    I = I or len(gates)
    x = torch.zeros((1, H))
    x[0, 3] = 1.0
    wg = torch.zeros((I, H))
    wu = torch.zeros((I, H))
    wg[:, 3] = torch.tensor(gates)
    wu[:, 3] = torch.tensor(ups)
    wd = torch.zeros((H, I)) if down is None else down
    return x.to(torch.bfloat16), wg.to(torch.bfloat16), wu.to(torch.bfloat16), wd.to(torch.bfloat16)


def test_shared_activation_special_values():
    import math

    gates = [0.0, 64.0, -64.0, 2.0, -3.0]
    ups = [5.0, 0.75, 1.0, -1.5, 0.5]
    x, wg, wu, wd = _onehot_shared(gates, ups)
    h, _ = oracle.shared_expert(x, wg, wu, wd, 1, 16, 5, out_in=torch.zeros((1, 16)).to(torch.bfloat16))
    expect = [0.0, 48.0, -64.0 / (1.0 + math.exp(64.0)) * 1.0,
              2.0 / (1.0 + math.exp(-2.0)) * -1.5, -3.0 / (1.0 + math.exp(3.0)) * 0.5]
    assert bits(h)[0, 0] == 0 and bits(h)[0, 1] == bits(bf([48.0]))[0]
    for i in (2, 3, 4):
        assert int(bits(h)[0, i]) == _nearest_bf16_exact(expect[i])


def test_shared_h_rounds_the_double_product_straight_to_bf16():
    # gate = -0.7578125, up = 1.5546875 (both BF16): silu(gate) * up in double
    # is -0.37597656760..., just beyond the tie -0.3759765625 between BF16
    # -0.375 (0xBEC0) and -0.376953125 (0xBEC1), by 1.4e-8 relative (far above
    # the error of exp).  Rounded straight to BF16 it gives 0xBEC1; rounded to
    # binary32 first it would land on the tie and go to the even 0xBEC0.
    x, wg, wu, wd = _onehot_shared([-0.7578125], [1.5546875])
    h, _ = oracle.shared_expert(x, wg, wu, wd, 1, 16, 1, out_in=torch.zeros((1, 16)).to(torch.bfloat16))
    assert int(bits(h)[0, 0]) == 0xBEC1


def test_shared_h_of_a_zero_gate_is_positive_zero():
    # silu(0) = 0 / (1 + 1) = +0; times up = -1 gives -0, which h stores as +0
    x, wg, wu, wd = _onehot_shared([0.0], [-1.0])
    h, _ = oracle.shared_expert(x, wg, wu, wd, 1, 16, 1, out_in=torch.zeros((1, 16)).to(torch.bfloat16))
    assert int(bits(h)[0, 0]) == 0x0000


def test_shared_h_keeps_silu_in_double():
    # gate = 18.75, up = 1.25: silu(18.75) = 18.75 (1 - 7.2e-9), so in double
    # h = 23.4375 (1 - 7.2e-9) = 23.43749983..., just under the BF16 tie 23.4375
    # between 23.375 (0x41BB) and 23.5 (0x41BC): it rounds down to 0x41BB.  With
    # silu rounded to binary32 first (to 18.75 exactly) the product would be the
    # tie itself and round to the even 0x41BC.
    x, wg, wu, wd = _onehot_shared([18.75], [1.25])
    h, _ = oracle.shared_expert(x, wg, wu, wd, 1, 16, 1, out_in=torch.zeros((1, 16)).to(torch.bfloat16))
    assert int(bits(h)[0, 0]) == 0x41BB


def test_shared_gate_and_up_round_their_double_sums_straight_to_bf16():
    # x = (1, 2^-8, 2^-30, 1, 0, ...).  Unit 0: gate = x . (1, 1, 1, 0, ...) =
    # 1 + 2^-8 + 2^-30 exactly in double, which rounds up to 1.0078125, and up =
    # 1, so h = bf16(silu(1.0078125)) = bf16(0.73832) = 0x3F3D (through binary32
    # the gate would be 1.0 and h = bf16(0.73106) = 0x3F3B).  Unit 1: gate = 64
    # (silu = 64 up to 1e-26) and up = 1 + 2^-8 + 2^-30 -> 1.0078125, so h =
    # 64.5 = 0x4281 (through binary32: 64 = 0x4280).
    H, I = 16, 2
    x = torch.zeros((1, H))
    x[0, :4] = torch.tensor([1.0, 2.0 ** -8, 2.0 ** -30, 1.0])
    wg, wu = torch.zeros((I, H)), torch.zeros((I, H))
    wg[0, :3], wu[0, 0] = 1.0, 1.0
    wg[1, 3], wu[1, :3] = 64.0, 1.0
    bf16 = torch.bfloat16
    h, _ = oracle.shared_expert(x.to(bf16), wg.to(bf16), wu.to(bf16), torch.zeros((H, I)).to(bf16), 1, H, I,
                                out_in=torch.zeros((1, H)).to(bf16))
    assert [int(v) for v in bits(h)[0]] == [0x3F3D, 0x4281]


def test_shared_down_rounds_its_double_sum_straight_to_bf16():
    # gate 64 and ups 2^-6, 2^-14, 2^-36 make h = (1, 2^-8, 2^-30) exactly;
    # a down row of ones sums them to 1 + 2^-8 + 2^-30, which rounds up to
    # 0x3F81 (through binary32 it would be the tie 1 + 2^-8 and give 0x3F80)
    down = torch.zeros((16, 3))
    down[7, :] = 1.0
    x, wg, wu, wd = _onehot_shared([64.0, 64.0, 64.0], [2.0 ** -6, 2.0 ** -14, 2.0 ** -36], down=down)
    h, out = oracle.shared_expert(x, wg, wu, wd, 1, 16, 3, accumulate=False)
    assert [int(v) for v in bits(h)[0]] == [0x3F80, 0x3B80, 0x3080]
    assert int(bits(out)[0, 7]) == 0x3F81


def test_shared_down_tiny_negative_is_positive_zero():
    # h = silu(64) * 2^-76 = 2^-70 (silu(64) = 64 up to 1e-26), one down weight
    # -2^-70: d = -2^-140, below half the smallest BF16 subnormal (2^-133), so
    # bf16(d) = -0, which is written as +0 when out is overwritten
    down = torch.zeros((16, 1))
    down[5, 0] = -2.0 ** -70
    x, wg, wu, wd = _onehot_shared([64.0], [2.0 ** -76], down=down)
    h, out = oracle.shared_expert(x, wg, wu, wd, 1, 16, 1, accumulate=False)
    assert int(bits(h)[0, 0]) == 0x1C80
    assert np.all(bits(out) == 0)


def test_shared_down_selects_h():
    # W_down one-hot: out[n] = bf16(out_in[n] + h[i(n)])
    gates, ups = [64.0, 64.0], [0.5, -0.25]  # h = 32, -16 exactly
    down = torch.zeros((16, 2))
    down[5, 0] = 1.0
    down[9, 1] = 1.0
    x, wg, wu, wd = _onehot_shared(gates, ups, down=down)
    out_in = torch.full((1, 16), 0.5).to(torch.bfloat16)
    _, out = oracle.shared_expert(x, wg, wu, wd, 1, 16, 2, out_in=out_in)
    expect = torch.full((1, 16), 0.5)
    expect[0, 5] = 32.5
    expect[0, 9] = -15.5
    assert torch.equal(out.float(), expect)


def test_shared_zero_input_or_zero_down_leaves_out():
    d = synth.shared_expert_inputs(9, b=2, H=64, I=96)
    out_in = synth.bf16(synth.normal(9, 50, 2 * 64), (2, 64))
    _, out = oracle.shared_expert(torch.zeros((2, 64)).to(torch.bfloat16), d["w_gate"], d["w_up"], d["w_down"],
                                  2, 64, 96, out_in=out_in)
    assert np.array_equal(bits(out), bits(out_in))
    _, out = oracle.shared_expert(d["x"], d["w_gate"], d["w_up"], torch.zeros_like(d["w_down"]), 2, 64, 96,
                                  out_in=out_in)
    assert np.array_equal(bits(out), bits(out_in))


def test_shared_matches_library_matmul():
    d = synth.shared_expert_inputs(10, b=3, H=64, I=96)
    out_in = synth.bf16(synth.normal(10, 50, 3 * 64), (3, 64))
    h, out = oracle.shared_expert(d["x"], d["w_gate"], d["w_up"], d["w_down"], 3, 64, 96, out_in=out_in)
    x = d["x"].double().numpy()
    gate = torch.from_numpy(x @ d["w_gate"].double().numpy().T).float().to(torch.bfloat16).double().numpy()
    up = torch.from_numpy(x @ d["w_up"].double().numpy().T).float().to(torch.bfloat16).double().numpy()
    href = torch.from_numpy(gate / (1.0 + np.exp(-gate)) * up).float().to(torch.bfloat16)
    assert np.array_equal(bits(h), bits(href))
    dd = torch.from_numpy(href.double().numpy() @ d["w_down"].double().numpy().T).float().to(torch.bfloat16)
    ref = (out_in.float() + dd.float()).to(torch.bfloat16)
    assert np.array_equal(bits(out), bits(ref))
    _, plain = oracle.shared_expert(d["x"], d["w_gate"], d["w_up"], d["w_down"], 3, 64, 96, accumulate=False)
    assert np.array_equal(bits(plain), bits(dd))


def test_shared_down_matches_library_matmul_and_composes():
    d = synth.shared_expert_inputs(12, b=2, H=64, I=96)
    h, out = oracle.shared_expert(d["x"], d["w_gate"], d["w_up"], d["w_down"], 2, 64, 96, accumulate=False)
    ref = torch.from_numpy(h.double().numpy() @ d["w_down"].double().numpy().T).float().to(torch.bfloat16)
    got = oracle.shared_down(h, d["w_down"], 2, 64, 96, accumulate=False)
    assert np.array_equal(bits(got), bits(ref))
    assert np.array_equal(bits(got), bits(out))
