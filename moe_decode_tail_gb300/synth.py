"""Seeded synthetic inputs for the MoE decode tail (CPU tensors).

This module only draws inputs: it holds none of the tail's arithmetic, and both
the CUDA path's tests/benchmark and the CPU oracle take their inputs from here.

Random numbers come from a counter-based generator, splitmix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): draw i
of stream s under seed S is splitmix64's output for the counter
``S + (s * 2**32 + i + 1) * 0x9E3779B97F4A7C15``, so a value never depends on
how many other values were drawn before it and every machine gets the same
bits.  Normals use the Box-Muller transform on two 53-bit uniforms, in double,
and are rounded once to the stored type (BF16 by round-to-nearest-even).

Workload shapes follow the decode configurations the tail is measured on:
EP finalize (route rows per partition slot), expert-TP finalize (K-partials of
every route row), the latent tail with its 3584 -> 7168 up-projection and the
fused shared expert.  Every recipe is stated in the docstring of its builder.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _u64_range(base: np.uint64, lo: int, hi: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        return _mix(base + np.arange(lo, hi, dtype=np.uint64) * _GOLDEN)


def _stream_base(seed: int, stream: int) -> np.uint64:
    return np.uint64((seed + ((stream << 32) + 1) * 0x9E3779B97F4A7C15) & (2**64 - 1))


def _chunked(n: int, fn) -> None:
    """Run fn(lo, hi) over [0, n) in chunks, on threads (numpy drops the GIL)."""
    spans = [(lo, min(n, lo + _CHUNK)) for lo in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for lo, hi in spans:
            fn(lo, hi)
        return
    with ThreadPoolExecutor(max_workers=min(len(spans), os.cpu_count() or 1)) as pool:
        list(pool.map(lambda span: fn(*span), spans))


def u64(seed: int, stream: int, n: int) -> np.ndarray:
    """n raw 64-bit draws of (seed, stream), counter-based."""
    out = np.empty(n, dtype=np.uint64)
    base = _stream_base(seed, stream)

    def fill(lo, hi):
        out[lo:hi] = _u64_range(base, lo, hi)

    _chunked(n, fill)
    return out


def _unit(bits: np.ndarray) -> np.ndarray:
    return ((bits >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1), double (53 random bits, never 0)."""
    return _unit(u64(seed, stream, n))


def normal(seed: int, stream: int, n: int, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """n normals N(mean, std^2), double: Box-Muller on draw i of streams
    2*stream and 2*stream+1 gives normals 2i (cosine) and 2i+1 (sine)."""
    half = (n + 1) // 2
    z = np.empty(2 * half, dtype=np.float64)
    b1, b2 = _stream_base(seed, 2 * stream), _stream_base(seed, 2 * stream + 1)

    def fill(lo, hi):
        r = np.sqrt(-2.0 * np.log(_unit(_u64_range(b1, lo, hi))))
        a = 2.0 * np.pi * _unit(_u64_range(b2, lo, hi))
        z[2 * lo:2 * hi:2] = r * np.cos(a) * std + mean
        z[2 * lo + 1:2 * hi:2] = r * np.sin(a) * std + mean

    _chunked(half, fill)
    return z[:n]


def bf16(values: np.ndarray, shape) -> torch.Tensor:
    """Double values stored as a BF16 tensor (FP32, then RN-even to BF16)."""
    return torch.from_numpy(values.astype(np.float32)).reshape(shape).to(torch.bfloat16)


def topk_experts(seed: int, stream: int, b: int, num_experts: int, K: int) -> np.ndarray:
    """[b, K] distinct expert ids per token, uniform without replacement."""
    keys = uniform(seed, stream, b * num_experts).reshape(b, num_experts)
    return np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int64)


def softmax_weights(seed: int, stream: int, b: int, K: int) -> torch.Tensor:
    """FP32 [b, K] route weights: softmax over the token's K N(0,1) logits
    (computed in double, rounded once to FP32)."""
    logits = normal(seed, stream, b * K).reshape(b, K)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    return torch.from_numpy((e / e.sum(axis=1, keepdims=True)).astype(np.float32))


def expert_major_order(experts: np.ndarray) -> np.ndarray:
    """Route (t, k) -> its position when the routes are sorted by expert, then
    token, then k (the permuted GEMM2 row order of an MoE layer)."""
    b, K = experts.shape
    flat = experts.reshape(-1)
    order = np.lexsort((np.arange(b * K), flat))
    pos = np.empty(b * K, dtype=np.int64)
    pos[order] = np.arange(b * K)
    return pos.reshape(b, K)


def ep_finalize_inputs(seed: int, *, b: int, tp: int, P: int, K: int, num_experts: int,
                       outlier_frac: float = 0.0, weight_before_norm: bool = True,
                       gamma_std: float = 0.1, gain_center: float = 1.0, eps: float = 1e-6) -> dict:
    """EP finalize inputs.

    Experts e live on slot e // (num_experts / tp).  Token t's K experts are
    uniform without replacement; slot s holds, grouped by expert then token,
    the GEMM2 rows of the routes whose expert it owns.  rows is BF16
    [tp, rows_per_slot, P] N(0,1) (rows_per_slot = the largest slot's count;
    the shorter slots' tail rows are random and never referenced);
    idx[s, t, k] is the route's row in slot s, or -1 where slot s does not own
    it.  round(outlier_frac * b * K) route rows, chosen by seed, are multiplied
    by 8 (exact in BF16).  Route weights FP32 softmax; gamma BF16
    N(0, gamma_std^2)."""
    assert num_experts % tp == 0
    per_slot = num_experts // tp
    experts = topk_experts(seed, 1, b, num_experts, K)
    slot_of = experts // per_slot
    counts = [int((slot_of == s).sum()) for s in range(tp)]
    rows_per_slot = max(1, max(counts))
    idx = np.full((tp, b, K), -1, dtype=np.int32)
    for s in range(tp):
        mask = slot_of == s
        ts, ks = np.nonzero(mask)
        order = np.lexsort((ks, ts, experts[ts, ks]))
        for r, o in enumerate(order):
            idx[s, ts[o], ks[o]] = r
    rows = bf16(normal(seed, 2, tp * rows_per_slot * P), (tp, rows_per_slot, P))
    n_out = int(round(outlier_frac * b * K))
    if n_out:  # scaled after rounding to BF16, so the x8 is exact
        pick = np.argsort(uniform(seed, 3, b * K), kind="stable")[:n_out]
        for p in pick:
            t, k = divmod(int(p), K)
            s = int(slot_of[t, k])
            rows[s, int(idx[s, t, k])] *= 8
    return dict(
        rows=rows, rows_per_slot=rows_per_slot, idx=torch.from_numpy(idx),
        w=softmax_weights(seed, 4, b, K),
        gamma=bf16(normal(seed, 5, P, std=gamma_std), (P,)),
        gain_center=gain_center, eps=eps, weight_before_norm=weight_before_norm,
        b=b, tp=tp, K=K, P=P, experts=torch.from_numpy(experts),
    )


def tp_finalize_inputs(seed: int, *, b: int, tp: int, P: int, K: int, num_experts: int = 128,
                       partial_std: float = 0.35, weight_before_norm: bool = True,
                       gamma_std: float = 0.1, gain_center: float = 1.0, eps: float = 1e-6) -> dict:
    """Expert-TP finalize inputs: every slot holds a K-partial of every route
    row.  partials BF16 [tp, b*K, P] N(0, partial_std^2), rows grouped by
    expert then token; idx[t, k] is route (t, k)'s row (shared by all slots);
    route weights FP32 softmax; gamma BF16 N(0, gamma_std^2)."""
    experts = topk_experts(seed, 1, b, num_experts, K)
    idx = expert_major_order(experts).astype(np.int32)
    num_rows = b * K
    return dict(
        partials=bf16(normal(seed, 2, tp * num_rows * P, std=partial_std), (tp, num_rows, P)),
        num_rows=num_rows, idx=torch.from_numpy(idx),
        w=softmax_weights(seed, 4, b, K),
        gamma=bf16(normal(seed, 5, P, std=gamma_std), (P,)),
        gain_center=gain_center, eps=eps, weight_before_norm=weight_before_norm,
        b=b, tp=tp, K=K, P=P,
    )


def latent_up_inputs(seed: int, *, b: int, tp: int = 8, L: int = 3584, H: int = 7168,
                     tp_s: int = 8, latent_std: float = 0.5, shared_std: float = 0.5,
                     w_std: float = 0.02, eps: float = 1e-6, with_weight: bool = True) -> dict:
    """Latent tail inputs: latent partials BF16 [tp, b, L] N(0, latent_std^2)
    (the finalized top-16 rows' latent partials of each slot), gamma BF16
    1 + N(0, 0.05^2), W_up BF16 [H, L] N(0, w_std^2) row-major, shared-expert
    partials BF16 [tp_s, b, H] N(0, shared_std^2)."""
    d = dict(
        latent=bf16(normal(seed, 10, tp * b * L, std=latent_std), (tp, b, L)),
        gamma=bf16(normal(seed, 11, L, std=0.05, mean=1.0), (L,)),
        shared=bf16(normal(seed, 12, tp_s * b * H, std=shared_std), (tp_s, b, H)) if tp_s else None,
        eps=eps, b=b, tp=tp, L=L, H=H, tp_s=tp_s,
    )
    if with_weight:
        d["w_up"] = bf16(normal(seed, 13, H * L, std=w_std), (H, L))
    return d


def shared_expert_inputs(seed: int, *, b: int, H: int = 7168, I: int = 6144,
                         w_std: float = 0.02, with_weights: bool = True) -> dict:
    """Fused shared expert inputs: x BF16 [b, H] N(0,1); W_gate, W_up BF16
    [I, H] and W_down BF16 [H, I], all N(0, w_std^2), row-major."""
    d = dict(x=bf16(normal(seed, 20, b * H), (b, H)), b=b, H=H, I=I)
    if with_weights:
        d["w_gate"] = bf16(normal(seed, 21, I * H, std=w_std), (I, H))
        d["w_up"] = bf16(normal(seed, 22, I * H, std=w_std), (I, H))
        d["w_down"] = bf16(normal(seed, 23, H * I, std=w_std), (H, I))
    return d


SEED_BASE = 0x5EED0000


def config(i: int, **overrides) -> dict:
    """The i-th decode workload (1-based), seeded with 0x5EED0000 + i.

    1 EP finalize, tiny: b=4, tp=2, P=512, top-4 of 8 experts (4 per slot).
    2 EP finalize, decode: b=64, tp=8, P=4096, top-8 of 128 experts (16 per
      slot), 1% of route rows x8.
    3 Expert-TP finalize: b=128, tp=8, P=4096, top-8, partials N(0, 0.35^2).
    4 Latent tail + up-projection: b=16, latent [8,16,3584], W_up [7168,3584],
      shared partials [8,16,7168].
    5 Fused shared expert: b=64, H=7168, I=6144 (added into the latent tail's
      output at b=64)."""
    seed = SEED_BASE + i
    if i == 1:
        kw = dict(b=4, tp=2, P=512, K=4, num_experts=8)
        kw.update(overrides)
        return ep_finalize_inputs(seed, **kw)
    if i == 2:
        kw = dict(b=64, tp=8, P=4096, K=8, num_experts=128, outlier_frac=0.01)
        kw.update(overrides)
        return ep_finalize_inputs(seed, **kw)
    if i == 3:
        kw = dict(b=128, tp=8, P=4096, K=8)
        kw.update(overrides)
        return tp_finalize_inputs(seed, **kw)
    if i == 4:
        kw = dict(b=16)
        kw.update(overrides)
        return latent_up_inputs(seed, **kw)
    if i == 5:
        kw = dict(b=64)
        kw.update(overrides)
        return shared_expert_inputs(seed, **kw)
    raise ValueError(f"no workload {i}")
