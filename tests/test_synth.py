"""The seeded input generators (moe_decode_tail_gb300/synth.py) against their
published definitions and the workloads' stated structure.

SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) seeded with 0 starts 0xE220A8397B1DCDAF,
0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC,
0x1B39896A51A8749B; the counter-based form here must give the same words.
The rest checks what the workloads state: uniforms in (0, 1), Box-Muller
normals with the requested moments, distinct top-K experts, routing tables
that place every route exactly once, the outlier count, and determinism
(including across the threaded chunks of a long draw)."""
import numpy as np
import pytest

from moe_decode_tail_gb300 import synth


def test_splitmix64_matches_the_published_sequence_from_seed_zero():
    words = synth._u64_range(np.uint64(0), 1, 6)
    assert [int(x) for x in words] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
                                       0xF88BB8A8724C81EC, 0x1B39896A51A8749B]


def test_draws_are_deterministic_and_chunking_does_not_change_them():
    n = synth._CHUNK + 1000  # two threaded chunks
    a = synth.u64(7, 3, n)
    b = synth.u64(7, 3, n)
    assert np.array_equal(a, b)
    # the tail of the long draw equals a draw of the same counters alone
    base = synth._stream_base(7, 3)
    assert np.array_equal(a[-1000:], synth._u64_range(base, n - 1000, n))
    assert not np.array_equal(synth.u64(7, 4, 1000), a[:1000])  # streams differ


def test_uniform_and_normal_moments():
    u = synth.uniform(11, 1, 200_000)
    assert u.min() > 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.005 and abs(u.var() - 1.0 / 12.0) < 0.002
    z = synth.normal(11, 2, 200_001, std=0.35, mean=1.0)
    assert z.shape == (200_001,)
    assert abs(z.mean() - 1.0) < 0.005 and abs(z.std() - 0.35) < 0.005
    # the cosine and sine halves of Box-Muller are each N(mean, std^2)
    assert abs(z[0::2].std() - 0.35) < 0.006 and abs(z[1::2].std() - 0.35) < 0.006


def test_topk_experts_are_distinct_and_uniform():
    e = synth.topk_experts(5, 1, 4000, 128, 8)
    assert e.shape == (4000, 8)
    assert all(len(set(row)) == 8 for row in e)
    counts = np.bincount(e.reshape(-1), minlength=128)
    assert counts.min() > 0.75 * counts.mean() and counts.max() < 1.25 * counts.mean()


@pytest.mark.parametrize("i", [1, 2])
def test_ep_routing_table_places_every_route_once(i):
    d = synth.config(i)
    b, tp, K, P = d["b"], d["tp"], d["K"], d["P"]
    idx, experts = d["idx"].numpy(), d["experts"].numpy()
    per_slot = {1: 4, 2: 16}[i]
    assert d["rows"].shape == (tp, d["rows_per_slot"], P)
    for t in range(b):
        for k in range(K):
            owner = experts[t, k] // per_slot
            local = [s for s in range(tp) if 0 <= idx[s, t, k] < d["rows_per_slot"]]
            assert local == [owner]  # exactly the owning slot holds the route
    for s in range(tp):  # each slot's rows 0..n-1 are used once each
        used = sorted(int(j) for j in idx[s].reshape(-1) if j >= 0)
        assert used == list(range(len(used)))
    assert d["rows_per_slot"] == max(max(len([j for j in idx[s].reshape(-1) if j >= 0]) for s in range(tp)), 1)


def test_config_2_scales_one_percent_of_the_route_rows_by_eight():
    d = synth.config(2)
    plain = synth.config(2, outlier_frac=0.0)
    diff = (d["rows"].float() != plain["rows"].float()).any(dim=2)
    assert int(diff.sum()) == round(0.01 * 64 * 8)  # 5 of 512 route rows
    ratio = d["rows"].float()[diff] / plain["rows"].float()[diff]
    assert bool(((ratio == 8) | (plain["rows"].float()[diff] == 0)).all())


def test_expert_tp_rows_are_grouped_by_expert_then_token():
    d = synth.config(3, b=32)
    idx = d["idx"].numpy()
    assert d["partials"].shape == (8, 32 * 8, 4096)
    assert sorted(idx.reshape(-1).tolist()) == list(range(32 * 8))  # a permutation of the rows
    experts = synth.topk_experts(synth.SEED_BASE + 3, 1, 32, 128, 8)
    order = sorted(((experts[t, k], t, k) for t in range(32) for k in range(8)))
    assert [idx[t, k] for _, t, k in order] == list(range(32 * 8))


def test_route_weights_are_a_softmax_per_token():
    w = synth.softmax_weights(9, 4, 64, 8).numpy()
    assert w.dtype == np.float32 and w.shape == (64, 8)
    assert np.all(w > 0) and np.allclose(w.sum(axis=1), 1.0, atol=1e-6)


def test_workload_shapes():
    c4 = synth.config(4)
    assert c4["latent"].shape == (8, 16, 3584) and c4["w_up"].shape == (7168, 3584)
    assert c4["shared"].shape == (8, 16, 7168) and c4["gamma"].shape == (3584,)
    c5 = synth.config(5, with_weights=False)
    assert c5["x"].shape == (64, 7168) and (c5["H"], c5["I"]) == (7168, 6144)
    with pytest.raises(ValueError):
        synth.config(6)
