"""Stored oracle outputs (tests/golden/*.txt, written by
tests/golden/make_golden.py from oracle/ and the seeded generators only).
On the CPU the oracle must still reproduce every stored bit (a change to its
arithmetic has to be deliberate); on the GPU the finalize outputs and the
latent norm's y must equal the stored bits."""
import importlib.util
import os

import numpy as np
import pytest
import torch

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "make_golden.py"))
make_golden = importlib.util.module_from_spec(spec)
spec.loader.exec_module(make_golden)


def stored(name):
    """{label: uint16 array} of a stored fixture."""
    out, label, rows = {}, None, []
    for line in open(os.path.join(HERE, f"{name}.txt")):
        if line.startswith("#"):
            continue
        parts = line.split()
        if parts and not all(len(p) == 4 for p in parts):  # "label [shape] sha256 ..."
            if label:
                out[label] = np.array(rows, dtype=np.uint16)
            label, rows = parts[0], []
        else:
            rows.append([int(p, 16) for p in parts])
    out[label] = np.array(rows, dtype=np.uint16)
    return out


def test_oracle_reproduces_the_stored_outputs():
    import oracle

    oracle.build()
    cases = list(make_golden.cases())
    # every stored fixture is recomputed (none silently skipped)
    assert sorted(c[0] for c in cases) == sorted(f[:-4] for f in os.listdir(HERE) if f.endswith(".txt"))
    for name, desc, tensors in cases:
        expect = open(os.path.join(HERE, f"{name}.txt")).read()
        assert make_golden.render(name, desc, tensors) == expect, f"{name}: the oracle's output changed"


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


@pytest.mark.gpu
def test_gpu_finalize_and_latent_norm_match_the_stored_bits():
    import moe_decode_tail_gb300 as mt
    from moe_decode_tail_gb300 import build as cuda_build
    from moe_decode_tail_gb300 import synth

    cuda_build.build()
    dev = "cuda"
    for name, kw in (("ep_config1", dict()), ("ep_config1_wan", dict(weight_before_norm=False))):
        d = synth.config(1, **kw)
        out = torch.empty((d["b"], d["P"]), dtype=torch.bfloat16, device=dev)
        mt.moe_tail_ep_finalize(d["rows"].to(dev), d["idx"].to(dev), d["w"].to(dev), d["gamma"].to(dev), out,
                                gain_center=d["gain_center"], eps=d["eps"], weight_before_norm=d["weight_before_norm"])
        assert np.array_equal(_bits(out), stored(name)["out"]), name
    d = synth.config(3, b=4, tp=2, P=512, K=4)
    out = torch.empty((4, 512), dtype=torch.bfloat16, device=dev)
    mt.moe_tail_tp_finalize(d["partials"].to(dev), d["idx"].to(dev), d["w"].to(dev), d["gamma"].to(dev), out,
                            gain_center=d["gain_center"], eps=d["eps"], weight_before_norm=True)
    assert np.array_equal(_bits(out), stored("tp_small")["out"])
    d = synth.latent_up_inputs(0x5EED0004, b=3, tp=2, L=512, H=384, tp_s=2)
    y = torch.empty((3, 512), dtype=torch.bfloat16, device=dev)
    mt.moe_tail_latent_norm(d["latent"].to(dev), d["gamma"].to(dev), y, eps=d["eps"])
    assert np.array_equal(_bits(y), stored("latent_small")["y"])
    assert mt.moe_tail_take_device_error() == 0
