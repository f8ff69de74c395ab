"""Write the stored oracle outputs under tests/golden/ (run from the repo root:
python tests/golden/make_golden.py).  Calls only oracle/ and the seeded input
generators; the pages print no worked example, so these files pin the oracle
against itself over time: any change to its arithmetic changes a stored bit
and must be justified by the passage it follows."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from moe_decode_tail_gb300 import synth  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def cases():
    """(name, inputs description, list of (label, BF16 tensor)) for each fixture."""
    d = synth.config(1)
    yield "ep_config1", "synth.config(1): EP b=4 tp=2 P=512 top-4 of 8, weight_before_norm", [
        ("out", oracle.ep_finalize(d["rows"], d["rows_per_slot"], d["idx"], d["w"], d["gamma"], d["gain_center"],
                                   d["eps"], True, d["b"], d["tp"], d["K"], d["P"]))]
    d = synth.config(1, weight_before_norm=False)
    yield "ep_config1_wan", "synth.config(1, weight_before_norm=False)", [
        ("out", oracle.ep_finalize(d["rows"], d["rows_per_slot"], d["idx"], d["w"], d["gamma"], d["gain_center"],
                                   d["eps"], False, d["b"], d["tp"], d["K"], d["P"]))]
    d = synth.config(3, b=4, tp=2, P=512, K=4)
    yield "tp_small", "synth.config(3, b=4, tp=2, P=512, K=4): expert-TP", [
        ("out", oracle.tp_finalize(d["partials"], d["num_rows"], d["idx"], d["w"], d["gamma"], d["gain_center"],
                                   d["eps"], True, d["b"], d["tp"], d["K"], d["P"]))]
    d = synth.latent_up_inputs(0x5EED0004, b=3, tp=2, L=512, H=384, tp_s=2)
    y, out = oracle.latent_tail(d["latent"], d["gamma"], d["eps"], d["w_up"], d["shared"], 2, 3, 2, 512, 384)
    yield "latent_small", "synth.latent_up_inputs(0x5EED0004, b=3, tp=2, L=512, H=384, tp_s=2)", [("y", y), ("out", out)]
    s = synth.shared_expert_inputs(0x5EED0005, b=3, H=384, I=256)
    h, out = oracle.shared_expert(s["x"], s["w_gate"], s["w_up"], s["w_down"], 3, 384, 256,
                                  out_in=torch.zeros((3, 384), dtype=torch.bfloat16))
    yield "shared_small", "synth.shared_expert_inputs(0x5EED0005, b=3, H=384, I=256), out_in = 0", [("h", h), ("out", out)]


def render(name, desc, tensors) -> str:
    lines = [f"# {name}: {desc}", "# oracle output bits (BF16, row-major, hex), one row per line"]
    for label, t in tensors:
        bits = t.contiguous().view(torch.int16).numpy().astype("uint16")
        lines.append(f"{label} {list(t.shape)} sha256 {hashlib.sha256(bits.tobytes()).hexdigest()}")
        for row in bits.reshape(bits.shape[0], -1):
            lines.append(" ".join(f"{v:04x}" for v in row))
    return "\n".join(lines) + "\n"


def main():
    oracle.build()
    for name, desc, tensors in cases():
        with open(os.path.join(HERE, f"{name}.txt"), "w") as f:
            f.write(render(name, desc, tensors))
        print("wrote", name)


if __name__ == "__main__":
    main()
