"""The algorithmic bytes bench.py divides by: each workload's count, from its
sizes, equals the figure worked out by hand from the workload definitions
(route rows, indices, weights, gains and outputs once; the latent tail's
partials, W_up, shared partials and output; the shared expert's weights, x,
h written and read, out read and written)."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_bytes", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name,sizes,expect", [
    ("ep", dict(b=4, tp=2, K=4, P=512), 21_696),                      # EP tiny
    ("ep", dict(b=64, tp=8, K=8, P=4096), 4_745_216),                 # EP decode
    ("tp", dict(b=128, tp=8, K=8, P=4096), 68_173_824),               # expert-TP
    ("latent", dict(b=16, tp=8, tp_s=8, L=3584, H=7168), 54_369_280),  # latent tail + up-projection
    ("shared", dict(b=64, H=7168, I=6144), 268_566_528),              # shared expert into out
])
def test_config_bytes_match_the_hand_counts(bench, name, sizes, expect):
    assert bench.config_bytes(name, sizes) == expect


def test_step_bytes_at_b64(bench):
    # one b = 64 step: EP rows 4,194,304 + idx 16,384 + w 2,048 + gamma 8,192 + out 524,288;
    # expert-TP partials 33,554,432 + idx 2,048 + w 2,048 + gamma 8,192 + out 524,288;
    # latent partials 3,670,016 + gamma 7,168 + W_up 51,380,224 + shared 7,340,032 + out 917,504;
    # shared expert weights 264,241,152 + x 917,504 + out read and written 1,835,008
    assert bench.BYTES == {"ep_finalize": 4_745_216, "tp_finalize": 34_091_008, "latent_up": 63_314_944,
                           "shared_expert": 266_993_664}
