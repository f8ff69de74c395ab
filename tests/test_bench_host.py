"""Host-side pieces of bench.py that need no GPU: the argument defaults keep
the timing contract, the end-to-end leg's packed buffers lay the step's
activations out aligned, without overlap, with the copied region ending before
the shared expert's output slot, the reference arm (the oracle on the host)
prints one contract line on rank 0 only, and the CUDA arm refuses to run
without a device."""
import importlib.util
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_defaults_keep_the_timing_contract(bench, monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    assert a.gpus == 1 and a.impl == "cuda" and a.warmup >= 3 and a.steps >= 1000
    assert a.composition == "two_branch_fused" and not a.sequential


def test_packed_layout_of_the_step_inputs(bench):
    B, TP, P, K, L, H = bench.B, bench.TP, bench.P, bench.K_ROUTES, bench.L, bench.H
    bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
    named = [("ep_rows", torch.empty((TP, 65, P), dtype=bf)), ("ep_idx", torch.empty((TP, B, K), dtype=i32)),
             ("ep_w", torch.empty((B, K), dtype=f32)), ("tp_part", torch.empty((TP, B * K, P), dtype=bf)),
             ("tp_idx", torch.empty((B, K), dtype=i32)), ("tp_w", torch.empty((B, K), dtype=f32)),
             ("latent", torch.empty((TP, B, L), dtype=bf)), ("x", torch.empty((B, H), dtype=bf)),
             ("shared9", torch.empty((TP + 1, B, H), dtype=bf))]
    offs, total = bench.packed_layout(named)
    spans = sorted((offs[k], offs[k] + t.numel() * t.element_size()) for k, t in named)
    assert all(o % 256 == 0 for o in offs.values())
    assert all(a_end <= b_start for (_, a_end), (b_start, _) in zip(spans, spans[1:]))
    assert spans[-1][1] <= total < spans[-1][1] + 256
    # the step copies everything up to the end of the latent tail's TP shared slots
    h2d = offs["shared9"] + TP * B * H * 2
    assert h2d == spans[-1][1] - B * H * 2


def _run_bench(*argv, env=None):
    import subprocess

    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], capture_output=True, text=True,
                          env=e, cwd=ROOT, timeout=600)


def test_reference_arm_prints_one_contract_line():
    # the oracle timed on the host cores: one JSON line with the contract's
    # keys, its cpu_baseline describing this run and an e2e of its own value
    import json

    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", env={"WORLD_SIZE": "1", "RANK": "0"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3",
                   env={"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the refusal without a CUDA device")
def test_cuda_arm_refuses_to_run_without_a_device():
    # no CPU fallback: the CUDA arm exits non-zero and says why
    r = _run_bench("--steps", "1", "--warmup", "3")
    assert r.returncode != 0 and "no CUDA device" in (r.stderr + r.stdout)


def test_traffic_is_reported_only_for_the_sources_it_was_measured_on(bench, monkeypatch, tmp_path):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "roofline_traffic.txt").write_text(
        "# comment lines are skipped\nsources_sha256 abc123\ntraffic shared_expert 270426112\n"
        "traffic shared_gate_up 181474560\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: "abc123")
    assert bench.traffic_record("shared_expert") == 270426112
    assert bench.traffic_record("shared_gate_up") == 181474560
    assert bench.traffic_record("latent_up") is None  # not profiled
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: "changed")
    assert bench.traffic_record("shared_expert") is None
    (tmp_path / "profiles" / "roofline_traffic.txt").unlink()
    assert bench.traffic_record("shared_expert") is None


def test_step_call_tables_cover_each_composition(bench):
    # every composition's calls: event pairs inside the 12 per-step events, positive
    # bytes, and launches adding up to the step's kernel count
    side = object()
    for comp, launches in (("two_branch", 6), ("two_branch_one_call", 6), ("latent_main", 6),
                           ("two_branch_fused", 5)):
        t = bench.step_calls(comp, side)
        assert all(0 <= i < j < bench.EVENTS_PER_STEP for c in t.values() for i, j in c["pairs"])
        assert all(c["bytes"] > 0 for c in t.values())
        assert sum(c["launches"] for c in t.values()) == launches, comp
    assert sum(c["launches"] for c in bench.step_calls("two_branch", None).values()) == 6  # sequential
    # the step's algorithmic bytes: the sequential step's per-call figures minus
    # the shared expert's read and second write of out (367,309,824 at b = 64)
    seq = bench.step_calls("two_branch", None)
    assert bench.STEP_BYTES == sum(c["bytes"] for c in seq.values()) - 2 * bench.B * bench.H * 2 == 367_309_824


def test_code_only_drops_comments_but_not_code(bench):
    src = "int a; // one\n/* two\n   lines */\nint b;   \n\n  x = y / z;  /* tail */\n"
    assert bench.code_only(src) == "int a;\nint b;\n  x = y / z;"
    # a comment edit leaves the hash's input unchanged, a code edit does not
    assert bench.code_only(src.replace("one", "uno")) == bench.code_only(src)
    assert bench.code_only(src.replace("y / z", "y * z")) != bench.code_only(src)


def test_kernel_sources_hash_covers_the_gemm_sources(bench):
    # the hash is of the files that define the measured kernels and their launch
    csrc = os.path.join(ROOT, "moe_decode_tail_gb300", "csrc")
    assert all(os.path.exists(os.path.join(csrc, f)) for f in bench.GEMM_SOURCES)
    assert {"decode_gemm.cu", "moe_tail_api.cu"} <= set(bench.GEMM_SOURCES)
    assert len(bench.kernel_sources_hash()) == 64


def test_clock_samples_summarised(bench, tmp_path):
    # nvidia-smi's CSV (noheader, nounits): clocks.sm, clocks.max.sm, power.draw,
    # reasons.active, hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    csv = tmp_path / "clocks.csv"
    csv.write_text("2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
                   "2055, 2070, 1010.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
                   "2070, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active\n"
                   "garbage line\n"
                   "2040, 2070, 980.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s = bench.ClockSampler(0)
    s.proc, s.path = Done(), str(csv)
    r = s.stop()
    # four samples (the one without a power reading still counts its clock), median 2062.5
    assert r["samples"] == 4 and r["sm_mhz"] == 2062.5 and r["sm_max_mhz"] == 2070 and r["power_w_max"] == 1010.0
    assert r["reasons"] == ["sw_power_cap"]
    assert not csv.exists()


def test_clock_sampler_without_nvidia_smi_says_so(bench):
    s = bench.ClockSampler(0)
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]
