"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/moe_tail_oracle.c (a sum in
the wrong order, a rounding dropped or added, a term, a sign or an operand
moved), builds the copy with the oracle's flags, and runs the pins
(tests/test_oracle_pins.py) against it in a child process, which must fail.
The unchanged copy must pass.  The copies run side by side, one child
each.  Only the copies are changed; the oracle itself is not touched."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_tail_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (what the mistake is, text in the oracle, what it becomes); the first match is changed
MUTATIONS = [
    ("EP slots summed in reverse order",
     "for (int s = 0; s < tp; ++s) {\n            for (int c = 0; c < P; ++c) part[c] = 0.0f;",
     "for (int s = tp - 1; s >= 0; --s) {\n            for (int c = 0; c < P; ++c) part[c] = 0.0f;"),
    ("EP slot partial not rounded to BF16", "o[c] = o[c] + bf16_round(part[c]);", "o[c] = o[c] + part[c];"),
    ("EP routes summed in reverse order",
     "for (int k = 0; k < K; ++k) {\n                int32_t j = idx[((int64_t)s * b + t) * K + k];",
     "for (int k = K - 1; k >= 0; --k) {\n                int32_t j = idx[((int64_t)s * b + t) * K + k];"),
    ("gain placement of weight_before_norm swapped", "float n = wbn ? v[c] * inv : (x[c] * inv) * g[c];",
     "float n = wbn ? (x[c] * inv) * g[c] : v[c] * inv;"),
    ("product order (x * inv) * g changed", "float n = wbn ? v[c] * inv : (x[c] * inv) * g[c];",
     "float n = wbn ? v[c] * inv : x[c] * (inv * g[c]);"),
    ("lane columns strided instead of contiguous", "int col = 256 * c + 8 * l + i;", "int col = 256 * c + l + 32 * i;"),
    ("butterfly offsets in reverse order", "for (int off = 1; off < 32; off <<= 1) {",
     "for (int off = 16; off >= 1; off >>= 1) {"),
    ("chunk sums folded in reverse order",
     "for (int c = 0; c < chunks; ++c) {\n        float a[32], nb[32];",
     "for (int c = chunks - 1; c >= 0; --c) {\n        float a[32], nb[32];"),
    ("a lane's columns added in reverse order", "for (int i = 0; i < 8; ++i) {\n                int col",
     "for (int i = 7; i >= 0; --i) {\n                int col"),
    ("eps dropped", "float den = mean + eps;", "float den = mean;"),
    ("mean by division instead of the rounded reciprocal", "float mean = ss * rcp;", "float mean = ss / (float)P;"),
    ("inverse RMS as sqrt of a reciprocal", "return 1.0f / sqrtf(den);", "return sqrtf(1.0f / den);"),
    ("-0 not made +0 in the expert-TP output", "out[(int64_t)t * P + c] = pz(oracle_bf16_from_f32(acc[c]));",
     "out[(int64_t)t * P + c] = oracle_bf16_from_f32(acc[c]);"),
    ("row 0 treated as not local", "if (j < 0 || (int64_t)j >= rows_per_slot) continue;",
     "if (j <= 0 || (int64_t)j >= rows_per_slot) continue;"),
    ("gain center not added", "for (int c = 0; c < P; ++c) g[c] = oracle_f32_from_bf16(gamma[c]) + gain_center;",
     "for (int c = 0; c < P; ++c) g[c] = oracle_f32_from_bf16(gamma[c]);"),
    ("expert-TP slot sum not rounded to BF16",
     "                x[c] = bf16_round(sum);\n            }\n            add_normalised_route",
     "                x[c] = sum;\n            }\n            add_normalised_route"),
    ("latent tail skips the first shared slot", "for (int s = 0; s < tp_s; ++s)", "for (int s = 1; s < tp_s; ++s)"),
    ("SiLU with the wrong sign", "double silu = gate / (1.0 + exp(-gate));", "double silu = gate / (1.0 + exp(gate));"),
    ("h multiplies gate instead of up", "pz(oracle_bf16_from_f64(silu * up))", "pz(oracle_bf16_from_f64(silu * gate))"),
    ("d added into out before its BF16 rounding",
     "float sum = oracle_f32_from_bf16(*o) + oracle_f32_from_bf16(db);", "float sum = oracle_f32_from_bf16(*o) + (float)acc;"),
    ("BF16 ties rounded away from zero", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;",
     "if (rest >= 0x8000u) keep += 1u;"),
    ("BF16 from binary64 through a plain binary32 rounding", "        u |= 1u; /* the odd one of the two neighbours */",
     "        u |= 0u;"),
    ("latent slot sum not rounded to BF16",
     "            x[c] = bf16_round(sum);\n        }\n        float inv",
     "            x[c] = sum;\n        }\n        float inv"),
    ("latent y as x * (inv * gamma)", "float n = (x[c] * inv) * oracle_f32_from_bf16(gamma[c]);",
     "float n = x[c] * (inv * oracle_f32_from_bf16(gamma[c]));"),
    ("latent y without gamma", "float n = (x[c] * inv) * oracle_f32_from_bf16(gamma[c]);", "float n = x[c] * inv;"),
    ("expert-TP routes summed in reverse order",
     "for (int k = 0; k < K; ++k) {\n            int32_t j = idx[(int64_t)t * K + k];",
     "for (int k = K - 1; k >= 0; --k) {\n            int32_t j = idx[(int64_t)t * K + k];"),
    ("expert-TP slots summed in reverse order",
     "for (int s = 0; s < tp; ++s)\n                    sum = sum + oracle_f32_from_bf16(partials",
     "for (int s = tp - 1; s >= 0; --s)\n                    sum = sum + oracle_f32_from_bf16(partials"),
    ("BF16 route weights read as FP32", "return w_is_bf16 ? oracle_f32_from_bf16(((const uint16_t*)w)[i]) : ((const float*)w)[i];",
     "return ((const float*)w)[i / 2];"),
    ("up-projection rounds through FP32", "out[(int64_t)t * H + n] = pz(oracle_bf16_from_f64(acc));",
     "out[(int64_t)t * H + n] = pz(oracle_bf16_from_f32((float)acc));"),
    ("gate not rounded to BF16 before SiLU", "double gate = oracle_f32_from_bf16(oracle_bf16_from_f64(ga));",
     "double gate = ga;"),
    ("latent y keeps -0", "y[(int64_t)t * L + c] = pz(oracle_bf16_from_f32(n));",
     "y[(int64_t)t * L + c] = oracle_bf16_from_f32(n);"),
    ("h rounded through binary32", "h_out[(int64_t)t * I + i] = pz(oracle_bf16_from_f64(silu * up));",
     "h_out[(int64_t)t * I + i] = pz(oracle_bf16_from_f32((float)(silu * up)));"),
    ("down output keeps -0", "uint16_t db = pz(oracle_bf16_from_f64(acc));", "uint16_t db = oracle_bf16_from_f64(acc);"),
    ("expert-TP ignores weight_before_norm",
     "add_normalised_route(x, g, wbn, eps, route_weight(w, w_is_bf16, (int64_t)t * K + k), P,",
     "add_normalised_route(x, g, 1, eps, route_weight(w, w_is_bf16, (int64_t)t * K + k), P,"),
    ("expert-TP row num_rows treated as local", "if (j < 0 || (int64_t)j >= num_rows) continue;",
     "if (j < 0 || (int64_t)j > num_rows) continue;"),
    ("latent out keeps -0", "out[(int64_t)t * H + n] = pz(oracle_bf16_from_f64(acc));",
     "out[(int64_t)t * H + n] = oracle_bf16_from_f64(acc);"),
    ("latent shared slots accumulated in binary32",
     "acc += (double)oracle_f32_from_bf16(shared[((int64_t)s * b + t) * H + n]);",
     "acc = (float)(acc + (double)oracle_f32_from_bf16(shared[((int64_t)s * b + t) * H + n]));"),
    ("latent norm without eps", "float inv = inverse_rms(oracle_sum_of_squares(x, L), L, eps);",
     "float inv = inverse_rms(oracle_sum_of_squares(x, L), L, 0.0f);"),
    ("h keeps -0", "h_out[(int64_t)t * I + i] = pz(oracle_bf16_from_f64(silu * up));",
     "h_out[(int64_t)t * I + i] = oracle_bf16_from_f64(silu * up);"),
    ("SiLU rounded to binary32", "double silu = gate / (1.0 + exp(-gate));",
     "double silu = (float)(gate / (1.0 + exp(-gate)));"),
    ("gate rounded through binary32", "double gate = oracle_f32_from_bf16(oracle_bf16_from_f64(ga));",
     "double gate = oracle_f32_from_bf16(oracle_bf16_from_f32((float)ga));"),
    ("up rounded through binary32", "double up = oracle_f32_from_bf16(oracle_bf16_from_f64(ua));",
     "double up = oracle_f32_from_bf16(oracle_bf16_from_f32((float)ua));"),
    ("d rounded through binary32", "uint16_t db = pz(oracle_bf16_from_f64(acc));",
     "uint16_t db = pz(oracle_bf16_from_f32((float)acc));"),
]
# indexing, layout and formula slips
MUTATIONS += [
    ("sum of squares over the gained row when the gains follow the norm",
     "for (int c = 0; c < P; ++c) v[c] = wbn ? x[c] * g[c] : x[c];", "for (int c = 0; c < P; ++c) v[c] = x[c] * g[c];"),
    ("gains dropped after the norm", "float n = wbn ? v[c] * inv : (x[c] * inv) * g[c];",
     "float n = wbn ? v[c] * inv : (x[c] * inv);"),
    ("gains applied twice before the norm", "float n = wbn ? v[c] * inv : (x[c] * inv) * g[c];",
     "float n = wbn ? (v[c] * inv) * g[c] : (x[c] * inv) * g[c];"),
    ("expert-TP sum not reset per token", "        for (int c = 0; c < P; ++c) acc[c] = 0.0f;\n", ""),
    ("EP output sum not reset per token", "        for (int c = 0; c < P; ++c) o[c] = 0.0f;\n", ""),
    ("EP slot partial not reset per slot", "            for (int c = 0; c < P; ++c) part[c] = 0.0f;\n", ""),
    ("EP index of token 0", "int32_t j = idx[((int64_t)s * b + t) * K + k];", "int32_t j = idx[((int64_t)s * b) * K + k];"),
    ("EP index token-major", "int32_t j = idx[((int64_t)s * b + t) * K + k];",
     "int32_t j = idx[((int64_t)t * tp + s) * K + k];"),
    ("EP rows of slot 0 for every slot", "const uint16_t* row = rows + ((int64_t)s * rows_per_slot + j) * P;",
     "const uint16_t* row = rows + ((int64_t)j) * P;"),
    ("expert-TP index of token 0", "int32_t j = idx[(int64_t)t * K + k];", "int32_t j = idx[(int64_t)k];"),
    ("expert-TP partials of slot 0 for every slot",
     "sum = sum + oracle_f32_from_bf16(partials[((int64_t)s * num_rows + j) * P + c]);",
     "sum = sum + oracle_f32_from_bf16(partials[((int64_t)j) * P + c]);"),
    ("route weight divides", "        float p = n * w;\n", "        float p = n / w;\n"),
    ("latent gamma of column 0", "float n = (x[c] * inv) * oracle_f32_from_bf16(gamma[c]);",
     "float n = (x[c] * inv) * oracle_f32_from_bf16(gamma[0]);"),
    ("latent mean over L + 1", "float inv = inverse_rms(oracle_sum_of_squares(x, L), L, eps);",
     "float inv = inverse_rms(oracle_sum_of_squares(x, L), L + 1, eps);"),
    ("W_up read transposed",
     "const uint16_t* wr = w_up + (int64_t)n * L;\n            double acc = 0.0;\n"
     "            for (int c = 0; c < L; ++c) acc += yd[c] * (double)oracle_f32_from_bf16(wr[c]);",
     "const uint16_t* wr = w_up + (int64_t)n;\n            double acc = 0.0;\n"
     "            for (int c = 0; c < L; ++c) acc += yd[c] * (double)oracle_f32_from_bf16(wr[(int64_t)c * H]);"),
    ("W_gate and W_up swapped",
     "const uint16_t* gr = w_gate + (int64_t)i * H;\n            const uint16_t* ur = w_up + (int64_t)i * H;",
     "const uint16_t* gr = w_up + (int64_t)i * H;\n            const uint16_t* ur = w_gate + (int64_t)i * H;"),
    ("W_down read transposed",
     "const uint16_t* dr = w_down + (int64_t)n * I;\n            double acc = 0.0;\n"
     "            for (int i = 0; i < I; ++i) acc += hd[i] * (double)oracle_f32_from_bf16(dr[i]);",
     "const uint16_t* dr = w_down + (int64_t)n;\n            double acc = 0.0;\n"
     "            for (int i = 0; i < I; ++i) acc += hd[i] * (double)oracle_f32_from_bf16(dr[(int64_t)i * H]);"),
    ("accumulate drops the old out", "float sum = oracle_f32_from_bf16(*o) + oracle_f32_from_bf16(db);",
     "float sum = oracle_f32_from_bf16(db);"),
    ("SiLU's exponent taken of up", "double silu = gate / (1.0 + exp(-gate));", "double silu = gate / (1.0 + exp(-up));"),
]

# roundings fused or moved
MUTATIONS += [
    ("each square fused into the lane's add", "                float sq = e * e;\n                acc = acc + sq;",
     "                acc = (float)((double)acc + (double)e * (double)e);"),
    ("EP running slot sum rounded to BF16", "o[c] = o[c] + bf16_round(part[c]);", "o[c] = bf16_round(o[c] + part[c]);"),
    ("expert-TP running slot sum rounded to BF16",
     "sum = sum + oracle_f32_from_bf16(partials[((int64_t)s * num_rows + j) * P + c]);",
     "sum = bf16_round(sum + oracle_f32_from_bf16(partials[((int64_t)s * num_rows + j) * P + c]));"),
    ("route product rounded to BF16", "        float p = n * w;\n", "        float p = bf16_round(n * w);\n"),
    ("normalised value rounded to BF16", "        float n = wbn ? v[c] * inv : (x[c] * inv) * g[c];\n",
     "        float n = bf16_round(wbn ? v[c] * inv : (x[c] * inv) * g[c]);\n"),
    ("gains rounded to BF16", "for (int c = 0; c < P; ++c) g[c] = oracle_f32_from_bf16(gamma[c]) + gain_center;",
     "for (int c = 0; c < P; ++c) g[c] = bf16_round(oracle_f32_from_bf16(gamma[c]) + gain_center);"),
    ("inverse RMS in double", "    return 1.0f / sqrtf(den);", "    return (float)(1.0 / sqrt((double)den));"),
]

# Mistakes that cannot change any result are not listed.  Examples: dropping
# the -0 -> +0 step of the EP output or of the accumulated down output (both
# sums start from +0 and add BF16 values, so neither can be -0 or a nonzero
# value below the smallest BF16 subnormal); starting the expert-TP slot sum
# from -0 (a -0 row changes neither the sum of squares nor the +0-started
# route sum); forming 1/P or mean + eps in double and rounding once to
# binary32 (double carries more than 2 * 24 + 2 bits, so one operation
# rounded twice is still correctly rounded).


def build_copy(tmp_path, source: str, name: str) -> str:
    src = tmp_path / f"{name}.c"
    src.write_text(source)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib), str(src), "-lm"], check=True, capture_output=True)
    return str(lib)


def run_pins(lib: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, MOE_TAIL_ORACLE_LIBRARY=lib, PYTHONPATH=ROOT)
    return subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                          capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every copy (the unchanged one under the key None, then each mutant)
    built and run against the pins, the child processes side by side."""
    from concurrent.futures import ThreadPoolExecutor

    source = open(SRC).read()
    names = [m[0] for m in MUTATIONS]
    assert len(set(names)) == len(names), "two mutations share a name"
    copies = [(None, source)]
    for what, old, new in MUTATIONS:
        assert old in source, f"mutation site not found: {what}"
        copies.append((what, source.replace(old, new, 1)))
    tmp = tmp_path_factory.mktemp("oracle_copies")

    def run(i_copy):
        i, (what, text) = i_copy
        return what, run_pins(build_copy(tmp, text, f"copy{i}"))

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as pool:
        return dict(pool.map(run, enumerate(copies)))


def test_unchanged_copy_passes_the_pins(outcomes):
    r = outcomes[None]
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("what", [m[0] for m in MUTATIONS])
def test_pins_catch_the_mistake(outcomes, what):
    # pytest exits 1 when tests fail; a crash or an error of the run itself
    # (another code) does not count as a pin catching the mistake
    r = outcomes[what]
    assert r.returncode == 1, f"no pin fails with: {what} (exit {r.returncode})\n{r.stdout[-1500:]}"
