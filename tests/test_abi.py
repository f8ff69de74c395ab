"""The C ABI library: it builds, loads, exports exactly what include/moe_tail.h
declares, and refuses bad arguments on the host before any CUDA call (these
tests pass fake device addresses and never launch anything)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from moe_decode_tail_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_tail.h")
EINVAL, OK = 1, 0
FAKE = 0x7F0000000000  # a 4 KiB-aligned address no call may dereference

# The refusal tests hand the library fake device addresses: run them only where
# no GPU is visible, so a regression in the checks can never launch on them.
host_only = pytest.mark.skipif(torch.cuda.is_available(), reason="fake device addresses: host-only")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    import moe_decode_tail_gb300 as mt

    return mt.lib()


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_\w+)\s*\(", text, re.M)))


def test_header_declares_the_four_calls_and_helpers():
    names = declared()
    for n in ("moe_tail_ep_finalize", "moe_tail_tp_finalize", "moe_tail_latent_up", "moe_shared_expert",
              "moe_tail_workspace_bytes", "moe_tail_status_str", "moe_tail_take_device_error"):
        assert n in names


@pytest.mark.parametrize("lang", [["gcc", "-std=c99", "-x", "c"], ["g++", "-std=c++17", "-x", "c++"]])
def test_headers_compile_as_c_and_cxx(tmp_path, lang):
    # a plain C (and C++) consumer of the ABI: both headers, no warnings
    src = tmp_path / "consumer.c"
    src.write_text('#include "moe_tail.h"\n#include "moe_tail_trace.h"\n#include "moe_tail_floor.h"\n'
                   "int main(void) { return moe_tail_workspace_bytes(0, 1, 8) == 0 ? 1 : 0; }\n")
    inc = os.path.join(ROOT, "include")
    subprocess.run(lang[:2] + ["-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I", inc] + lang[2:]
                   + [str(src)], check=True, capture_output=True)


def test_c_program_links_and_calls_the_host_entries(tmp_path, lib):
    # a C program linked against the library calls the entries that need no
    # device: workspace sizes, status strings, and a refused call (b = 0 with
    # null pointers succeeds; a bad size is refused before any CUDA call)
    src = tmp_path / "host.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "moe_tail.h"
int main(void) {
  if (moe_tail_workspace_bytes(0, 16, 3584) < (size_t)16 * 3584 * 2) return 1;
  if (moe_tail_workspace_bytes(2, 16, 3584) != 0) return 2;
  if (strlen(moe_tail_status_str(MOE_TAIL_EINVAL)) == 0) return 3;
  if (moe_tail_latent_up(0, 0, 1e-6f, 0, 0, 0, 0, 1, 8, 8, 0, 0, 0, 0) != MOE_TAIL_OK) return 4;
  if (moe_tail_latent_up(0, 0, 1e-6f, 0, 0, 0, 1, 0, 8, 8, 0, 0, 0, 0) != MOE_TAIL_EINVAL) return 5;
  puts("ok");
  return 0;
}
""")
    exe = tmp_path / "host"
    libdir = os.path.dirname(cuda_build.LIB)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe), cuda_build.LIB, "-Wl,-rpath," + libdir], check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)


def test_library_exports_every_declared_symbol(lib):
    for n in declared():
        assert hasattr(lib, n), n


def test_library_exports_nothing_else():
    out = subprocess.run(["nm", "-D", "--defined-only", cuda_build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.split() and line.split()[-2] in "TtDdBbRr"}
    exported = {e for e in exported if not e.startswith("_")}
    assert exported == set(declared())


def a(x=0):
    return ctypes.c_void_p(FAKE + x)


def ep(lib, **kw):
    args = dict(rows=a(), rps=16, idx=a(), w=a(), wd=0, gamma=a(), gc=1.0, eps=1e-6, wbn=1, b=4, tp=2, K=4, P=512,
                out=a(1 << 20), stream=None)
    args.update(kw)
    return lib.moe_tail_ep_finalize(args["rows"], args["rps"], args["idx"], args["w"], args["wd"], args["gamma"],
                                    args["gc"], args["eps"], args["wbn"], args["b"], args["tp"], args["K"], args["P"],
                                    args["out"], args["stream"])


def tp(lib, **kw):
    args = dict(q=a(), rows=16, idx=a(), w=a(), wd=0, gamma=a(), gc=1.0, eps=1e-6, wbn=1, b=4, tp=2, K=4, P=512,
                out=a(1 << 20), stream=None)
    args.update(kw)
    return lib.moe_tail_tp_finalize(args["q"], args["rows"], args["idx"], args["w"], args["wd"], args["gamma"],
                                    args["gc"], args["eps"], args["wbn"], args["b"], args["tp"], args["K"], args["P"],
                                    args["out"], args["stream"])


@host_only
@pytest.mark.parametrize("fn", [ep, tp])
@pytest.mark.parametrize("bad", [
    dict(tp=0), dict(tp=33), dict(K=0), dict(K=33), dict(P=7), dict(P=4), dict(P=516 + 2), dict(P=32776),
    dict(b=-1), dict(b=65536), dict(wd=2), dict(gamma=None), dict(out=None), dict(w=None), dict(idx=None),
    dict(out=a(8)), dict(gamma=a(4)), dict(idx=a(2)), dict(w=a(2)),
    dict(out=a(0)),  # out overlaps the rows / partials
])
def test_finalize_refuses_bad_arguments(lib, fn, bad):
    assert fn(lib, **bad) == EINVAL


@host_only
@pytest.mark.parametrize("fn", [ep, tp])
def test_finalize_b_zero_does_nothing(lib, fn):
    # b = 0 succeeds without touching memory, even with null pointers
    assert fn(lib, b=0, rows=None, idx=None, w=None, gamma=None, out=None) == OK if fn is ep else \
        fn(lib, b=0, q=None, idx=None, w=None, gamma=None, out=None) == OK


@host_only
def test_bf16_weights_need_only_2_byte_alignment_but_fp32_need_4(lib):
    assert ep(lib, w=a(2), wd=0) == EINVAL
    # with BF16 weights a 2-byte aligned pointer passes the checks; moving out
    # to overlap the gamma vector is refused instead, so nothing launches
    assert ep(lib, w=a(2), wd=1, out=a(0), rps=0, rows=None) == EINVAL


def fin_flags(lib, which, **kw):
    args = dict(rows=a(), n=8, idx=a(1 << 24), w=a(2 << 24), wd=0, gamma=a(3 << 24), gc=1.0, eps=1e-6, wbn=1, b=4,
                tp=2, K=4, P=512, out=a(4 << 24), flags=2, stream=None)
    args.update(kw)
    fn = lib.moe_tail_ep_finalize_flags if which == "ep" else lib.moe_tail_tp_finalize_flags
    return fn(args["rows"], args["n"], args["idx"], args["w"], args["wd"], args["gamma"], args["gc"], args["eps"],
              args["wbn"], args["b"], args["tp"], args["K"], args["P"], args["out"], args["flags"], args["stream"])


@host_only
@pytest.mark.parametrize("which", ["ep", "tp"])
@pytest.mark.parametrize("bad", [dict(flags=1), dict(flags=4), dict(flags=-1), dict(tp=0), dict(P=100),
                                 dict(idx=None), dict(out=a(3 << 24))])
def test_finalize_flags_refuse_bad_arguments(lib, which, bad):
    assert fin_flags(lib, which, **bad) == EINVAL


@host_only
@pytest.mark.parametrize("which", ["ep", "tp"])
def test_finalize_flags_b_zero(lib, which):
    assert fin_flags(lib, which, b=0, rows=None, idx=None, w=None, out=None) == OK


def latent(lib, **kw):
    args = dict(lat=a(), gamma=a(1 << 28), eps=1e-6, w=a(2 << 28), sh=a(3 << 28), tp_s=8, b=16, tp=8, L=3584, H=7168,
                out=a(4 << 28), ws=a(5 << 28), wsb=16 * 3584 * 2, stream=None)
    args.update(kw)
    return lib.moe_tail_latent_up(args["lat"], args["gamma"], args["eps"], args["w"], args["sh"], args["tp_s"],
                                  args["b"], args["tp"], args["L"], args["H"], args["out"], args["ws"], args["wsb"],
                                  args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(tp=0), dict(tp_s=-1), dict(tp_s=33), dict(L=3583), dict(H=7170), dict(L=4), dict(b=-2),
    dict(sh=None), dict(tp_s=0), dict(ws=None), dict(wsb=16 * 3584 * 2 - 1), dict(out=a(5 << 28)),
    dict(ws=a(4 << 28)), dict(lat=a(3)), dict(w=a(8)), dict(L=40000),
])
def test_latent_up_refuses_bad_arguments(lib, bad):
    assert latent(lib, **bad) == EINVAL


@host_only
def test_latent_up_b_zero(lib):
    assert latent(lib, b=0, lat=None, w=None, out=None, ws=None) == OK


def norm(lib, **kw):
    args = dict(lat=a(), gamma=a(1 << 24), eps=1e-6, b=16, tp=8, L=3584, y=a(2 << 24), flags=0, stream=None)
    args.update(kw)
    return lib.moe_tail_latent_norm(args["lat"], args["gamma"], args["eps"], args["b"], args["tp"], args["L"],
                                    args["y"], args["flags"], args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(tp=0), dict(tp=33), dict(L=3583), dict(L=4), dict(L=40000), dict(b=-1), dict(b=65536), dict(lat=None),
    dict(gamma=None), dict(y=None), dict(y=a(8)), dict(lat=a(4)), dict(y=a(16)),  # y over the latent partials
    dict(flags=1), dict(flags=4), dict(flags=-1),
])
def test_latent_norm_refuses_bad_arguments(lib, bad):
    assert norm(lib, **bad) == EINVAL


def up(lib, **kw):
    args = dict(y=a(), w=a(1 << 28), sh=a(2 << 28), tp_s=8, b=16, L=3584, H=7168, out=a(3 << 28), flags=0,
                stream=None)
    args.update(kw)
    return lib.moe_tail_up_project(args["y"], args["w"], args["sh"], args["tp_s"], args["b"], args["L"], args["H"],
                                   args["out"], args["flags"], args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(tp_s=-1), dict(tp_s=33), dict(L=3583), dict(H=7170), dict(H=4), dict(b=-2), dict(sh=None), dict(tp_s=0),
    dict(y=None), dict(w=None), dict(out=None), dict(flags=2), dict(flags=-1), dict(out=a(8)),
    dict(out=a(2 << 28)), dict(out=a(16)),  # out over shared, over y
])
def test_up_project_refuses_bad_arguments(lib, bad):
    assert up(lib, **bad) == EINVAL


@host_only
def test_latent_steps_b_zero(lib):
    assert norm(lib, b=0, lat=None, gamma=None, y=None, flags=2) == OK
    assert up(lib, b=0, y=None, w=None, out=None, flags=1) == OK


def latent_flags(lib, **kw):
    args = dict(lat=a(), gamma=a(1 << 28), eps=1e-6, w=a(2 << 28), sh=a(3 << 28), tp_s=8, b=16, tp=8, L=3584,
                H=7168, out=a(4 << 28), y=a(5 << 28), flags=3, stream=None)
    args.update(kw)
    return lib.moe_tail_latent_up_flags(args["lat"], args["gamma"], args["eps"], args["w"], args["sh"],
                                        args["tp_s"], args["b"], args["tp"], args["L"], args["H"], args["out"],
                                        args["y"], args["flags"], args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(tp=0), dict(tp_s=33), dict(L=3583), dict(H=7170), dict(b=-1), dict(sh=None), dict(tp_s=0),
    dict(y=None), dict(lat=None), dict(out=None), dict(flags=4), dict(flags=-1), dict(y=a(8)),
    dict(y=a(4 << 28)), dict(y=a(16)), dict(out=a(5 << 28)), dict(y=a(3 << 28)),  # y over out, latent, shared
])
def test_latent_up_flags_refuses_bad_arguments(lib, bad):
    assert latent_flags(lib, **bad) == EINVAL


@host_only
def test_latent_up_flags_b_zero(lib):
    assert latent_flags(lib, b=0, lat=None, w=None, out=None, y=None) == OK


def noalloc(lib, **kw):
    args = dict(lat=a(), gamma=a(1 << 28), eps=1e-6, w=a(2 << 28), sh=a(3 << 28), tp_s=8, b=16, tp=8, L=3584,
                H=7168, out=a(4 << 28), stream=None)
    args.update(kw)
    return lib.moe_tail_latent_up_noalloc(args["lat"], args["gamma"], args["eps"], args["w"], args["sh"],
                                          args["tp_s"], args["b"], args["tp"], args["L"], args["H"], args["out"],
                                          args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(tp=0), dict(tp=33), dict(tp_s=-1), dict(tp_s=33), dict(L=3583), dict(L=4), dict(L=40000), dict(H=7170),
    dict(H=4), dict(H=(1 << 24) + 8), dict(b=-2), dict(b=65536), dict(sh=None), dict(tp_s=0), dict(lat=None),
    dict(gamma=None), dict(w=None), dict(out=None), dict(lat=a(3)), dict(w=a(8)), dict(out=a(8)),
    dict(out=a(16)), dict(out=a(3 << 28)),  # out over the latent, over shared
    dict(b=147),  # y (147 x 3584 BF16) larger than the built-in 1 MiB scratch
])
def test_latent_up_noalloc_refuses_bad_arguments(lib, bad):
    assert noalloc(lib, **bad) == EINVAL


@host_only
def test_latent_up_noalloc_b_zero(lib):
    assert noalloc(lib, b=0, lat=None, gamma=None, w=None, out=None) == OK


def shared(lib, **kw):
    args = dict(x=a(), wg=a(1 << 28), wu=a(2 << 28), wd=a(3 << 28), b=64, H=7168, I=6144, out=a(4 << 28), acc=1,
                ws=a(5 << 28), wsb=64 * 6144 * 2, stream=None)
    args.update(kw)
    return lib.moe_shared_expert(args["x"], args["wg"], args["wu"], args["wd"], args["b"], args["H"], args["I"],
                                 args["out"], args["acc"], args["ws"], args["wsb"], args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(H=7169), dict(I=6140 + 2), dict(H=0), dict(b=-1), dict(x=None), dict(wd=None), dict(ws=None),
    dict(wsb=64 * 6144 * 2 - 2), dict(out=a(0)), dict(ws=a(4 << 28)), dict(x=a(8)), dict(out=a(4 << 28 | 8)),
])
def test_shared_expert_refuses_bad_arguments(lib, bad):
    assert shared(lib, **bad) == EINVAL


def gate_up(lib, **kw):
    args = dict(x=a(), wg=a(1 << 28), wu=a(2 << 28), b=64, H=7168, I=6144, h=a(3 << 28), flags=0, stream=None)
    args.update(kw)
    return lib.moe_shared_gate_up(args["x"], args["wg"], args["wu"], args["b"], args["H"], args["I"], args["h"],
                                  args["flags"], args["stream"])


def down(lib, **kw):
    args = dict(h=a(), wd=a(1 << 28), b=64, H=7168, I=6144, out=a(2 << 28), acc=1, flags=0, stream=None)
    args.update(kw)
    return lib.moe_shared_down(args["h"], args["wd"], args["b"], args["H"], args["I"], args["out"], args["acc"],
                               args["flags"], args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(H=7169), dict(I=6142), dict(b=-1), dict(x=None), dict(wu=None), dict(h=None), dict(h=a(8)),
    dict(h=a(16)), dict(flags=4), dict(flags=7), dict(wg=a(4)),  # h over x
])
def test_shared_gate_up_refuses_bad_arguments(lib, bad):
    assert gate_up(lib, **bad) == EINVAL


@host_only
@pytest.mark.parametrize("bad", [
    dict(H=4), dict(I=6150), dict(b=65536), dict(h=None), dict(wd=None), dict(out=None), dict(out=a(8)),
    dict(out=a(16)), dict(flags=4), dict(h=a(2)),  # out over h
])
def test_shared_down_refuses_bad_arguments(lib, bad):
    assert down(lib, **bad) == EINVAL


def down_persistent(lib, **kw):
    args = dict(h=a(), wd=a(1 << 28), b=64, H=7168, I=6144, out=a(2 << 28), acc=1, ctas=0, flags=0, stream=None)
    args.update(kw)
    return lib.moe_shared_down_persistent(args["h"], args["wd"], args["b"], args["H"], args["I"], args["out"],
                                          args["acc"], args["ctas"], args["flags"], args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(H=4), dict(I=6150), dict(b=65536), dict(h=None), dict(wd=None), dict(out=None), dict(out=a(8)),
    dict(out=a(16)), dict(flags=2), dict(h=a(2)), dict(ctas=-1), dict(ctas=65536),  # out over h
])
def test_shared_down_persistent_refuses_bad_arguments(lib, bad):
    assert down_persistent(lib, **bad) == EINVAL


@host_only
def test_shared_down_persistent_b_zero(lib):
    assert down_persistent(lib, b=0, h=None, out=None, flags=1, ctas=65535) == OK


@host_only
def test_shared_steps_b_zero(lib):
    assert gate_up(lib, b=0, x=None, h=None) == OK
    assert gate_up(lib, b=0, x=None, h=None, flags=3) == OK  # both promises are valid flags
    assert down(lib, b=0, h=None, out=None, flags=1) == OK


def test_workspace_bytes(lib):
    assert lib.moe_tail_workspace_bytes(0, 16, 3584) == 16 * 3584 * 2
    assert lib.moe_tail_workspace_bytes(1, 3, 100) == 768  # rounded up to 256 bytes
    assert lib.moe_tail_workspace_bytes(2, 3, 100) == 0
    assert lib.moe_tail_workspace_bytes(0, -1, 100) == 0


def test_status_strings(lib):
    assert lib.moe_tail_status_str(0) == b"ok"
    assert lib.moe_tail_status_str(1) == b"invalid argument"
    assert lib.moe_tail_status_str(99) == b"unknown status"


@host_only
@pytest.mark.parametrize("name", ["ep", "tp", "fin_flags_ep", "fin_flags_tp", "latent", "norm", "up", "latent_flags",
                                  "noalloc", "shared", "gate_up", "down"])
def test_default_arguments_pass_every_check(lib, name):
    # Each refusal test changes one argument of these defaults, so the defaults
    # themselves must be accepted: with no GPU visible the call then fails at its
    # first CUDA call (MOE_TAIL_ECUDA, or ENOTSUP where a tensor map cannot be
    # encoded), never with EINVAL.
    if name.startswith("fin_flags_"):
        rc = fin_flags(lib, name[len("fin_flags_"):])
    else:
        rc = globals()[name](lib)
    assert rc in (2, 3), rc


def test_binding_has_every_declared_call_under_the_same_name():
    import moe_decode_tail_gb300 as mt

    missing = [n for n in declared() if not callable(getattr(mt, n, None))]
    assert not missing, missing
    assert set(declared()) <= set(mt.__all__)


@host_only
def test_width_caps_are_exact(lib):
    # H (and I) up to 2^24 pass the checks and 2^24 + 8 is refused, as the
    # header states; shapes are kept small elsewhere (L = 8, b = 1, no shared
    # partials) so that no buffer overlaps another at the cap
    cap = 1 << 24
    for n, want in ((cap, (2, 3)), (cap + 8, (EINVAL,))):
        assert latent(lib, H=n, L=8, b=1, tp_s=0, sh=None, wsb=lib.moe_tail_workspace_bytes(0, 1, 8)) in want
        assert up(lib, H=n, L=8, b=1, tp_s=0, sh=None) in want
        assert latent_flags(lib, H=n, L=8, b=1, tp_s=0, sh=None) in want
        assert noalloc(lib, H=n, L=8, b=1, tp_s=0, sh=None) in want
        assert shared(lib, H=n, I=8, b=1, wsb=lib.moe_tail_workspace_bytes(1, 1, 8)) in want
        assert shared(lib, H=8, I=n, b=1, wsb=max(256, 2 * n)) in want
        assert gate_up(lib, H=n, I=8, b=1) in want
        assert gate_up(lib, H=8, I=n, b=1) in want
        assert down(lib, H=n, I=8, b=1) in want
        assert down(lib, H=8, I=n, b=1) in want


@host_only
def test_token_cap_is_exact(lib):
    for b, want in ((65535, (2, 3)), (65536, (EINVAL,))):
        assert ep(lib, b=b, out=a(1 << 30)) in want
        assert norm(lib, b=b, L=8, y=a(1 << 30)) in want
        assert shared(lib, b=b, H=8, I=8, wsb=-(-16 * b // 256) * 256) in want
        assert gate_up(lib, b=b, H=8, I=8) in want
        assert down(lib, b=b, H=8, I=8) in want


def test_kernel_form_accepts_known_forms_and_refuses_the_rest(lib):
    # host-side only: the setting is a process-wide value, no CUDA call
    lib.moe_tail_set_kernel_form.argtypes = [ctypes.c_int, ctypes.c_int]
    for call in (0, 1, 2):  # MOE_TAIL_FORM_EP, _TP, _LATENT
        for form in (0, 1, 2):
            assert lib.moe_tail_set_kernel_form(call, form) == OK
        assert lib.moe_tail_set_kernel_form(call, 3) == EINVAL
        assert lib.moe_tail_set_kernel_form(call, -1) == EINVAL
        assert lib.moe_tail_set_kernel_form(call, 0) == OK  # back to the library's choice
    assert lib.moe_tail_set_kernel_form(3, 0) == EINVAL
    assert lib.moe_tail_set_kernel_form(-1, 0) == EINVAL


def _floor_lib():
    cuda_build.build(floor=True)
    fl = ctypes.CDLL(cuda_build.FLOOR_LIB)
    P_, i32 = ctypes.c_void_p, ctypes.c_int
    fl.moe_tail_floor_empty.argtypes = [i32, i32, i32, i32, P_]
    fl.moe_tail_floor_read.argtypes = [P_, ctypes.c_size_t, i32, i32, i32, i32, P_, P_]
    fl.moe_tail_floor_gather.argtypes = [P_, i32, P_, ctypes.c_int64, i32, i32, i32, i32, P_, P_]
    return fl


def test_floor_library_exports_exactly_its_header():
    # the measurement-only library: the three calls of include/moe_tail_floor.h, nothing else
    _floor_lib()
    out = subprocess.run(["nm", "-D", "--defined-only", cuda_build.FLOOR_LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.split() and line.split()[-2] in "TtDdBbRr"}
    exported = {e for e in exported if not e.startswith("_")}
    header = open(os.path.join(ROOT, "include", "moe_tail_floor.h")).read()
    assert exported == set(re.findall(r"^int (moe_tail_floor_\w+)\(", header, re.M))
    assert exported == {"moe_tail_floor_empty", "moe_tail_floor_read", "moe_tail_floor_gather"}


@host_only
def test_floor_calls_refuse_bad_shapes_before_launching():
    fl = _floor_lib()
    ok = a()
    for gx, gy, thr, cl in ((0, 1, 32, 1), (2, 0, 32, 1), (2, 1, 33, 1), (2, 1, 2048, 1), (2, 1, 800, 1),
                            (3, 1, 32, 2), (16, 1, 32, 16)):
        assert fl.moe_tail_floor_empty(gx, gy, thr, cl, None) == 1
        assert fl.moe_tail_floor_read(ok, 4096, gx, gy, thr, cl, ok, None) == 1
        assert fl.moe_tail_floor_gather(ok, 8, ok, 16, gx, gy, thr, cl, ok, None) == 1
    # bad sizes and pointers: a size not a multiple of 16, more than one trip's worth, null or misaligned
    assert fl.moe_tail_floor_read(ok, 4008, 2, 1, 32, 1, ok, None) == 1
    assert fl.moe_tail_floor_read(ok, 2 * 32 * 16 * 16 + 16, 2, 1, 32, 1, ok, None) == 1
    assert fl.moe_tail_floor_read(None, 4096, 2, 1, 32, 1, ok, None) == 1
    assert fl.moe_tail_floor_read(a(8), 4096, 2, 1, 32, 1, ok, None) == 1
    assert fl.moe_tail_floor_gather(ok, 0, ok, 16, 2, 1, 32, 1, ok, None) == 1
    assert fl.moe_tail_floor_gather(a(2), 8, ok, 16, 2, 1, 32, 1, ok, None) == 1
    # valid shapes pass the checks and then fail at the launch without a GPU
    assert fl.moe_tail_floor_empty(2, 64, 256, 2, None) == 2
    assert fl.moe_tail_floor_read(ok, 4096, 2, 1, 32, 1, ok, None) == 2


def up_sd(lib, **kw):
    args = dict(y=a(), w=a(1 << 28), sh=a(2 << 28), tp_s=8, h=a(3 << 28), wd=a(4 << 28), b=64, L=3584, I=6144,
                H=7168, out=a(5 << 28), d=a(6 << 28), flags=1, stream=None)
    args.update(kw)
    lib.moe_tail_up_project_shared_down.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] + [ctypes.c_void_p] * 2 + \
        [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_void_p]
    return lib.moe_tail_up_project_shared_down(args["y"], args["w"], args["sh"], args["tp_s"], args["h"], args["wd"],
                                               args["b"], args["L"], args["I"], args["H"], args["out"], args["d"],
                                               args["flags"], args["stream"])


@host_only
@pytest.mark.parametrize("bad", [
    dict(tp_s=-1), dict(tp_s=33), dict(L=3583), dict(I=6140), dict(I=4), dict(I=(1 << 24) + 8), dict(H=7170),
    dict(H=4), dict(b=-2), dict(b=65536), dict(sh=None), dict(tp_s=0), dict(y=None), dict(w=None), dict(h=None),
    dict(wd=None), dict(out=None), dict(flags=2), dict(flags=-1), dict(out=a(8)), dict(d=a(8)), dict(h=a(4)),
    dict(out=a(2 << 28)), dict(out=a(16)), dict(out=a(3 << 28)), dict(out=a(4 << 28)),  # out over shared, y, h, w_down
    dict(d=a(1 << 28)), dict(d=a(3 << 28)), dict(d=a(5 << 28)),  # d over w_up, h, out
])
def test_up_project_shared_down_refuses_bad_arguments(lib, bad):
    assert up_sd(lib, **bad) == EINVAL


@host_only
def test_up_project_shared_down_accepts_its_defaults_and_b_zero(lib):
    # the defaults pass every check (then fail at the first CUDA call without a
    # GPU); b = 0 succeeds with null pointers; no shared partials and no d_out
    # are both allowed
    assert up_sd(lib) in (2, 3)
    assert up_sd(lib, sh=None, tp_s=0, d=None) in (2, 3)
    assert up_sd(lib, b=0, y=None, w=None, sh=None, tp_s=0, h=None, wd=None, out=None, d=None) == OK
