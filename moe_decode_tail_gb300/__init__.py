"""GB300-native MoE decode tail: thin Python binding of libmoetail.so.

Every function here only marshals torch CUDA tensors into the C ABI of
``include/moe_tail.h`` (same names, sizes read from tensor shapes); all of the
tail's arithmetic runs in the library's CUDA kernels.  There is no CPU path:
if the library is missing or a call is refused, these functions raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

__all__ = [
    "MoeTailError", "lib", "moe_tail_ep_finalize", "moe_tail_tp_finalize", "moe_tail_latent_up",
    "moe_shared_expert", "moe_tail_workspace_bytes", "moe_tail_status_str", "moe_tail_take_device_error",
    "moe_tail_latent_up_noalloc", "NOALLOC_SCRATCH_BYTES", "moe_tail_selftest_wait_timeout",
    "moe_tail_latent_norm", "moe_tail_up_project", "WEIGHTS_STATIC", "INPUTS_READY",
    "moe_shared_gate_up", "moe_shared_down", "moe_tail_latent_up_flags", "moe_tail_ep_finalize_flags",
    "moe_tail_tp_finalize_flags", "moe_tail_set_kernel_form", "kernel_form", "FORM_EP", "FORM_TP", "FORM_LATENT",
    "FORM_LATENT_ONE_KERNEL", "moe_tail_set_stage_wait_limit", "moe_tail_up_project_shared_down",
    "moe_shared_down_persistent",
]

OK, EINVAL, ECUDA, ENOTSUP = 0, 1, 2, 3
NOALLOC_SCRATCH_BYTES = 1 << 20  # MOE_TAIL_NOALLOC_SCRATCH_BYTES
W_FP32, W_BF16 = 0, 1
WEIGHTS_STATIC = 1  # MOE_TAIL_WEIGHTS_STATIC
INPUTS_READY = 2  # MOE_TAIL_INPUTS_READY
FORM_EP, FORM_TP, FORM_LATENT = 0, 1, 2  # MOE_TAIL_FORM_*: the calls whose kernel form can be pinned
FORM_LATENT_ONE_KERNEL = 1  # MOE_TAIL_FORM_LATENT_ONE_KERNEL


class MoeTailError(RuntimeError):
    def __init__(self, name: str, status: int):
        super().__init__(f"{name}: {status_string(status)} ({status})")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built).  The
    MOE_TAIL_LIBRARY environment variable selects another build of it (the
    trace build, whose records moe_decode_tail_gb300.trace reads) before the first call."""
    global _lib
    if _lib is None:
        path = os.environ.get("MOE_TAIL_LIBRARY", LIB)
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with moe_decode_tail_gb300.build.build()")
        L = ctypes.CDLL(path)
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        fin = [P, i64, P, P, i32, P, f32, f32, i32, i32, i32, i32, i32, P, P]
        L.moe_tail_ep_finalize.argtypes = fin
        L.moe_tail_tp_finalize.argtypes = fin
        fin_flags = fin[:-1] + [i32, P]
        L.moe_tail_ep_finalize_flags.argtypes = fin_flags
        L.moe_tail_tp_finalize_flags.argtypes = fin_flags
        L.moe_tail_latent_up.argtypes = [P, P, f32, P, P, i32, i32, i32, i32, i32, P, P, sz, P]
        L.moe_shared_expert.argtypes = [P, P, P, P, i32, i32, i32, P, i32, P, sz, P]
        L.moe_tail_latent_up_noalloc.argtypes = [P, P, f32, P, P, i32, i32, i32, i32, i32, P, P]
        L.moe_tail_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
        L.moe_tail_latent_norm.argtypes = [P, P, f32, i32, i32, i32, P, i32, P]
        L.moe_tail_up_project.argtypes = [P, P, P, i32, i32, i32, i32, P, i32, P]
        L.moe_tail_latent_up_flags.argtypes = [P, P, f32, P, P, i32, i32, i32, i32, i32, P, P, i32, P]
        L.moe_shared_gate_up.argtypes = [P, P, P, i32, i32, i32, P, i32, P]
        L.moe_shared_down.argtypes = [P, P, i32, i32, i32, P, i32, i32, P]
        L.moe_shared_down_persistent.argtypes = [P, P, i32, i32, i32, P, i32, i32, i32, P]
        L.moe_tail_workspace_bytes.argtypes = [i32, i32, i32]
        L.moe_tail_workspace_bytes.restype = sz
        L.moe_tail_status_str.argtypes = [i32]
        L.moe_tail_status_str.restype = ctypes.c_char_p
        L.moe_tail_take_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.moe_tail_set_kernel_form.argtypes = [i32, i32]
        L.moe_tail_set_stage_wait_limit.argtypes = [ctypes.c_ulonglong]
        L.moe_tail_up_project_shared_down.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, P, P, i32, P]
        for name in ("moe_tail_ep_finalize", "moe_tail_tp_finalize", "moe_tail_latent_up", "moe_shared_expert",
                     "moe_tail_take_device_error", "moe_tail_latent_up_noalloc", "moe_tail_selftest_wait_timeout",
                     "moe_tail_latent_norm", "moe_tail_up_project", "moe_shared_gate_up", "moe_shared_down",
                     "moe_tail_latent_up_flags", "moe_tail_ep_finalize_flags", "moe_tail_tp_finalize_flags",
                     "moe_tail_set_kernel_form", "moe_tail_set_stage_wait_limit",
                     "moe_tail_up_project_shared_down", "moe_shared_down_persistent"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_tail_status_str(status).decode()


def _check(name: str, status: int) -> None:
    if status != OK:
        raise MoeTailError(name, status)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _dims(name: str, t, n: int) -> tuple:
    """The shape of t, which must have n dimensions."""
    if t.dim() != n:
        raise ValueError(f"{name} must have {n} dimensions, got shape {tuple(t.shape)}")
    return tuple(t.shape)


def _like(name: str, t, dtype, shape) -> None:
    """t must be dtype with exactly this shape: the C entry points receive only
    a pointer and take the layout from the sizes, so a tensor of another type
    or shape would be read (or written) as if it had this one."""
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _finalize_args(kind: str, src, permuted_idx, route_weights, gamma, out) -> tuple:
    """Shapes of a finalize call: src [tp, rows, P] BF16, route weights [b, K]
    FP32 or BF16, permuted_idx int32 [tp, b, K] (EP) or [b, K] (expert-TP),
    gamma BF16 [P], out BF16 [b, P].  Returns (tp, rows, P, b, K)."""
    tp, rows, P = _dims(kind, src, 3)
    b, K = _dims("route_weights", route_weights, 2)
    _like(kind, src, torch.bfloat16, (tp, rows, P))
    _weights(route_weights)
    _like("permuted_idx", permuted_idx, torch.int32, (tp, b, K) if kind == "rows" else (b, K))
    _like("gamma", gamma, torch.bfloat16, (P,))
    _like("out", out, torch.bfloat16, (b, P))
    _cuda(src, permuted_idx, route_weights, gamma, out)
    return tp, rows, P, b, K


def _latent_args(latent, gamma, w_up, shared, out, y) -> tuple:
    """Shapes of a latent-tail call: latent BF16 [tp, b, L], gamma BF16 [L],
    w_up BF16 [H, L], shared BF16 [tp_s, b, H] or None, out BF16 [b, H], y
    BF16 [b, L] or None.  Returns (tp, b, L, H, tp_s)."""
    tp, b, L = _dims("latent", latent, 3)
    H, _ = _dims("w_up", w_up, 2)
    tp_s = 0 if shared is None else _dims("shared", shared, 3)[0]
    _like("latent", latent, torch.bfloat16, (tp, b, L))
    _like("gamma", gamma, torch.bfloat16, (L,))
    _like("w_up", w_up, torch.bfloat16, (H, L))
    if shared is not None:
        _like("shared", shared, torch.bfloat16, (tp_s, b, H))
    _like("out", out, torch.bfloat16, (b, H))
    if y is not None:
        _like("y", y, torch.bfloat16, (b, L))
    _cuda(latent, gamma, w_up, shared, out, y)
    return tp, b, L, H, tp_s


def _weights(w: torch.Tensor) -> int:
    if w.dtype == torch.float32:
        return W_FP32
    if w.dtype == torch.bfloat16:
        return W_BF16
    raise ValueError("route weights must be FP32 or BF16")


def moe_tail_ep_finalize(rows, permuted_idx, route_weights, gamma, out, *, gain_center=1.0, eps=1e-6,
                         weight_before_norm=True, stream=None) -> torch.Tensor:
    """EP finalize into out (BF16 [b, P]); rows BF16 [tp, rows_per_slot, P],
    permuted_idx int32 [tp, b, K], route_weights [b, K], gamma BF16 [P]."""
    tp, rows_per_slot, P, b, K = _finalize_args("rows", rows, permuted_idx, route_weights, gamma, out)
    _check("moe_tail_ep_finalize", lib().moe_tail_ep_finalize(
        _p(rows), rows_per_slot, _p(permuted_idx), _p(route_weights), _weights(route_weights), _p(gamma),
        gain_center, eps, int(bool(weight_before_norm)), b, tp, K, P, _p(out), _stream(stream)))
    return out


def moe_tail_tp_finalize(partials, permuted_idx, route_weights, gamma, out, *, gain_center=1.0, eps=1e-6,
                         weight_before_norm=True, stream=None) -> torch.Tensor:
    """Expert-TP finalize into out (BF16 [b, P]); partials BF16 [tp, num_rows, P],
    permuted_idx int32 [b, K], route_weights [b, K], gamma BF16 [P]."""
    tp, num_rows, P, b, K = _finalize_args("partials", partials, permuted_idx, route_weights, gamma, out)
    _check("moe_tail_tp_finalize", lib().moe_tail_tp_finalize(
        _p(partials), num_rows, _p(permuted_idx), _p(route_weights), _weights(route_weights), _p(gamma),
        gain_center, eps, int(bool(weight_before_norm)), b, tp, K, P, _p(out), _stream(stream)))
    return out


def moe_tail_ep_finalize_flags(rows, permuted_idx, route_weights, gamma, out, *, gain_center=1.0, eps=1e-6,
                               weight_before_norm=True, inputs_ready=False, stream=None) -> torch.Tensor:
    """moe_tail_ep_finalize with the promise inputs_ready: rows, indices, route
    weights and gamma are not written by work still in flight on the stream."""
    tp, rows_per_slot, P, b, K = _finalize_args("rows", rows, permuted_idx, route_weights, gamma, out)
    _check("moe_tail_ep_finalize_flags", lib().moe_tail_ep_finalize_flags(
        _p(rows), rows_per_slot, _p(permuted_idx), _p(route_weights), _weights(route_weights), _p(gamma),
        gain_center, eps, int(bool(weight_before_norm)), b, tp, K, P, _p(out), INPUTS_READY if inputs_ready else 0,
        _stream(stream)))
    return out


def moe_tail_tp_finalize_flags(partials, permuted_idx, route_weights, gamma, out, *, gain_center=1.0, eps=1e-6,
                               weight_before_norm=True, inputs_ready=False, stream=None) -> torch.Tensor:
    """moe_tail_tp_finalize with the promise inputs_ready: partials, indices,
    route weights and gamma are not written by work still in flight on the stream."""
    tp, num_rows, P, b, K = _finalize_args("partials", partials, permuted_idx, route_weights, gamma, out)
    _check("moe_tail_tp_finalize_flags", lib().moe_tail_tp_finalize_flags(
        _p(partials), num_rows, _p(permuted_idx), _p(route_weights), _weights(route_weights), _p(gamma),
        gain_center, eps, int(bool(weight_before_norm)), b, tp, K, P, _p(out), INPUTS_READY if inputs_ready else 0,
        _stream(stream)))
    return out


def moe_tail_workspace_bytes(which: int, b: int, dim: int) -> int:
    return int(lib().moe_tail_workspace_bytes(which, b, dim))


def moe_tail_latent_up(latent, gamma, w_up, shared, out, workspace, *, eps=1e-6, stream=None) -> torch.Tensor:
    """Latent tail into out (BF16 [b, H]): latent BF16 [tp, b, L], gamma BF16 [L],
    w_up BF16 [H, L], shared BF16 [tp_s, b, H] or None, workspace uint8 CUDA
    tensor of at least moe_tail_workspace_bytes(0, b, L) bytes (y after the call)."""
    tp, b, L, H, tp_s = _latent_args(latent, gamma, w_up, shared, out, None)
    _cuda(workspace)
    _check("moe_tail_latent_up", lib().moe_tail_latent_up(
        _p(latent), _p(gamma), eps, _p(w_up), _p(shared), tp_s, b, tp, L, H, _p(out), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def moe_tail_latent_up_flags(latent, gamma, w_up, shared, out, y, *, eps=1e-6, inputs_ready=False,
                             weights_static=False, stream=None) -> torch.Tensor:
    """The latent tail into out (BF16 [b, H]) and y (BF16 [b, L]), with the
    split calls' promises: inputs_ready (latent and gamma, as for
    moe_tail_latent_norm) and weights_static (w_up, as for moe_tail_up_project).
    The norm and the up-projection, or with the latent tail's kernel form
    pinned to one kernel (moe_tail_set_kernel_form(FORM_LATENT, FORM_LATENT_ONE_KERNEL)) one kernel
    that forms y on chip (slower on GB300); the result is bit for bit that of
    the two split calls either way."""
    tp, b, L, H, tp_s = _latent_args(latent, gamma, w_up, shared, out, y)
    flags = (INPUTS_READY if inputs_ready else 0) | (WEIGHTS_STATIC if weights_static else 0)
    _check("moe_tail_latent_up_flags", lib().moe_tail_latent_up_flags(
        _p(latent), _p(gamma), eps, _p(w_up), _p(shared), tp_s, b, tp, L, H, _p(out), _p(y), flags,
        _stream(stream)))
    return out


def moe_tail_latent_norm(latent, gamma, y, *, eps=1e-6, inputs_ready=False, stream=None) -> torch.Tensor:
    """The latent tail's first step into y (BF16 [b, L]): the slot-summed latent
    BF16 [tp, b, L], RMS-normalised and scaled by gamma BF16 [L].
    inputs_ready: latent and gamma are not written by work still in flight on
    the stream, so the kernel may read them before the preceding kernel ends."""
    tp, b, L = _dims("latent", latent, 3)
    _like("latent", latent, torch.bfloat16, (tp, b, L))
    _like("gamma", gamma, torch.bfloat16, (L,))
    _like("y", y, torch.bfloat16, (b, L))
    _cuda(latent, gamma, y)
    _check("moe_tail_latent_norm", lib().moe_tail_latent_norm(
        _p(latent), _p(gamma), eps, b, tp, L, _p(y), INPUTS_READY if inputs_ready else 0, _stream(stream)))
    return y


def moe_tail_up_project(y, w_up, shared, out, *, weights_static=False, stream=None) -> torch.Tensor:
    """The latent tail's second step into out (BF16 [b, H]): y BF16 [b, L] times
    w_up BF16 [H, L] transposed, plus shared BF16 [tp_s, b, H] (or None).
    weights_static: w_up is not written by work still in flight on the stream,
    so the kernel may request weight tiles before the preceding kernel ends."""
    b, L = _dims("y", y, 2)
    H, _ = _dims("w_up", w_up, 2)
    tp_s = 0 if shared is None else _dims("shared", shared, 3)[0]
    _like("y", y, torch.bfloat16, (b, L))
    _like("w_up", w_up, torch.bfloat16, (H, L))
    if shared is not None:
        _like("shared", shared, torch.bfloat16, (tp_s, b, H))
    _like("out", out, torch.bfloat16, (b, H))
    _cuda(y, w_up, shared, out)
    _check("moe_tail_up_project", lib().moe_tail_up_project(
        _p(y), _p(w_up), _p(shared), tp_s, b, L, H, _p(out), WEIGHTS_STATIC if weights_static else 0,
        _stream(stream)))
    return out


def moe_tail_up_project_shared_down(y, w_up, shared, h, w_down, out, d_out=None, *, weights_static=False,
                                    stream=None) -> torch.Tensor:
    """The up-projection of y (BF16 [b, L]) with w_up (BF16 [H, L]) plus the
    shared partials (BF16 [tp_s, b, H] or None) plus bf16(d), d the down
    projection of h (BF16 [b, I]) with w_down (BF16 [H, I]), in one kernel,
    into out (BF16 [b, H]); d_out (BF16 [b, H], optional) receives bf16(d)."""
    b, L = _dims("y", y, 2)
    H, _ = _dims("w_up", w_up, 2)
    _, I = _dims("h", h, 2)
    tp_s = 0 if shared is None else _dims("shared", shared, 3)[0]
    _like("y", y, torch.bfloat16, (b, L))
    _like("w_up", w_up, torch.bfloat16, (H, L))
    if shared is not None:
        _like("shared", shared, torch.bfloat16, (tp_s, b, H))
    _like("h", h, torch.bfloat16, (b, I))
    _like("w_down", w_down, torch.bfloat16, (H, I))
    _like("out", out, torch.bfloat16, (b, H))
    if d_out is not None:
        _like("d_out", d_out, torch.bfloat16, (b, H))
    _cuda(y, w_up, shared, h, w_down, out, d_out)
    _check("moe_tail_up_project_shared_down", lib().moe_tail_up_project_shared_down(
        _p(y), _p(w_up), _p(shared), tp_s, _p(h), _p(w_down), b, L, I, H, _p(out), _p(d_out),
        WEIGHTS_STATIC if weights_static else 0, _stream(stream)))
    return out


def moe_shared_gate_up(x, w_gate, w_up, h, *, weights_static=False, inputs_ready=False, stream=None) -> torch.Tensor:
    """The shared expert's gate/up projection and SiLU into h (BF16 [b, I]):
    x BF16 [b, H], w_gate and w_up BF16 [I, H].  inputs_ready promises that x
    is not being written by work in flight on the stream (h is written only
    after that work ends)."""
    b, H = _dims("x", x, 2)
    I, _ = _dims("w_gate", w_gate, 2)
    _like("x", x, torch.bfloat16, (b, H))
    _like("w_gate", w_gate, torch.bfloat16, (I, H))
    _like("w_up", w_up, torch.bfloat16, (I, H))
    _like("h", h, torch.bfloat16, (b, I))
    _cuda(x, w_gate, w_up, h)
    _check("moe_shared_gate_up", lib().moe_shared_gate_up(
        _p(x), _p(w_gate), _p(w_up), b, H, I, _p(h),
        (WEIGHTS_STATIC if weights_static else 0) | (INPUTS_READY if inputs_ready else 0), _stream(stream)))
    return h


def moe_shared_down(h, w_down, out, *, accumulate=True, weights_static=False, stream=None) -> torch.Tensor:
    """The shared expert's down projection of h (BF16 [b, I]) with w_down BF16
    [H, I], written into out (BF16 [b, H]) or added into it (accumulate)."""
    b, I = _dims("h", h, 2)
    H, _ = _dims("w_down", w_down, 2)
    _like("h", h, torch.bfloat16, (b, I))
    _like("w_down", w_down, torch.bfloat16, (H, I))
    _like("out", out, torch.bfloat16, (b, H))
    _cuda(h, w_down, out)
    _check("moe_shared_down", lib().moe_shared_down(
        _p(h), _p(w_down), b, H, I, _p(out), int(bool(accumulate)), WEIGHTS_STATIC if weights_static else 0,
        _stream(stream)))
    return out


def moe_shared_down_persistent(h, w_down, out, *, accumulate=True, ctas=0, weights_static=False,
                               stream=None) -> torch.Tensor:
    """The down projection as a persistent kernel: ctas CTAs (0: one per output
    tile, at most one per SM) walk the output tiles over the whole K range with
    two alternating tensor-memory accumulators.  Same arguments and result as
    moe_shared_down, up to the order of d's FP32 sum."""
    b, I = _dims("h", h, 2)
    H, _ = _dims("w_down", w_down, 2)
    _like("h", h, torch.bfloat16, (b, I))
    _like("w_down", w_down, torch.bfloat16, (H, I))
    _like("out", out, torch.bfloat16, (b, H))
    _cuda(h, w_down, out)
    _check("moe_shared_down_persistent", lib().moe_shared_down_persistent(
        _p(h), _p(w_down), b, H, I, _p(out), int(bool(accumulate)), int(ctas),
        WEIGHTS_STATIC if weights_static else 0, _stream(stream)))
    return out


def moe_tail_latent_up_noalloc(latent, gamma, w_up, shared, out, *, eps=1e-6, stream=None) -> torch.Tensor:
    """The latent tail without a workspace, for callers that cannot allocate
    device memory (a plugin given only its input and output buffers, a host
    whose device memory is all held by its own pool, a path that must not
    call cudaMalloc): y lives in a fixed array of NOALLOC_SCRATCH_BYTES inside
    the library, shared by every call.  Same arguments as moe_tail_latent_up
    minus the workspace; b * L * 2 must not exceed NOALLOC_SCRATCH_BYTES.
    Calls that may overlap on the GPU race on the shared array."""
    tp, b, L, H, tp_s = _latent_args(latent, gamma, w_up, shared, out, None)
    if b * L * 2 > NOALLOC_SCRATCH_BYTES:
        raise ValueError(f"moe_tail_latent_up_noalloc: y needs {b * L * 2} bytes, more than the library's "
                         f"built-in {NOALLOC_SCRATCH_BYTES}-byte scratch; use moe_tail_latent_up with a workspace")
    _check("moe_tail_latent_up_noalloc", lib().moe_tail_latent_up_noalloc(
        _p(latent), _p(gamma), eps, _p(w_up), _p(shared), tp_s, b, tp, L, H, _p(out), _stream(stream)))
    return out


def moe_shared_expert(x, w_gate, w_up, w_down, out, workspace, *, accumulate=True, stream=None) -> torch.Tensor:
    """Fused shared expert into out (BF16 [b, H]): x BF16 [b, H], w_gate/w_up BF16
    [I, H], w_down BF16 [H, I], workspace of at least moe_tail_workspace_bytes(1, b, I)
    bytes (h after the call); out += down(...) when accumulate."""
    b, H = _dims("x", x, 2)
    I, _ = _dims("w_gate", w_gate, 2)
    _like("x", x, torch.bfloat16, (b, H))
    _like("w_gate", w_gate, torch.bfloat16, (I, H))
    _like("w_up", w_up, torch.bfloat16, (I, H))
    _like("w_down", w_down, torch.bfloat16, (H, I))
    _like("out", out, torch.bfloat16, (b, H))
    _cuda(x, w_gate, w_up, w_down, out, workspace)
    _check("moe_shared_expert", lib().moe_shared_expert(
        _p(x), _p(w_gate), _p(w_up), _p(w_down), b, H, I, _p(out), int(bool(accumulate)), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def moe_tail_status_str(status: int) -> str:
    return status_string(status)


def moe_tail_take_device_error() -> int:
    """Bits raised by bounded waits inside the kernels since the last read (0: none)."""
    bits = ctypes.c_uint(0)
    _check("moe_tail_take_device_error", lib().moe_tail_take_device_error(ctypes.byref(bits)))
    return int(bits.value)


def moe_tail_set_kernel_form(call: int, form: int) -> None:
    """Pin the kernel form of a call (FORM_EP, FORM_TP, FORM_LATENT; form 0 is
    the library's choice, see include/moe_tail.h).  Every form of a call gives
    the same bits; the setting is process-wide."""
    _check("moe_tail_set_kernel_form", lib().moe_tail_set_kernel_form(call, form))


def moe_tail_set_stage_wait_limit(limit_ns: int) -> None:
    """Failure-detection test hook: the operand-stage wait limit (ns) of the
    GEMM and staged finalize kernels for later calls; 0 restores the default.
    A limit shorter than a memory trip makes calls abort (device error bit 1)."""
    _check("moe_tail_set_stage_wait_limit", lib().moe_tail_set_stage_wait_limit(limit_ns))


class kernel_form:
    """Context manager: the call's kernel form pinned inside the block, the
    library's choice again after it."""

    def __init__(self, call: int, form: int):
        self.call, self.form = call, form

    def __enter__(self):
        moe_tail_set_kernel_form(self.call, self.form)
        return self

    def __exit__(self, *exc):
        moe_tail_set_kernel_form(self.call, 0)
        return False


def moe_tail_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the failure-detection self-test: a bounded wait that expires after
    limit_us and reports it through moe_tail_take_device_error()."""
    _check("moe_tail_selftest_wait_timeout", lib().moe_tail_selftest_wait_timeout(limit_us, _stream(stream)))
