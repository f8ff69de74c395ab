"""CPU oracle of the MoE decode tail -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  It wraps ``moe_tail_oracle.c`` (plain
C, FP32 with one rounding per operation for the finalize steps, double for the
GEMMs) with ctypes and shares no code with the CUDA path.  Tensors in and out
are CPU torch tensors (BF16 as torch.bfloat16); see the C file for the formula
each function follows and the page section it comes from.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_tail_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libmoetail_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing"]

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (contraction off: no fused multiply-add).
    MOE_TAIL_ORACLE_LIBRARY names another build of it to use instead (the
    tests that plant mistakes in a copy of the source use this)."""
    other = os.environ.get("MOE_TAIL_ORACLE_LIBRARY")
    if other:
        return other
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, i32, i64, f32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        L.oracle_ep_finalize.argtypes = [P, i64, P, P, i32, P, f32, f32, i32, i32, i32, i32, i32, P]
        L.oracle_tp_finalize.argtypes = [P, i64, P, P, i32, P, f32, f32, i32, i32, i32, i32, i32, P]
        L.oracle_latent_norm.argtypes = [P, P, f32, i32, i32, i32, P]
        L.oracle_latent_up.argtypes = [P, P, P, i32, i32, i32, i32, P]
        L.oracle_shared_expert.argtypes = [P, P, P, P, i32, i32, i32, P, P, i32]
        L.oracle_shared_down.argtypes = [P, P, i32, i32, i32, P, i32]
        L.oracle_sum_of_squares.argtypes = [P, i32]
        L.oracle_sum_of_squares.restype = f32
        L.oracle_inverse_rms.argtypes = [f32, i32, f32]
        L.oracle_inverse_rms.restype = f32
        L.oracle_bf16_from_f32.argtypes = [f32]
        L.oracle_bf16_from_f32.restype = ctypes.c_uint16
        L.oracle_bf16_from_f64.argtypes = [f64]
        L.oracle_bf16_from_f64.restype = ctypes.c_uint16
        L.oracle_f32_from_bf16.argtypes = [ctypes.c_uint16]
        L.oracle_f32_from_bf16.restype = f32
        for name in ("oracle_ep_finalize", "oracle_tp_finalize", "oracle_latent_norm",
                     "oracle_latent_up", "oracle_shared_expert", "oracle_shared_down"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _c(t: torch.Tensor) -> torch.Tensor:
    assert t.device.type == "cpu"
    return t.contiguous()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _weights(w: torch.Tensor):
    w = _c(w)
    if w.dtype == torch.bfloat16:
        return w, 1
    assert w.dtype == torch.float32
    return w, 0


def _check(rc: int, name: str) -> None:
    if rc == -2:
        raise MemoryError(f"{name}: host allocation failed")
    if rc != 0:
        raise ValueError(f"{name}: arguments refused ({rc})")


def ep_finalize(rows, rows_per_slot, idx, w, gamma, gain_center, eps, weight_before_norm,
                b, tp, K, P) -> torch.Tensor:
    """BF16 [b, P]: the EP finalize of rows [tp, rows_per_slot, P] (see C file)."""
    rows, idx, gamma = _c(rows), _c(idx), _c(gamma)
    w, wb = _weights(w)
    out = torch.empty((b, P), dtype=torch.bfloat16)
    _check(lib().oracle_ep_finalize(_ptr(rows), rows_per_slot, _ptr(idx), _ptr(w), wb, _ptr(gamma),
                                    gain_center, eps, int(weight_before_norm), b, tp, K, P, _ptr(out)),
           "ep_finalize")
    return out


def tp_finalize(partials, num_rows, idx, w, gamma, gain_center, eps, weight_before_norm,
                b, tp, K, P) -> torch.Tensor:
    """BF16 [b, P]: the expert-TP finalize of partials [tp, num_rows, P]."""
    partials, idx, gamma = _c(partials), _c(idx), _c(gamma)
    w, wb = _weights(w)
    out = torch.empty((b, P), dtype=torch.bfloat16)
    _check(lib().oracle_tp_finalize(_ptr(partials), num_rows, _ptr(idx), _ptr(w), wb, _ptr(gamma),
                                    gain_center, eps, int(weight_before_norm), b, tp, K, P, _ptr(out)),
           "tp_finalize")
    return out


def latent_norm(latent, gamma, eps, b, tp, L) -> torch.Tensor:
    """BF16 [b, L]: y = RMS norm of the slot-summed latent partials."""
    latent, gamma = _c(latent), _c(gamma)
    y = torch.empty((b, L), dtype=torch.bfloat16)
    _check(lib().oracle_latent_norm(_ptr(latent), _ptr(gamma), eps, b, tp, L, _ptr(y)), "latent_norm")
    return y


def latent_up(y, w_up, shared, tp_s, b, L, H) -> torch.Tensor:
    """BF16 [b, H]: y . w_up^T plus the slot-summed shared partials (double)."""
    y, w_up = _c(y), _c(w_up)
    shared = None if shared is None else _c(shared)
    out = torch.empty((b, H), dtype=torch.bfloat16)
    _check(lib().oracle_latent_up(_ptr(y), _ptr(w_up), _ptr(shared), tp_s if shared is not None else 0,
                                  b, L, H, _ptr(out)), "latent_up")
    return out


def latent_tail(latent, gamma, eps, w_up, shared, tp_s, b, tp, L, H):
    """(y, out): the latent tail's norm then its up-projection."""
    y = latent_norm(latent, gamma, eps, b, tp, L)
    return y, latent_up(y, w_up, shared, tp_s, b, L, H)


def shared_expert(x, w_gate, w_up, w_down, b, H, I, out_in=None, accumulate=True):
    """(h, out): the fused shared expert; out = out_in + down(h) (accumulate)."""
    x, w_gate, w_up, w_down = _c(x), _c(w_gate), _c(w_up), _c(w_down)
    h = torch.empty((b, I), dtype=torch.bfloat16)
    if accumulate:
        out = _c(out_in).clone()
    else:
        out = torch.empty((b, H), dtype=torch.bfloat16)
    _check(lib().oracle_shared_expert(_ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(w_down), b, H, I,
                                      _ptr(h), _ptr(out), int(accumulate)), "shared_expert")
    return h, out


def shared_down(h, w_down, b, H, I, out_in=None, accumulate=True):
    """BF16 [b, H]: the shared expert's down projection of h [b, I] (double),
    added into out_in (accumulate) or alone."""
    h, w_down = _c(h), _c(w_down)
    out = _c(out_in).clone() if accumulate else torch.empty((b, H), dtype=torch.bfloat16)
    _check(lib().oracle_shared_down(_ptr(h), _ptr(w_down), b, H, I, _ptr(out), int(accumulate)), "shared_down")
    return out


def sum_of_squares(v: np.ndarray) -> float:
    v = np.ascontiguousarray(v, dtype=np.float32)
    return float(lib().oracle_sum_of_squares(v.ctypes.data_as(ctypes.c_void_p), v.size))


def inverse_rms(ss: float, P: int, eps: float) -> float:
    """1 / sqrt(ss * (float)(1/P) + eps), each step one FP32 operation."""
    return float(lib().oracle_inverse_rms(ss, P, eps))


def bf16_from_f32(x: float) -> int:
    return int(lib().oracle_bf16_from_f32(x))


def bf16_from_f64(x: float) -> int:
    return int(lib().oracle_bf16_from_f64(x))


def f32_from_bf16(h: int) -> float:
    return float(lib().oracle_f32_from_bf16(h))
