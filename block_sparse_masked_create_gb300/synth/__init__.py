"""Seeded synthetic inputs (splitmix64 -> Box-Muller -> bf16), shared by the oracle tests and the CUDA path.

Holds none of the attention method: only counter-based random numbers, so that both sides read identical
inputs. The C source next to this file is compiled on first use (gcc, no architecture flags).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libfasynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into libfasynth.so next to it (if missing or stale)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-D_GNU_SOURCE", _SRC,
                               "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            lib.synth_stream_state.restype = u64
            lib.synth_stream_state.argtypes = [u64, u64]
            lib.synth_draw_u64.restype = u64
            lib.synth_draw_u64.argtypes = [u64, u64, u64]
            lib.synth_bf16_from_double.restype = ctypes.c_uint16
            lib.synth_bf16_from_double.argtypes = [dbl]
            lib.synth_normal_bf16.restype = None
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, dbl, ctypes.c_void_p]
            lib.synth_normal_f64.restype = None
            lib.synth_normal_f64.argtypes = [u64, u64, u64, u64, dbl, dbl, ctypes.c_void_p]
            lib.synth_uniform_int.restype = None
            lib.synth_uniform_int.argtypes = [u64, u64, ctypes.POINTER(u64), i64, i64, i64, ctypes.c_void_p]
            lib.synth_permutation.restype = None
            lib.synth_permutation.argtypes = [u64, u64, i64, ctypes.c_void_p]
            _lib = lib
    return _lib


def draw_u64(seed: int, tid: int, k: int) -> int:
    return int(_load().synth_draw_u64(seed, tid, k))


def stream_state(seed: int, tid: int) -> int:
    return int(_load().synth_stream_state(seed, tid))


def bf16_bits_from_double(x: float) -> int:
    return int(_load().synth_bf16_from_double(float(x)))


def normal_bf16_bits(seed: int, tid: int, shape, first: int = 0, mean: float = 0.0,
                     std: float = 1.0) -> np.ndarray:
    """uint16 bf16 bit patterns, elements [first, first+prod(shape)) of stream (seed, tid)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().synth_normal_bf16(seed, tid, first, n, mean, std, out.ctypes.data)
    return out.reshape(shape)


def normal_f64(seed: int, tid: int, shape, first: int = 0, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    if n:
        _load().synth_normal_f64(seed, tid, first, n, mean, std, out.ctypes.data)
    return out.reshape(shape)


def uniform_ints(seed: int, tid: int, lo: int, hi: int, count: int, cursor: int = 0):
    """`count` sequential draws uniform on [lo, hi]; returns (values int64, new cursor)."""
    out = np.empty(count, dtype=np.int64)
    cur = ctypes.c_uint64(cursor)
    if count:
        _load().synth_uniform_int(seed, tid, ctypes.byref(cur), lo, hi, count, out.ctypes.data)
    return out, int(cur.value)


def permutation(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().synth_permutation(seed, tid, n, out.ctypes.data)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)
