"""Seeded synthetic inputs for the elementwise / row ops.

This package draws numbers and nothing else: it holds none of the ops'
arithmetic.  The oracle checks and the CUDA path both receive the arrays it
returns; that is the only thing they share.  The generator itself lives in
``synth.c`` (counter-based splitmix64, multi-threaded); this module loads it
and lays the draws out as the workloads in :mod:`synth.workloads` describe.

Arrays come back as numpy: ``float32`` for f32 tensors, ``uint16`` bit
patterns for bf16 tensors, ``int32`` for ids and positions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
LIB_PATH = os.path.join(_HERE, "libsynth.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so beside it (gcc, a second or so)."""
    stale = (not os.path.exists(LIB_PATH)) or os.path.getmtime(LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB_PATH)
            u64, i64, dbl, vp, i32 = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                      ctypes.c_void_p, ctypes.c_int)
            lib.syn_normal_f32.argtypes = [u64, u64, i64, i64, dbl, dbl, dbl, vp, i32]
            lib.syn_uniform_f32.argtypes = [u64, u64, i64, i64, dbl, dbl, vp, i32]
            lib.syn_randint_i32.argtypes = [u64, u64, i64, i64, i64, i64, vp, i32]
            lib.syn_unit_f64.argtypes = [u64, u64, i64, i64, vp, i32]
            lib.syn_raw_u64.argtypes = [u64, u64, i64, i64, vp]
            lib.syn_stream_key.argtypes = [u64, u64]
            lib.syn_stream_key.restype = u64
            lib.syn_f32_to_bf16.argtypes = [vp, vp, i64, i32]
            for f in (lib.syn_normal_f32, lib.syn_uniform_f32, lib.syn_randint_i32,
                      lib.syn_unit_f64, lib.syn_raw_u64, lib.syn_f32_to_bf16):
                f.restype = None
            _lib = lib
    return _lib


def threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def stream_id(name: str) -> int:
    """Stable 64-bit id of a named tensor stream (FNV-1a of the name)."""
    h = 0xCBF29CE484222325
    for ch in name.encode():
        h ^= ch
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _n(shape) -> int:
    return int(np.prod(shape, dtype=np.int64)) if len(shape) else 1


def normal(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0,
           clip: float = 0.0, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().syn_normal_f32(seed, stream_id(name), offset, out.size, mean, std, clip,
                           out.ctypes.data, threads())
    return out


def uniform(seed: int, name: str, shape, lo: float, hi: float, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().syn_uniform_f32(seed, stream_id(name), offset, out.size, lo, hi, out.ctypes.data,
                            threads())
    return out


def randint(seed: int, name: str, shape, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.int32)
    _load().syn_randint_i32(seed, stream_id(name), offset, out.size, lo, hi, out.ctypes.data,
                            threads())
    return out


def units(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().syn_unit_f64(seed, stream_id(name), offset, n, out.ctypes.data, threads())
    return out


def raw_u64(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().syn_raw_u64(seed, stream_id(name), offset, n, out.ctypes.data)
    return out


def stream_key(seed: int, name: str) -> int:
    return int(_load().syn_stream_key(seed, stream_id(name)))


def to_bf16(a: np.ndarray) -> np.ndarray:
    """Round generated f32 values to bf16 storage (nearest-even), as uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().syn_f32_to_bf16(a.ctypes.data, out.ctypes.data, a.size, threads())
    return out


def normal_bf16(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0,
                clip: float = 0.0, chunk: int = 1 << 26) -> np.ndarray:
    """normal() rounded to bf16, drawn in slices so no full-size f32 copy is held."""
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    lib = _load()
    tmp = np.empty(min(chunk, max(flat.size, 1)), dtype=np.float32)
    for s in range(0, flat.size, chunk):
        m = min(chunk, flat.size - s)
        lib.syn_normal_f32(seed, stream_id(name), s, m, mean, std, clip, tmp.ctypes.data,
                           threads())
        lib.syn_f32_to_bf16(tmp.ctypes.data, flat[s:s + m].ctypes.data, m, threads())
    return out


def uniform_bf16(seed: int, name: str, shape, lo: float, hi: float) -> np.ndarray:
    return to_bf16(uniform(seed, name, shape, lo, hi))
