"""The oracle: a plain, slow, single-threaded CPU reference of the ops, in C
(``oracle.c``), loaded through ctypes.

TEST INFRASTRUCTURE.  Only ``tests/``, the ``smoke()`` check in
``__graft_entry__.py`` and the ``cpu_baseline`` leg (and ``--impl reference``
arm) of ``bench.py`` may import this package.  The product path never does,
and it shares no code with the CUDA sources.

Every function takes and returns numpy arrays: f32 inputs as ``float32``;
bf16 data is widened with :func:`bf16_widen` first and the f32 results are
rounded with :func:`bf16_round` where a test needs storage bits.  Each op is
the definition the pages give, written out step by step in f32; the
citations sit beside each function in ``oracle.c``.

``Oracle(mutant=k)`` loads a build with the k-th planted mistake of the
pages' pitfalls table and the further planted mistakes (s01..s24), so tests can
show that the pins reject each one.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
_lock = threading.Lock()
_cache: dict[int, "Oracle"] = {}


class OracleError(ValueError):
    pass


def lib_path(mutant: int = 0) -> str:
    return os.path.join(_HERE, "liboracle.so" if mutant == 0 else f"liboracle_m{mutant:02d}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    path = lib_path(mutant)
    stale = (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC)
    if force or stale:
        flags = list(CFLAGS) + ([f"-DORACLE_MUTANT={mutant}"] if mutant else [])
        tmp = path + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *flags, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, path)
    return path


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray):
    return a.ctypes.data


class Oracle:
    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        lib = ctypes.CDLL(build(mutant))
        i64, f32, vp, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
        u64 = ctypes.c_uint64
        sig = {
            "orc_rmsnorm": [vp, vp, vp, i64, i64, f32],
            "orc_add": [vp, vp, vp, i64],
            "orc_layernorm": [vp, vp, vp, vp, i64, i64, f32],
            "orc_add_rmsnorm": [vp, vp, vp, vp, vp, i64, i64, f32, i32],
            "orc_rope": [vp, vp, vp, i64, i64, i64, i64, vp, f32, i32],
            "orc_rope_cos_sin": [vp, i64, i64, vp],
            "orc_rope_multi": [vp, vp, vp, i64, i64, i64, i64, vp, vp, f32, i32],
            "orc_qk_norm_rope": [vp, vp, vp, vp, i64, i64, i64, f32, i64, vp, f32, i32, i32],
            "orc_silu_mul": [vp, vp, vp, i64],
            "orc_embedding": [vp, vp, vp, i64, i64, i64],
            "orc_argmax": [vp, i64],
            "orc_argmax_rows": [vp, vp, i64, i64],
            "orc_sample_rows": [vp, vp, i64, i64, i32, f32, i64, f32, vp, vp, vp],
            "orc_sample_rows_seeded": [vp, vp, i64, i64, i32, f32, i64, f32, u64, u64, vp, vp, vp],
            "orc_pcg64_seeded_state": [u64, vp],
            "orc_pcg64_raw": [u64, u64, u64, u64, i64, vp, vp],
            "orc_pcg64_advance": [u64, u64, u64, u64, u64, u64, vp],
            "orc_pcg64_uniforms": [u64, u64, i64, vp],
            "orc_bf16_widen": [vp, vp, i64],
            "orc_bf16_round": [vp, vp, i64],
            "orc_mutant": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int32 if name == "orc_argmax" else (
                None if name.startswith(("orc_bf16", "orc_pcg64")) else ctypes.c_int)
        assert lib.orc_mutant() == mutant
        self.lib = lib

    @staticmethod
    def _check(st: int, what: str):
        if st != 0:
            raise OracleError(f"{what}: oracle status {st}")

    # -- storage -------------------------------------------------------------
    def bf16_widen(self, bits: np.ndarray) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float32)
        self.lib.orc_bf16_widen(_ptr(bits), _ptr(out), bits.size)
        return out

    def bf16_round(self, x: np.ndarray) -> np.ndarray:
        x = _f32(x)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.orc_bf16_round(_ptr(x), _ptr(out), x.size)
        return out

    # -- ops -------------------------------------------------------------------
    def rmsnorm(self, x, w, eps: float, out: np.ndarray | None = None) -> np.ndarray:
        x, w = _f32(x), _f32(w)
        d = x.shape[-1]
        rows = x.size // d if d else 0
        if w.size != d:
            raise OracleError("rmsnorm: w must have d entries")
        y = np.empty_like(x) if out is None else out
        self._check(self.lib.orc_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, d, eps), "rmsnorm")
        return y

    def layernorm(self, x, g, b, eps: float) -> np.ndarray:
        """LayerNorm of every row of x with gain g and bias b (None: no bias)."""
        x, g = _f32(x), _f32(g)
        d = x.shape[-1]
        bb = None if b is None else _f32(b)
        if g.size != d or (bb is not None and bb.size != d):
            raise OracleError("layernorm: g and b have d entries")
        y = np.empty_like(x)
        self._check(self.lib.orc_layernorm(_ptr(x), _ptr(g), None if bb is None else _ptr(bb), _ptr(y),
                                           x.size // d, d, eps), "layernorm")
        return y

    def add(self, a, b) -> np.ndarray:
        a, b = _f32(a), _f32(b)
        if a.shape != b.shape:
            raise OracleError("add: shapes differ")
        y = np.empty_like(a)
        self._check(self.lib.orc_add(_ptr(a), _ptr(b), _ptr(y), a.size), "add")
        return y

    def add_rmsnorm(self, x, residual, w, eps: float, h_bf16: bool = False):
        x, r, w = _f32(x), _f32(residual), _f32(w)
        d = x.shape[-1]
        y = np.empty_like(x)
        h = np.empty_like(x)
        self._check(self.lib.orc_add_rmsnorm(_ptr(x), _ptr(r), _ptr(w), _ptr(y), _ptr(h),
                                             x.size // d, d, eps, int(h_bf16)), "add_rmsnorm")
        return y, h

    def rope(self, x, pos, inv_freq, r: int, mu: float, layout: int,
             in_place: bool = False) -> np.ndarray:
        x = _f32(x) if not in_place else x
        if in_place and (x.dtype != np.float32 or not x.flags.c_contiguous):
            raise OracleError("rope in place needs a contiguous float32 array")
        T, H, D = x.shape
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        om = _f32(inv_freq)
        if pos.size != T or om.size < r // 2:
            raise OracleError("rope: pos needs T entries and inv_freq r/2")
        y = x if in_place else np.empty_like(x)
        self._check(self.lib.orc_rope(_ptr(x), _ptr(y), _ptr(pos), T, H, D, r, _ptr(om), mu,
                                      layout), "rope")
        return y

    def rope_multi(self, x, pos, dims, inv_freq, mu: float, layout: int) -> np.ndarray:
        """Multi-axis RoPE: x [T, H, D], pos [T, A], dims [A] (even, summing to at
        most D), inv_freq the concatenated per-axis frequencies."""
        x = _f32(x)
        T, H, D = x.shape
        dims_a = np.ascontiguousarray(dims, dtype=np.int64)
        A = dims_a.size
        pos = np.ascontiguousarray(pos, dtype=np.int32).reshape(T, A)
        om = _f32(inv_freq)
        if om.size < int(dims_a.sum()) // 2:
            raise OracleError("rope_multi: inv_freq needs sum(dims)/2 entries")
        y = np.empty_like(x)
        self._check(self.lib.orc_rope_multi(_ptr(x), _ptr(y), _ptr(pos), T, H, D, A, _ptr(dims_a), _ptr(om), mu,
                                            layout), "rope_multi")
        return y

    def rope_cos_sin(self, inv_freq, r: int, length: int) -> np.ndarray:
        """The [length, r/2, 2] table of (cos, sin) per position and pair."""
        om = _f32(inv_freq)
        if om.size < r // 2:
            raise OracleError("rope_cos_sin: inv_freq needs r/2 entries")
        out = np.empty((length, r // 2, 2), dtype=np.float32)
        self._check(self.lib.orc_rope_cos_sin(_ptr(out), length, r, _ptr(om)), "rope_cos_sin")
        return out

    def qk_norm_rope(self, x, g, eps: float, pos, inv_freq, r: int, mu: float, layout: int,
                     n_bf16: bool = False) -> np.ndarray:
        """RMSNorm of every head row of x [T, H, D] with gain g [D], the result
        stored (rounded to bf16 when n_bf16), then RoPE."""
        x, g = _f32(x), _f32(g)
        T, H, D = x.shape
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        om = _f32(inv_freq)
        if g.size != D or pos.size != T or om.size < r // 2:
            raise OracleError("qk_norm_rope: g has D entries, pos T, inv_freq r/2")
        y = np.empty_like(x)
        self._check(self.lib.orc_qk_norm_rope(_ptr(x), _ptr(g), _ptr(y), _ptr(pos), T, H, D, eps, r,
                                              _ptr(om), mu, layout, int(n_bf16)), "qk_norm_rope")
        return y

    def silu_mul(self, gate, up) -> np.ndarray:
        g, u = _f32(gate), _f32(up)
        y = np.empty_like(g)
        self._check(self.lib.orc_silu_mul(_ptr(g), _ptr(u), _ptr(y), g.size), "silu_mul")
        return y

    def embedding(self, table, ids) -> np.ndarray:
        table = _f32(table)
        V, d = table.shape
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        out = np.empty((ids.size, d), dtype=np.float32)
        self._check(self.lib.orc_embedding(_ptr(table), _ptr(ids), _ptr(out), ids.size, d, V),
                    "embedding")
        return out

    def argmax(self, x) -> np.ndarray:
        x = _f32(x)
        if x.ndim == 1:
            x = x.reshape(1, -1)
        rows, n = x.shape
        out = np.empty(rows, dtype=np.int32)
        st = self.lib.orc_argmax_rows(_ptr(x), _ptr(out), rows, n)
        if st == -3:
            raise OracleError("argmax: empty row")
        self._check(st, "argmax")
        return out

    METHODS = {"greedy": 0, "temperature": 1, "top_k": 2, "top_p": 3, "min_p": 4}

    def sample(self, x, method: str, u, temperature: float = 1.0, top_k: int = 1, top_p: float = 1.0,
               min_p: float = 0.0) -> np.ndarray:
        """One draw per row of x [rows, n] by the inverse CDF at u[row]."""
        x = _f32(x)
        if x.ndim == 1:
            x = x.reshape(1, -1)
        rows, n = x.shape
        u = np.ascontiguousarray(np.broadcast_to(np.asarray(u, np.float32), (rows,)), dtype=np.float32)
        out = np.empty(rows, dtype=np.int32)
        idx = np.empty(n, dtype=np.int64)
        buf = np.empty(n, dtype=np.float32)
        m = self.METHODS[method]
        pp = top_p if method == "top_p" else min_p
        self._check(self.lib.orc_sample_rows(_ptr(x), _ptr(out), rows, n, m, temperature, top_k, pp, _ptr(u),
                                             _ptr(idx), _ptr(buf)), "sample")
        return out

    def sample_seeded(self, x, method: str, seed: int, offset: int, temperature: float = 1.0, top_k: int = 1,
                      top_p: float = 1.0, min_p: float = 0.0) -> np.ndarray:
        """One draw per row of x [rows, n]; row r draws with the uniform of
        draw offset + r of the PCG64 stream seeded with `seed`."""
        x = _f32(x)
        if x.ndim == 1:
            x = x.reshape(1, -1)
        rows, n = x.shape
        out = np.empty(rows, dtype=np.int32)
        u = np.empty(rows, dtype=np.float32)
        idx = np.empty(n, dtype=np.int64)
        buf = np.empty(n, dtype=np.float32)
        pp = top_p if method == "top_p" else min_p
        self._check(self.lib.orc_sample_rows_seeded(_ptr(x), _ptr(out), rows, n, self.METHODS[method], temperature,
                                                    top_k, pp, seed, offset, _ptr(u), _ptr(idx), _ptr(buf)),
                    "sample_seeded")
        return out

    # -- the seeded generator (PCG64) ----------------------------------------------
    @staticmethod
    def _split(v: int) -> tuple[int, int]:
        v &= (1 << 128) - 1
        return v >> 64, v & ((1 << 64) - 1)

    def pcg64_seeded_state(self, seed: int) -> int:
        """The 128-bit state the seed plants."""
        st = np.empty(2, dtype=np.uint64)
        self.lib.orc_pcg64_seeded_state(seed, _ptr(st))
        return (int(st[0]) << 64) | int(st[1])

    def pcg64_raw(self, state: int, inc: int, count: int) -> tuple[np.ndarray, int]:
        """`count` 64-bit outputs from (state, inc), each after its step, and
        the final state."""
        out = np.empty(count, dtype=np.uint64)
        st = np.empty(2, dtype=np.uint64)
        self.lib.orc_pcg64_raw(*self._split(state), *self._split(inc), count, _ptr(out), _ptr(st))
        return out, (int(st[0]) << 64) | int(st[1])

    def pcg64_advance(self, state: int, inc: int, delta: int) -> int:
        """The state `delta` steps after `state` (0 <= delta < 2^128)."""
        st = np.empty(2, dtype=np.uint64)
        self.lib.orc_pcg64_advance(*self._split(state), *self._split(inc), *self._split(delta), _ptr(st))
        return (int(st[0]) << 64) | int(st[1])

    def pcg64_uniforms(self, seed: int, offset: int, n: int) -> np.ndarray:
        """The uniforms of draws offset .. offset + n - 1 of the seeded stream."""
        u = np.empty(n, dtype=np.float32)
        self.lib.orc_pcg64_uniforms(seed, offset, n, _ptr(u))
        return u

    def argmax_one(self, x) -> int:
        """The pages' single-row routine as written, -1 for an empty row too."""
        x = _f32(x).reshape(-1)
        return int(self.lib.orc_argmax(_ptr(x), x.size))


def get(mutant: int = 0) -> Oracle:
    with _lock:
        if mutant not in _cache:
            _cache[mutant] = Oracle(mutant)
        return _cache[mutant]
