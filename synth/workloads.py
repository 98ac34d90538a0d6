"""The synthetic workloads: shapes, dtypes, value distributions and planted
structure of every op case, drawn from :mod:`synth`.

Each workload is a name that says what it is, a seed, and op cases.  An op
case builder returns ``(arrays, params)``: ``arrays`` maps tensor names to
numpy arrays (f32 as ``float32``, bf16 as ``uint16`` bit patterns, ids and
positions as ``int32``), ``params`` holds the scalars (eps, r, mu, layout) and
the storage dtype.  ``rows=(r0, r1)`` draws only that slice of the leading
dimension, with the same values the full draw would hold there (the streams
are counter-based), so a bounded sample of a full-size workload costs only its
own size.

Inputs are built here and nowhere else; nothing in this module computes any
op's result.
"""
from __future__ import annotations

import numpy as np

from . import normal, normal_bf16, randint, to_bf16, uniform, units

TINY = "tiny-f32"
DECODE = "llama3-8b-decode-T64-bf16"
PREFILL = "llama3-8b-prefill-T8192-bf16"
ROPE_VARIANTS = "rope-variants-T4096-f32"
WIDE = "wide-argmax-rmsnorm-f32"

SEEDS = {TINY: 0, DECODE: 1, PREFILL: 2, ROPE_VARIANTS: 3, WIDE: 4}

NAN = np.float32(np.nan)


def _rows(shape, rows):
    """Leading-dim slice (r0, r1) of `shape` and the flat element offset of r0."""
    if rows is None:
        return tuple(shape), 0
    r0, r1 = rows
    inner = int(np.prod(shape[1:], dtype=np.int64))
    return (r1 - r0, *shape[1:]), r0 * inner


def _store(a32: np.ndarray, dtype: str) -> np.ndarray:
    return a32 if dtype == "f32" else to_bf16(a32)


def _normal(seed, name, shape, std, dtype, rows=None, mean=0.0, clip=0.0):
    shp, off = _rows(shape, rows)
    if dtype == "bf16" and off == 0 and clip == 0.0 and mean == 0.0:
        return normal_bf16(seed, name, shp, 0.0, std)
    return _store(normal(seed, name, shp, mean, std, clip, offset=off), dtype)


def inv_freq(base: float, r_formula: int, npairs: int, scale_from: int | None = None,
             scale: float = 1.0) -> np.ndarray:
    """omega_i = base^(-2i / r_formula) for i < npairs, in double, rounded to f32;
    entries i >= scale_from are multiplied by `scale` (the YaRN-style slow band)."""
    i = np.arange(npairs, dtype=np.float64)
    w = base ** (-2.0 * i / r_formula)
    if scale_from is not None:
        w = np.where(i >= scale_from, w * scale, w)
    return w.astype(np.float32)


# ---- per-op builders ---------------------------------------------------------

def _rmsnorm(seed, tag, rows_, d, dtype, rows=None, zero_rows=()):
    x = normal(seed, f"{tag}.x", _rows((rows_, d), rows)[0], 0.0, 1.0,
               offset=_rows((rows_, d), rows)[1])
    r0 = 0 if rows is None else rows[0]
    for z in zero_rows:
        if 0 <= z - r0 < x.shape[0]:
            x[z - r0] = 0.0
    w = uniform(seed, f"{tag}.w", (d,), 0.5, 1.5)
    return ({"x": _store(x, dtype), "w": _store(w, dtype)},
            {"dtype": dtype, "eps": 1e-5, "rows": x.shape[0], "d": d})


def _add_rmsnorm(seed, tag, rows_, d, dtype, rows=None):
    x = _normal(seed, f"{tag}.x", (rows_, d), 1.0, dtype, rows)
    res = _normal(seed, f"{tag}.residual", (rows_, d), 1.0, dtype, rows)
    w = _store(uniform(seed, f"{tag}.w", (d,), 0.5, 1.5), dtype)
    return ({"x": x, "residual": res, "w": w},
            {"dtype": dtype, "eps": 1e-5, "rows": x.shape[0], "d": d})


def _add(seed, tag, rows_, d, dtype, rows=None):
    a = _normal(seed, f"{tag}.a", (rows_, d), 1.0, dtype, rows)
    b = _normal(seed, f"{tag}.b", (rows_, d), 1.0, dtype, rows)
    return {"a": a, "b": b}, {"dtype": dtype, "n": a.size}


def _silu_mul(seed, tag, rows_, d, std, dtype, rows=None):
    g = _normal(seed, f"{tag}.gate", (rows_, d), std, dtype, rows)
    u = _normal(seed, f"{tag}.up", (rows_, d), std, dtype, rows)
    return {"gate": g, "up": u}, {"dtype": dtype, "n": g.size}


def _rope(seed, tag, T, H, D, r, pos, omega, mu, layout, dtype, rows=None, in_place=False):
    x = _normal(seed, f"{tag}.x", (T, H, D), 1.0, dtype, rows)
    p = pos if rows is None else pos[rows[0]:rows[1]]
    return ({"x": x, "pos": np.ascontiguousarray(p, dtype=np.int32),
             "inv_freq": np.ascontiguousarray(omega, dtype=np.float32)},
            {"dtype": dtype, "T": x.shape[0], "H": H, "D": D, "r": r, "mu": mu,
             "layout": layout, "in_place": in_place})


def _embedding(seed, tag, V, d, n, std, dtype, rows=None):
    table = _normal(seed, f"{tag}.table", (V, d), std, dtype)
    ids = randint(seed, f"{tag}.ids", _rows((n,), rows)[0], 0, V, offset=_rows((n,), rows)[1])
    return {"table": table, "ids": ids}, {"dtype": dtype, "n": ids.size, "d": d, "V": V}


def _argmax_plain(seed, tag, rows_, n, std, dtype, rows=None):
    x = _normal(seed, f"{tag}.x", (rows_, n), std, dtype, rows)
    return {"x": x}, {"dtype": dtype, "rows": x.shape[0], "n": n}


def _argmax_planted(seed, tag, rows_, n, std, nan_frac, tie_frac, rows=None, block=64):
    """N(0, std) clipped at 7 std; each entry NaN with probability nan_frac; in a
    tie_frac share of rows two distinct random entries set to 7.5 std, above
    every draw, so the row's maximum is an exact tie."""
    r0, r1 = (0, rows_) if rows is None else rows
    out = np.empty((r1 - r0, n), dtype=np.float32)
    tie_u = units(seed, f"{tag}.tie_rows", rows_)
    pick = units(seed, f"{tag}.tie_pos", 2 * rows_)
    top = np.float32(7.5 * std)
    for b0 in range(r0, r1, block):
        b1 = min(r1, b0 + block)
        blk = normal(seed, f"{tag}.x", (b1 - b0, n), 0.0, std, 7.0, offset=b0 * n)
        u = units(seed, f"{tag}.nan", (b1 - b0) * n, offset=b0 * n).reshape(b1 - b0, n)
        blk[u < nan_frac] = NAN
        for r in range(b0, b1):
            if tie_u[r] < tie_frac:
                i = int(pick[2 * r] * n)
                j = int(pick[2 * r + 1] * (n - 1))
                j = j + 1 if j >= i else j
                blk[r - b0, i] = top
                blk[r - b0, j] = top
        out[b0 - r0:b1 - r0] = blk
    return {"x": out}, {"dtype": "f32", "rows": out.shape[0], "n": n}


def _tiny_silu(seed):
    g = normal(seed, "silu.gate", (4, 128), 0.0, 3.0)
    u = normal(seed, "silu.up", (4, 128), 0.0, 3.0)
    g[0, 0], g[0, 1] = -1e4, 1e4
    g[1, 0] = -1e4
    u[1, 0] = -abs(u[1, 0]) - 0.5
    g[1, 1], g[1, 2] = 100.0, -100.0
    return {"gate": g, "up": u}, {"dtype": "f32", "n": g.size}


def _tiny_argmax(seed):
    n = 1000
    x = normal(seed, "argmax.x", (4, n), 0.0, 1.0, 7.0)
    pick = units(seed, "argmax.pick", 16)
    # row 0: the maximum appears twice (7.5 lies above every clipped draw)
    i = int(pick[0] * n)
    j = int(pick[1] * (n - 1))
    j = j + 1 if j >= i else j
    x[0, i] = x[0, j] = 7.5
    # row 1: NaN first, five more NaN at random places, and a tie at the top
    x[1, 0] = NAN
    for k in range(5):
        x[1, 1 + int(pick[2 + k] * (n - 1))] = NAN
    x[1, 500] = x[1, 900] = 7.5
    # row 2: no number at all
    x[2, :] = NAN
    # row 3: every entry -inf (a number; the first one wins)
    x[3, :] = -np.inf
    return {"x": x}, {"dtype": "f32", "rows": 4, "n": n}


# ---- the workloads -------------------------------------------------------------

def cases(workload: str) -> dict:
    """Op-case builders of a workload: name -> callable(rows=None) -> (arrays, params)."""
    s = SEEDS[workload]
    if workload == TINY:
        return {
            "rmsnorm": lambda rows=None: _rmsnorm(s, "rmsnorm", 4, 64, "f32", rows, zero_rows=(3,)),
            "rope_q": lambda rows=None: _rope(
                s, "rope.q", 4, 4, 16, 16, np.array([0, 1, 7, 100], np.int32),
                inv_freq(10000.0, 16, 8), 1.0, 0, "f32", rows),
            "silu_mul": lambda rows=None: _tiny_silu(s),
            "embedding": lambda rows=None: _embedding(s, "embedding", 1000, 64, 4, 1.0, "f32", rows),
            "argmax": lambda rows=None: _tiny_argmax(s),
        }
    if workload == DECODE:
        T = 64
        pos = randint(s, "rope.pos", (T,), 0, 8192)
        om = inv_freq(500000.0, 128, 64)
        return {
            "add_rmsnorm": lambda rows=None: _add_rmsnorm(s, "add_rmsnorm", T, 4096, "bf16", rows),
            "rope_q": lambda rows=None: _rope(s, "rope.q", T, 32, 128, 128, pos, om, 1.0, 0, "bf16", rows),
            "rope_k": lambda rows=None: _rope(s, "rope.k", T, 8, 128, 128, pos, om, 1.0, 0, "bf16", rows),
            "silu_mul": lambda rows=None: _silu_mul(s, "silu", T, 14336, 2.0, "bf16", rows),
            "argmax": lambda rows=None: _argmax_plain(s, "argmax", T, 128256, 4.0, "bf16", rows),
        }
    if workload == PREFILL:
        T = 8192
        pos = np.arange(T, dtype=np.int32)
        om = inv_freq(500000.0, 128, 64)
        return {
            "embedding": lambda rows=None: _embedding(s, "embedding", 128256, 4096, T, 0.02, "bf16", rows),
            "add_rmsnorm": lambda rows=None: _add_rmsnorm(s, "add_rmsnorm", T, 4096, "bf16", rows),
            "rope_q": lambda rows=None: _rope(s, "rope.q", T, 32, 128, 128, pos, om, 1.0, 0, "bf16", rows),
            "rope_k": lambda rows=None: _rope(s, "rope.k", T, 8, 128, 128, pos, om, 1.0, 0, "bf16", rows),
            "rope_q_interleaved": lambda rows=None: _rope(
                s, "rope.q", T, 32, 128, 128, pos, om, 1.0, 1, "bf16", rows),
            "rope_k_interleaved": lambda rows=None: _rope(
                s, "rope.k", T, 8, 128, 128, pos, om, 1.0, 1, "bf16", rows),
            "silu_mul": lambda rows=None: _silu_mul(s, "silu", T, 14336, 2.0, "bf16", rows),
            "add": lambda rows=None: _add(s, "add", T, 4096, "bf16", rows),
            "rmsnorm": lambda rows=None: _rmsnorm(s, "rmsnorm", T, 4096, "bf16", rows),
            "argmax": lambda rows=None: _argmax_plain(s, "argmax", T, 128256, 4.0, "bf16", rows),
        }
    if workload == ROPE_VARIANTS:
        T = 4096
        pos = randint(s, "rope.pos", (T,), 0, 1 << 20)
        return {
            "rope_q": lambda rows=None: _rope(
                s, "rope.q", T, 32, 128, 64, pos, inv_freq(10000.0, 64, 32), 1.0, 1, "f32", rows,
                in_place=True),
            "rope_k": lambda rows=None: _rope(
                s, "rope.k", T, 8, 128, 128, pos,
                inv_freq(10000.0, 64, 64, scale_from=16, scale=0.125), 1.2, 0, "f32", rows,
                in_place=True),
        }
    if workload == WIDE:
        return {
            "argmax": lambda rows=None: _argmax_planted(s, "argmax", 1024, 152064, 4.0, 0.01, 0.05, rows),
            "rmsnorm": lambda rows=None: _rmsnorm(s, "rmsnorm", 1024, 16384, "f32", rows),
        }
    raise KeyError(workload)


ALL = (TINY, DECODE, PREFILL, ROPE_VARIANTS, WIDE)
