"""Pins of the oracle: checks that tie it to something other than itself.

Each ``pin_*`` takes an oracle handle and raises AssertionError when the oracle
breaks the fact it checks.  The facts come from the pages (worked examples and
the test catalog of "Elementwise kernels in C", section 3 and 4), from the
mathematics (closed forms, invariants, brute force in float64), and from
library routines that reduce to the same definition (torch float64
``rms_norm`` / ``silu``, ``numpy.nanargmax``, numpy fancy indexing, torch's
bf16 rounding).  ``KILLS`` names, for each planted mistake s01..s15 of the
pages' pitfalls table (section 5), the pin that the table says must reject it.
"""
from __future__ import annotations

import numpy as np
import torch

from golden_io import load, printed_close

RNG = np.random.default_rng(1234)  # pins draw their own small cases


def _rand(*shape, scale=1.0):
    return (RNG.standard_normal(shape) * scale).astype(np.float32)


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def _same_bits(a, b) -> bool:
    return np.array_equal(_bits(a), _bits(b))


# ---- RMSNorm -------------------------------------------------------------------

def pin_hand_example(o):
    g = load("rmsnorm_worked_example.txt")
    y = o.rmsnorm(g["x"].reshape(1, -1), g["w"], g["eps"])
    assert printed_close(y.ravel(), g["y"], 7), ("rmsnorm worked example", y)
    for name in ("rope_half_worked_example.txt", "rope_interleaved_worked_example.txt"):
        g = load(name)
        x = g["x"].astype(np.float32).reshape(1, 1, -1)
        y = o.rope(x, [g["pos"]], g["inv_freq"], g["r"], g["mu"], g["layout"])
        assert printed_close(y.ravel(), g["y"], 7), (name, y)
    g = load("silu_mul_worked_example.txt")
    y = o.silu_mul(g["gate"], g["up"])
    assert printed_close(y, g["y"], 7), ("silu_mul worked example", y)
    g = load("argmax_worked_example.txt")
    assert int(o.argmax(g["x"])[0]) == g["index"]


def pin_rmsnorm_eps_is_inside_the_root(o):
    g = load("rmsnorm_eps_inside_root.txt")
    y = o.rmsnorm(g["x"].reshape(1, -1), g["w"], g["eps"])
    assert printed_close(y.ravel(), g["y"], 4), y
    z = o.rmsnorm(np.zeros((2, 33), np.float32), np.full(33, 1.25, np.float32), 1e-5)
    assert not np.isnan(z).any() and np.all(z == 0.0)


def pin_rmsnorm_rows_are_independent_and_in_place(o):
    d = 37
    w = RNG.uniform(0.5, 1.5, d).astype(np.float32)
    batch = _rand(12, d)
    batch[5] *= 1e-3
    batch[7] *= 1e3
    full = o.rmsnorm(batch, w, 1e-5)
    for b in range(1, 13):
        part = o.rmsnorm(batch[:b], w, 1e-5)
        assert _same_bits(part, full[:b]), f"batch of {b}"
    for r in range(12):
        alone = o.rmsnorm(batch[r:r + 1], w, 1e-5)
        assert _same_bits(alone, full[r:r + 1]), f"row {r} alone"
    x = batch.copy()
    o.rmsnorm(x, w, 1e-5, out=x)
    assert _same_bits(x, full)


def pin_rmsnorm_library(o):
    for d in (1, 7, 64, 1000, 4096):
        x = _rand(5, d, scale=3.0)
        w = RNG.uniform(0.5, 1.5, d).astype(np.float32)
        y = o.rmsnorm(x, w, 1e-5).astype(np.float64)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x).double(), (d,),
                                           torch.from_numpy(w).double(), 1e-5).numpy()
        err = np.abs(y - ref) / np.maximum(np.abs(ref), 1e-30)
        assert err.max() <= 2e-6, (d, err.max())


def pin_rmsnorm_closed_forms(o):
    x = _rand(6, 257)
    w = RNG.uniform(0.5, 1.5, 257).astype(np.float32)
    base = o.rmsnorm(x, w, 0.0)
    for k in (-20, -3, 1, 9, 30):  # power-of-two scale: exact at eps = 0
        assert _same_bits(o.rmsnorm(x * np.float32(2.0 ** k), w, 0.0), base), k
    for c in (0.37, 11.0):
        y = o.rmsnorm(x * np.float32(c), w, 0.0)
        assert np.allclose(y, base, rtol=2e-6, atol=0)
    rms = np.sqrt(np.mean((base.astype(np.float64) / w) ** 2, axis=1))
    assert np.allclose(rms, 1.0, atol=2e-6), rms


def pin_layernorm(o):
    """LayerNorm against float64 torch layer_norm, its closed forms (zero mean
    and unit variance of (y - b) / g at eps = 0, invariance to a constant
    shift by a power of two), and a constant row giving exactly b."""
    for d in (1, 7, 64, 1000, 4096):
        x = _rand(5, d, scale=3.0) + np.float32(0.75)
        g = RNG.uniform(0.5, 1.5, d).astype(np.float32)
        b = _rand(d, scale=0.2)
        y = o.layernorm(x, g, b, 1e-5).astype(np.float64)
        ref = torch.nn.functional.layer_norm(torch.from_numpy(x).double(), (d,), torch.from_numpy(g).double(),
                                             torch.from_numpy(b).double(), 1e-5).numpy()
        scale = np.abs(ref - b).max(axis=-1, keepdims=True) + np.abs(b).max() + 1e-30
        assert np.all(np.abs(y - ref) <= 4e-6 * scale), d
        y0 = o.layernorm(x, g, None, 1e-5).astype(np.float64)
        assert np.all(np.abs(y0 - (ref - b)) <= 4e-6 * scale), d
    x = _rand(6, 513)
    g = RNG.uniform(0.5, 1.5, 513).astype(np.float32)
    b = _rand(513, scale=0.3)
    z = (o.layernorm(x, g, b, 0.0).astype(np.float64) - b) / g
    assert np.allclose(z.mean(axis=1), 0.0, atol=1e-6) and np.allclose((z ** 2).mean(axis=1), 1.0, atol=4e-6)
    shifted = o.layernorm(x + np.float32(4.0), g, b, 0.0)
    assert np.allclose(shifted, o.layernorm(x, g, b, 0.0), rtol=0, atol=2e-5)
    const = np.full((2, 40), 3.25, np.float32)
    assert _same_bits(o.layernorm(const, g[:40], b[:40], 1e-5), np.broadcast_to(b[:40], (2, 40)))


def pin_add_rmsnorm_composition(o):
    d = 300
    x, r = _rand(4, d), _rand(4, d)
    w = RNG.uniform(0.5, 1.5, d).astype(np.float32)
    y, h = o.add_rmsnorm(x, r, w, 1e-5)
    assert _same_bits(h, x + r)  # numpy's f32 add is the IEEE sum
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x + r).double(), (d,),
                                       torch.from_numpy(w).double(), 1e-5).numpy()
    assert np.allclose(y, ref, rtol=2e-6, atol=0)
    yb, hb = o.add_rmsnorm(x, r, w, 1e-5, h_bf16=True)
    hb_ref = torch.from_numpy(x + r).bfloat16().float().numpy()
    assert _same_bits(hb, hb_ref)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(hb_ref).double(), (d,),
                                       torch.from_numpy(w).double(), 1e-5).numpy()
    assert np.allclose(yb, ref, rtol=2e-6, atol=0)


# ---- RoPE ----------------------------------------------------------------------

def _brute_rope(x, pos, om, r, mu, layout):
    """float64 2x2 rotation matrices on each pair, the angle taken as the f32
    product of the position and the frequency."""
    x = x.astype(np.float64)
    y = x.copy()
    T, H, D = x.shape
    for t in range(T):
        for i in range(r // 2):
            th = float(np.float32(np.float32(pos[t]) * np.float32(om[i])))
            R = mu * np.array([[np.cos(th), -np.sin(th)], [np.sin(th), np.cos(th)]])
            ia, ib = (i, i + r // 2) if layout == 0 else (2 * i, 2 * i + 1)
            for h in range(H):
                y[t, h, [ia, ib]] = R @ x[t, h, [ia, ib]]
    return y


def _pair_idx(r, layout):
    i = np.arange(r // 2)
    return (i, i + r // 2) if layout == 0 else (2 * i, 2 * i + 1)


def pin_rope_interleaved_layout_and_position_zero(o):
    g = load("rope_interleaved_worked_example.txt")
    y = o.rope(g["x"].astype(np.float32).reshape(1, 1, -1), [g["pos"]], g["inv_freq"], g["r"],
               g["mu"], g["layout"])
    assert printed_close(y.ravel(), g["y"], 7), y
    x = _rand(3, 2, 12)
    om = RNG.uniform(0.001, 2.0, 5).astype(np.float32)
    for layout in (0, 1):
        y = o.rope(x, [0, 0, 0], om, 10, 1.0, layout)
        assert _same_bits(y, x), layout


def pin_rope_partial_rotary_and_scaling(o):
    T, H, D, r = 5, 3, 24, 10
    x = _rand(T, H, D)
    pos = RNG.integers(0, 5000, T).astype(np.int32)
    om = RNG.uniform(0.001, 1.0, r // 2).astype(np.float32)
    for layout in (0, 1):
        y1 = o.rope(x, pos, om, r, 1.0, layout)
        assert _same_bits(y1[..., r:], x[..., r:]), "tail must pass through"
        y2 = o.rope(x, pos, om, r, 2.0, layout)
        assert _same_bits(y2[..., :r], (y1[..., :r] * np.float32(2.0))), "mu = 2 doubles"
        ref = _brute_rope(x, pos, om, r, 1.0, layout)  # [T, H, D] indexing, per token
        a, b = _pair_idx(r, layout)
        norm = np.sqrt(x[..., a].astype(np.float64) ** 2 + x[..., b].astype(np.float64) ** 2)
        for idx in (a, b):
            assert np.all(np.abs(y1[..., idx] - ref[..., idx]) <= 2e-6 * norm + 1e-30)
        xi = x.copy()
        o.rope(xi, pos, om, r, 1.0, layout, in_place=True)
        assert _same_bits(xi, y1), "in place equals out of place"


def pin_rope_is_a_rotation(o):
    for trial in range(8):
        T, H = int(RNG.integers(1, 6)), int(RNG.integers(1, 5))
        r = 2 * int(RNG.integers(1, 9))
        D = r + int(RNG.integers(0, 5))
        layout = trial % 2
        mu = float(RNG.choice([1.0, 1.2, 0.5]))
        x = _rand(T, H, D)
        pos = RNG.integers(0, 1 << 20, T).astype(np.int32)
        om = RNG.uniform(1e-4, 1.5, r // 2).astype(np.float32)
        y = o.rope(x, pos, om, r, mu, layout)
        a, b = _pair_idx(r, layout)
        n0 = np.hypot(x[..., a].astype(np.float64), x[..., b].astype(np.float64))
        n1 = np.hypot(y[..., a].astype(np.float64), y[..., b].astype(np.float64))
        assert np.all(np.abs(n1 - mu * n0) <= 1e-6 * mu * n0 + 1e-30), (trial, layout)


def pin_rope_brute_force(o):
    for layout in (0, 1):
        x = _rand(4, 3, 10)
        pos = np.array([0, 3, 77, 4095], np.int32)
        om = RNG.uniform(1e-3, 1.0, 4).astype(np.float32)
        y = o.rope(x, pos, om, 8, 1.2, layout)
        ref = _brute_rope(x, pos, om, 8, 1.2, layout)
        a, b = _pair_idx(8, layout)
        norm = np.hypot(x[..., a].astype(np.float64), x[..., b].astype(np.float64))
        for idx in (a, b):
            assert np.all(np.abs(y[..., idx] - ref[..., idx]) <= 2e-6 * 1.2 * norm + 1e-30)


def pin_rope_multi_axis(o):
    """Multi-axis RoPE ("Operations", section 3): one axis is plain RoPE; each
    slice equals RoPE of that slice alone at its axis's position (bit exact);
    an axis's position moves only its slice; float64 brute force."""
    T, H, D = 4, 3, 40
    dims = [12, 10, 10]  # 32 rotated entries, 8 pass through
    x = _rand(T, H, D)
    pos = RNG.integers(0, 3000, (T, 3)).astype(np.int32)
    om = RNG.uniform(1e-3, 1.0, 16).astype(np.float32)
    for layout in (0, 1):
        y = o.rope_multi(x, pos, dims, om, 1.1, layout)
        assert _same_bits(y[..., 32:], x[..., 32:]), "entries past the slices pass through"
        off = foff = 0
        for a, d in enumerate(dims):
            sl = np.ascontiguousarray(x[..., off:off + d])
            ref = o.rope(sl, pos[:, a], om[foff:foff + d // 2], d, 1.1, layout)
            assert _same_bits(y[..., off:off + d], ref), (layout, a)
            brute = _brute_rope(sl, pos[:, a], om[foff:foff + d // 2], d, 1.1, layout)
            assert np.all(np.abs(y[..., off:off + d] - brute) <= 2e-6 * 1.1 * np.abs(sl).max() * 2)
            off, foff = off + d, foff + d // 2
        moved = pos.copy()
        moved[:, 1] += 17
        y2 = o.rope_multi(x, moved, dims, om, 1.1, layout)
        assert _same_bits(y2[..., :12], y[..., :12]) and _same_bits(y2[..., 22:], y[..., 22:])
        assert not np.array_equal(y2[..., 12:22], y[..., 12:22])
    om1 = RNG.uniform(1e-3, 1.0, D // 2).astype(np.float32)
    assert _same_bits(o.rope_multi(x, pos[:, :1], [D], om1, 1.0, 0), o.rope(x, pos[:, 0], om1, D, 1.0, 0))


def pin_rope_relative_position(o):
    D, r = 16, 16
    om = (10000.0 ** (-2.0 * np.arange(8) / 16)).astype(np.float32)
    q, k = _rand(1, 1, D), _rand(1, 1, D)
    for layout in (0, 1):
        dots = []
        for shift in (0, 5, 20, 50):  # angles stay below 100 rad, where their f32 rounding is < 4e-6
            qr = o.rope(q, [37 + shift], om, r, 1.0, layout).astype(np.float64)
            kr = o.rope(k, [12 + shift], om, r, 1.0, layout).astype(np.float64)
            dots.append(float(np.sum(qr * kr)))
        scale = np.linalg.norm(q) * np.linalg.norm(k)
        assert max(dots) - min(dots) <= 2e-5 * scale, (layout, dots)
        # and the dot product does change with the offset itself
        qr = o.rope(q, [38], om, r, 1.0, layout).astype(np.float64)
        kr = o.rope(k, [12], om, r, 1.0, layout).astype(np.float64)
        assert abs(float(np.sum(qr * kr)) - dots[0]) > 1e-4 * scale


def pin_rope_layout_equivalence(o):
    T, H, D, r = 3, 2, 12, 8
    x = _rand(T, H, D)
    pos = np.array([1, 9, 300], np.int32)
    om = RNG.uniform(1e-3, 1.0, r // 2).astype(np.float32)
    perm = np.arange(D)  # P: entry 2i -> i, 2i+1 -> i + r/2 (rotated part only)
    perm[:r] = np.concatenate([np.arange(0, r, 2), np.arange(1, r, 2)])
    inter = o.rope(x, pos, om, r, 1.0, 1)
    half = o.rope(np.ascontiguousarray(x[..., perm]), pos, om, r, 1.0, 0)
    back = np.empty_like(half)
    back[..., perm] = half
    assert _same_bits(back, inter)


def pin_rope_cos_sin_table(o):
    om = RNG.uniform(1e-4, 1.5, 16).astype(np.float32)
    tab = o.rope_cos_sin(om, 32, 3000)
    assert tab.shape == (3000, 16, 2)
    assert np.all(tab[0, :, 0] == 1.0) and np.all(tab[0, :, 1] == 0.0), "position 0: cos 1, sin 0"
    th = (np.arange(3000, dtype=np.float32)[:, None] * om[None, :]).astype(np.float64)  # the f32 angle
    assert np.all(np.abs(tab[..., 0] - np.cos(th)) <= 2 ** -24 * 1.0001), "cos within half an ulp of 1"
    assert np.all(np.abs(tab[..., 1] - np.sin(th)) <= 2 ** -24 * 1.0001)
    norm = tab[..., 0].astype(np.float64) ** 2 + tab[..., 1].astype(np.float64) ** 2
    assert np.all(np.abs(norm - 1.0) <= 2.5e-7)
    # the table drives the same rotation as the formed angles: rotate by hand
    x = _rand(5, 2, 32)
    pos = np.array([0, 1, 77, 2999, 1234], np.int32)
    y = o.rope(x, pos, om, 32, 1.0, 0)
    for t, p in enumerate(pos):
        c, sn = tab[p, :, 0], tab[p, :, 1]
        a, b = x[t, :, :16], x[t, :, 16:]
        assert _same_bits(y[t, :, :16], (a * c - b * sn).astype(np.float32))
        assert _same_bits(y[t, :, 16:], (a * sn + b * c).astype(np.float32))


def pin_qk_norm_rope_per_head(o):
    """QK-norm normalises each head over head_dim alone ("Operations", section 5),
    then rotates: against float64 torch rms_norm over the last dim of [T, H, D]
    followed by float64 rotations; heads are independent of one another."""
    T, H, D, r = 3, 4, 16, 12
    x = _rand(T, H, D, scale=2.0)
    x[:, 2] *= 50.0  # one loud head must not change its neighbours
    g = RNG.uniform(0.5, 1.5, D).astype(np.float32)
    pos = np.array([0, 5, 300], np.int32)
    om = RNG.uniform(1e-3, 1.0, r // 2).astype(np.float32)
    for layout in (0, 1):
        y = o.qk_norm_rope(x, g, 1e-5, pos, om, r, 1.0, layout)
        n = torch.nn.functional.rms_norm(torch.from_numpy(x).double(), (D,), torch.from_numpy(g).double(),
                                         1e-5).numpy()
        ref = _brute_rope(n, pos, om, r, 1.0, layout)
        assert np.allclose(y, ref, rtol=0, atol=4e-6 * np.abs(n).max()), layout
        quiet = x.copy()
        quiet[:, 2] /= 50.0
        y2 = o.qk_norm_rope(quiet, g, 1e-5, pos, om, r, 1.0, layout)
        for h in (0, 1, 3):
            assert _same_bits(y2[:, h], y[:, h]), "other heads must not depend on head 2"
    # with eps = 0, a power-of-two scale of one head leaves its output unchanged
    y0 = o.qk_norm_rope(x, g, 0.0, pos, om, r, 1.0, 0)
    xs = x.copy()
    xs[:, 1] *= np.float32(8.0)
    assert _same_bits(o.qk_norm_rope(xs, g, 0.0, pos, om, r, 1.0, 0), y0)


# ---- SiLU-mul ------------------------------------------------------------------

def pin_silu_mul_saturates_without_nan(o):
    g = np.array([-1e4, -1e4, 100.0, -100.0, 1e4, -88.0, 0.0], np.float32)
    u = np.array([2.0, -3.0, 1.5, 2.0, 0.25, 1.0, 7.0], np.float32)
    y = o.silu_mul(g, u)
    assert not np.isnan(y).any()
    assert y[0] == 0 and np.signbit(y[0]), "silu(-1e4) * u (u > 0) is -0"
    assert y[1] == 0 and not np.signbit(y[1]), "silu(-1e4) * u (u < 0) is +0"
    assert y[2] == np.float32(150.0), "large gate: y = g * u"
    assert y[3] == 0 and np.signbit(y[3])
    assert y[4] == np.float32(2500.0)
    assert 0 > y[5] > -1e-35
    assert y[6] == 0


def pin_silu_library(o):
    g = RNG.uniform(-80, 80, 4000).astype(np.float32)
    g[:100] = RNG.uniform(-1, 1, 100)
    u = _rand(4000, scale=2.0)
    y = o.silu_mul(g, u).astype(np.float64)
    ref = (torch.nn.functional.silu(torch.from_numpy(g).double()) * torch.from_numpy(u).double()).numpy()
    err = np.abs(y - ref) / np.maximum(np.abs(ref), 1e-300)
    assert err.max() <= 1e-6, err.max()


# ---- Sampling ("Operations", section 8) --------------------------------------------

def sampling_probs_f64(x, method, t=1.0, k=1, p=1.0):
    """The distribution each method draws from, in float64, written from the
    definition independently of the oracle: (probabilities per index, the
    order the draw walks, the smallest margin of any keep/cut decision)."""
    x = np.asarray(x, np.float64)
    valid = ~np.isnan(x)
    vi = np.nonzero(valid)[0]
    order_sorted = list(vi[np.lexsort((vi, -x[vi]))])  # descending value, then ascending index
    probs = np.zeros_like(x)
    margin = np.inf
    if method == "temperature" or method == "min_p":
        z = torch.from_numpy(np.where(valid, x / t, -np.inf))
        sm = torch.softmax(z, 0).numpy()
        if method == "min_p":
            thr = p * sm.max()
            keep = sm >= thr
            margin = np.min(np.abs(sm[valid] - thr)) / sm.max()
            sm = np.where(keep, sm, 0.0)
            sm = sm / sm.sum()
        probs = sm
        order = np.arange(len(x))
    else:
        cand = order_sorted[:k] if method == "top_k" else order_sorted
        z = torch.from_numpy(x[cand] / t)
        sm = torch.softmax(z, 0).numpy()
        if method == "top_p":
            c = np.cumsum(sm)
            keep = c <= p
            keep[0] = True
            margin = np.min(np.abs(c - p))
            sm = np.where(keep, sm, 0.0)
            sm = sm / sm.sum()
        probs[cand] = sm
        order = np.array(order_sorted)
    return probs, order, margin


def _grid_counts(o, x, method, n_grid, **kw):
    u = ((np.arange(n_grid) + 0.5) / n_grid).astype(np.float32)
    rows = np.repeat(np.asarray(x, np.float32).reshape(1, -1), n_grid, axis=0)
    drawn = o.sample(rows, method, u, **kw)
    # every method keeps at least one entry of a row that holds a number
    assert np.all(drawn >= 0), (method, "a row with numbers drew nothing")
    return np.bincount(drawn, minlength=rows.shape[1])


def pin_sampling_draws_in_proportion(o):
    """Inverse-CDF property: over a fine grid of u, each index is drawn
    n_grid * p_i times (+-2), p_i from the float64 definition."""
    for trial in range(6):
        x = _rand(60, scale=2.0)
        x[[5, 17]] = x[3]  # exact ties
        x[11] = np.nan
        for method, kw in (("temperature", dict(temperature=0.8)), ("top_k", dict(temperature=1.3, top_k=7)),
                           ("top_p", dict(temperature=0.9, top_p=0.6)), ("min_p", dict(temperature=1.0, min_p=0.2))):
            pr, order, margin = sampling_probs_f64(x, method, t=kw["temperature"], k=kw.get("top_k", 1),
                                                   p=kw.get("top_p", kw.get("min_p", 1.0)))
            if margin < 1e-4:
                continue  # a keep/cut decision within rounding of its threshold
            counts = _grid_counts(o, x, method, 4000, **kw)
            assert np.all(np.abs(counts - 4000 * pr) <= 2.5), (trial, method, np.abs(counts - 4000 * pr).max())
            assert counts[11] == 0, "NaN is never drawn"


def pin_sampling_limits(o):
    """Greedy is argmax; top-k with k = 1, and top-p with a tiny p (only the
    first entry is ever kept), give the argmax too; a row of NaN gives -1."""
    x = _rand(8, 300, scale=3.0)
    x[2, 7] = x[2, 250] = 50.0  # tie at the maximum: the lower index
    x[3] = np.nan
    u = RNG.random(8).astype(np.float32)
    want = o.argmax(x)
    assert np.array_equal(o.sample(x, "greedy", u), want)
    assert np.array_equal(o.sample(x, "top_k", u, temperature=0.7, top_k=1), want)
    assert np.array_equal(o.sample(x, "top_p", u, temperature=1.0, top_p=1e-9), want)
    assert o.sample(x[3:4], "temperature", [0.5])[0] == -1
    # min_p = 0 keeps everything: the same draws as temperature sampling
    assert np.array_equal(o.sample(x, "min_p", u, temperature=0.9, min_p=0.0),
                          o.sample(x, "temperature", u, temperature=0.9))


# ---- The seeded generator of sample_categorical (PCG64) ---------------------------
# numpy's PCG64 bit generator is the same generator (128-bit LCG with the
# default multiplier, XSL-RR output after each step), implemented
# independently: its state can be set to any (state, increment), stepped
# (random_raw) and jumped (advance), which pins the oracle's step, output
# permutation and jump-ahead.  The seeding procedure and the uniform are
# definitions ("Operations" section 8 leaves them open); they are checked by
# composing numpy's steps the way the definition says.

PCG_INC = (0x5851F42D4C957F2D << 64) | 0x14057B7EF767814F  # the generator's default increment
_M128 = (1 << 128) - 1


def _numpy_pcg(state: int, inc: int):
    bg = np.random.PCG64()
    bg.state = {"bit_generator": "PCG64", "state": {"state": state & _M128, "inc": inc & _M128},
                "has_uint32": 0, "uinteger": 0}
    return bg


def _rand128() -> int:
    return int.from_bytes(RNG.bytes(16), "little")


def pin_pcg64_steps_as_numpy(o):
    """Outputs and final state from arbitrary (state, odd increment) equal
    numpy's PCG64 random_raw from the same state."""
    for trial in range(20):
        state, inc = _rand128(), _rand128() | 1
        if trial == 0:
            state, inc = 0, PCG_INC
        got, end = o.pcg64_raw(state, inc, 64)
        bg = _numpy_pcg(state, inc)
        want = bg.random_raw(64)
        assert np.array_equal(got, want), (trial, got[:3], want[:3])
        assert end == bg.state["state"]["state"], trial


def pin_pcg64_jump_ahead(o):
    """The jump of delta steps equals numpy's advance(delta), for small,
    large and wrapping distances, and equals delta single steps."""
    for trial in range(8):
        state, inc = _rand128(), _rand128() | 1
        for delta in (0, 1, 2, 3, 7, 1000, 12345677, (1 << 40) + 7, (1 << 64) - 1, (1 << 64) + 3,
                      (1 << 127) + 5, _M128):
            bg = _numpy_pcg(state, inc)
            bg.advance(delta)
            assert o.pcg64_advance(state, inc, delta) == bg.state["state"]["state"], (trial, delta)
        _, stepped = o.pcg64_raw(state, inc, 513)
        assert o.pcg64_advance(state, inc, 513) == stepped


def pin_pcg64_seeding_and_uniforms(o):
    """Seeding: state 0, a step, plus the seed, a step (numpy's steps).  Draw
    j of the seeded stream is the output after j + 1 further steps; its
    uniform is the top 24 bits times 2^-24.  Consecutive windows of draws
    agree with one long run, and offsets past 2^64 continue the stream."""
    for seed in (0, 1, 42, 2 ** 63 + 11, 2 ** 64 - 1):
        bg = _numpy_pcg(0, PCG_INC)
        bg.random_raw(1)
        s1 = bg.state["state"]["state"]
        bg = _numpy_pcg(s1 + seed, PCG_INC)
        bg.random_raw(1)
        seeded = bg.state["state"]["state"]
        assert o.pcg64_seeded_state(seed) == seeded, seed
        for offset in (0, 1, 1000, 2 ** 32 + 5, 2 ** 64 - 3):
            bg = _numpy_pcg(seeded, PCG_INC)
            bg.advance(offset)
            raw = bg.random_raw(9)
            want = ((raw >> np.uint64(40)).astype(np.float64) * 2.0 ** -24).astype(np.float32)
            got = o.pcg64_uniforms(seed, offset, 9)
            assert _same_bits(got, want), (seed, offset, got, want)
            assert np.all((got >= 0) & (got < 1))
            if offset + 4 < 2 ** 64:
                assert _same_bits(o.pcg64_uniforms(seed, offset + 4, 5), got[4:])


def pin_pcg64_uniformity(o):
    """A million uniforms of one seed are flat over 256 bins (chi-square
    within six standard deviations of its mean), multiples of 2^-24 with
    mean 1/2; another seed's stream is uncorrelated with it."""
    n = 1 << 20
    u = o.pcg64_uniforms(7, 0, n).astype(np.float64)
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
    counts = np.bincount((u * 256).astype(np.int64), minlength=256)
    e = n / 256
    chi2 = float(((counts - e) ** 2 / e).sum())
    assert abs(chi2 - 255) < 6 * np.sqrt(2 * 255), chi2
    assert abs(u.mean() - 0.5) < 6 * np.sqrt(1 / 12 / n), u.mean()
    v = o.pcg64_uniforms(8, 0, n).astype(np.float64)
    assert abs(np.corrcoef(u, v)[0, 1]) < 6 / np.sqrt(n)


def pin_sampling_seeded_draws(o):
    """The seeded draw of row r is the draw at the uniform of stream draw
    offset + r: the same seed gives the same draws, another seed others."""
    x = _rand(64, 500, scale=2.0)
    for method, kw in (("temperature", dict(temperature=0.8)), ("top_k", dict(temperature=1.1, top_k=20)),
                       ("top_p", dict(temperature=0.9, top_p=0.8)), ("min_p", dict(temperature=1.0, min_p=0.1))):
        for seed, offset in ((3, 0), (3, 64), (2 ** 64 - 5, 2 ** 40)):
            bg = _numpy_pcg(o.pcg64_seeded_state(seed), PCG_INC)
            bg.advance(offset)
            u = ((bg.random_raw(64) >> np.uint64(40)).astype(np.float64) * 2.0 ** -24).astype(np.float32)
            got = o.sample_seeded(x, method, seed, offset, **kw)
            assert np.array_equal(got, o.sample(x, method, u, **kw)), (method, seed, offset)
            assert np.array_equal(got, o.sample_seeded(x, method, seed, offset, **kw))
        other = o.sample_seeded(x, method, 4, 0, **kw)
        assert not np.array_equal(other, o.sample_seeded(x, method, 3, 0, **kw)), method


# ---- Embedding / add / argmax / bf16 ---------------------------------------------

def pin_embedding_gathers_rows(o):
    table = _rand(50, 9)
    ids = np.array([7, 7, 0, 49, 3, 7, 12], np.int32)  # repeated and out of order
    out = o.embedding(table, ids)
    assert _same_bits(out, table[ids])
    for bad in ([50], [-1]):
        try:
            o.embedding(table, np.array(bad, np.int32))
        except ValueError:
            pass
        else:
            raise AssertionError("an id outside [0, V) must be reported")


def pin_add_in_place(o):
    a, b = _rand(1000), _rand(1000)
    assert _same_bits(o.add(a, b), a + b)
    ta = torch.from_numpy(a).bfloat16()
    tb = torch.from_numpy(b).bfloat16()
    wide_a, wide_b = ta.float().numpy(), tb.float().numpy()
    got = o.bf16_round(o.add(wide_a, wide_b))
    want = (ta + tb).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), "bf16 add: f32 sum rounded to nearest even"


def pin_bf16_storage(o):
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 3.4e38, -3.4e38,
                         1e-40, -1e-40, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9,
                         1.0 + 2 ** -8 + 2 ** -9, 65504.0, 2.0 ** -126], np.float32)
    vals = np.concatenate([specials, _rand(20000, scale=100.0),
                           (np.arange(1, 5000, dtype=np.uint32) << 15).view(np.float32)])
    got = o.bf16_round(vals)
    want = torch.from_numpy(vals).bfloat16().view(torch.int16).numpy().view(np.uint16)
    finite = ~np.isnan(vals)
    assert np.array_equal(got[finite], want[finite])
    assert np.all(np.isnan(o.bf16_widen(got[~finite])))
    back = o.bf16_widen(want)
    assert _same_bits(back[finite],
                      torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy()[finite])


def pin_argmax_ties_nan_and_empty(o):
    nan, inf = np.nan, np.inf
    assert list(o.argmax(np.array([[3, 9, 9, 1], [9, 3, 9, 9]], np.float32))) == [1, 0]
    assert int(o.argmax(np.array([nan, 1, 2, 2], np.float32))[0]) == 2
    assert int(o.argmax(np.array([nan, nan], np.float32))[0]) == -1
    assert int(o.argmax(np.array([-inf, -inf, -inf], np.float32))[0]) == 0
    assert int(o.argmax(np.array([nan, -inf, nan], np.float32))[0]) == 1
    assert int(o.argmax(np.array([-0.0, 0.0], np.float32))[0]) == 0
    assert int(o.argmax(np.array([0.0, -0.0], np.float32))[0]) == 0
    assert int(o.argmax(np.array([1, inf, nan, inf], np.float32))[0]) == 1
    assert o.argmax_one(np.zeros(0, np.float32)) == -1
    try:
        o.argmax(np.zeros((3, 0), np.float32))
    except ValueError:
        pass
    else:
        raise AssertionError("an empty row must be rejected")


def pin_argmax_library(o):
    x = _rand(40, 513)
    x[RNG.random(x.shape) < 0.05] = np.nan
    x[3, 100] = x[3, 300] = 50.0
    x[4, :] = np.round(x[4] * 2) / 2  # many exact ties
    got = o.argmax(x)
    assert np.array_equal(got, np.nanargmax(x, axis=1)), "nanargmax: first max, NaN ignored"


PINS = {name[4:]: fn for name, fn in dict(globals()).items() if name.startswith("pin_")}

# planted mistake (pitfalls table, section 5) -> the pin that must reject it
KILLS = {
    1: "rmsnorm_eps_is_inside_the_root",
    2: "rmsnorm_eps_is_inside_the_root",
    3: "hand_example",
    4: "rope_interleaved_layout_and_position_zero",
    5: "rope_interleaved_layout_and_position_zero",
    6: "rope_is_a_rotation",
    7: "rope_partial_rotary_and_scaling",
    8: "rope_partial_rotary_and_scaling",
    9: "silu_mul_saturates_without_nan",
    10: "silu_mul_saturates_without_nan",
    11: "embedding_gathers_rows",
    12: "argmax_ties_nan_and_empty",
    13: "argmax_ties_nan_and_empty",
    14: "argmax_ties_nan_and_empty",
    15: "rmsnorm_rows_are_independent_and_in_place",
    16: "qk_norm_rope_per_head",
    17: "layernorm",
    18: "sampling_limits",
    19: "rope_multi_axis",
    20: "sampling_draws_in_proportion",
    21: "sampling_limits",
    22: "pcg64_steps_as_numpy",
    23: "pcg64_jump_ahead",
    24: "pcg64_steps_as_numpy",
}
