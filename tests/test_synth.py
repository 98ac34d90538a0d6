"""The seeded generator: replays plain splitmix64, draws slices consistently,
and lays out the workloads' shapes, dtypes and planted structure (CPU only)."""
import numpy as np

import synth
from synth import workloads as W

M64 = (1 << 64) - 1


def _splitmix64(state, n):
    """Sequential splitmix64 (Steele, Lea, Flood 2014), written out plainly."""
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_stream_is_sequential_splitmix64():
    key = synth.stream_key(7, "some.tensor")
    assert list(synth.raw_u64(7, "some.tensor", 50)) == _splitmix64(key, 50)
    assert list(synth.raw_u64(7, "some.tensor", 10, offset=40)) == _splitmix64(key, 50)[40:]


def test_slices_and_threads_agree():
    full = synth.normal(3, "x", (300000,), 0.0, 2.0)
    part = synth.normal(3, "x", (1000,), 0.0, 2.0, offset=123456)
    assert np.array_equal(full[123456:124456], part)
    assert not np.array_equal(full, synth.normal(4, "x", (300000,), 0.0, 2.0))
    assert not np.array_equal(full, synth.normal(3, "y", (300000,), 0.0, 2.0))


def test_distributions():
    z = synth.normal(1, "z", (400000,), 0.5, 2.0).astype(np.float64)
    assert abs(z.mean() - 0.5) < 0.02 and abs(z.std() - 2.0) < 0.02
    u = synth.uniform(1, "u", (400000,), 0.5, 1.5)
    assert u.min() >= 0.5 and u.max() <= 1.5 and abs(u.mean() - 1.0) < 0.01
    k = synth.randint(1, "k", (400000,), 0, 1000)
    assert k.min() == 0 and k.max() == 999
    c = synth.normal(1, "c", (400000,), 0.0, 1.0, clip=2.0)
    assert c.max() == np.float32(2.0) and c.min() == np.float32(-2.0)


def test_bf16_storage_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)
    b = synth.to_bf16(x)
    assert list(b) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000]
    big = synth.normal_bf16(2, "b", (1000, 77), 0.0, 1.0, chunk=4096)
    assert np.array_equal(big, synth.to_bf16(synth.normal(2, "b", (1000, 77), 0.0, 1.0)))


def test_workload_shapes_and_plants():
    a, p = W.cases(W.TINY)["rmsnorm"]()
    assert a["x"].shape == (4, 64) and np.all(a["x"][3] == 0) and p["eps"] == 1e-5
    a, p = W.cases(W.TINY)["argmax"]()
    x = a["x"]
    assert np.isnan(x[1, 0]) and np.all(np.isnan(x[2])) and np.all(x[3] == -np.inf)
    assert np.sum(x[0] == np.float32(7.5)) == 2
    a, p = W.cases(W.TINY)["silu_mul"]()
    assert a["gate"][0, 0] == -1e4 and a["up"][1, 0] < 0
    a, p = W.cases(W.DECODE)["rope_q"]()
    assert a["x"].dtype == np.uint16 and a["x"].shape == (64, 32, 128)
    assert a["inv_freq"].shape == (64,) and a["pos"].max() < 8192
    a, p = W.cases(W.ROPE_VARIANTS)["rope_k"](rows=(10, 20))
    full_pos = W.cases(W.ROPE_VARIANTS)["rope_k"](rows=(0, 20))[0]["pos"]
    assert np.array_equal(a["pos"], full_pos[10:20]) and p["mu"] == 1.2 and p["in_place"]
    om = a["inv_freq"]
    assert om.shape == (64,) and abs(om[16] / om[15] - 0.125 * 10000 ** (-2 / 64)) < 1e-6


def test_planted_ties_are_row_maxima():
    a, p = W.cases(W.WIDE)["argmax"](rows=(0, 60))
    x = a["x"]
    assert x.shape == (60, 152064)
    frac_nan = np.isnan(x).mean()
    assert 0.008 < frac_nan < 0.012
    top = np.float32(30.0)
    tied = np.where((x == top).sum(axis=1) == 2)[0]
    assert len(tied) >= 1
    for r in tied:
        assert np.nanmax(x[r]) == top
    same = W.cases(W.WIDE)["argmax"](rows=(20, 25))[0]["x"]
    assert np.array_equal(same, x[20:25], equal_nan=True)
