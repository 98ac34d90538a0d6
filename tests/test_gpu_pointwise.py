"""SiLU-mul, residual add and embedding gather on the GPU against the oracle,
through the C ABI: saturation and ragged tails, aliases, unaligned paths, the
full-size workloads, and the embedding id guard."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import assert_rel, bits, to_dev, to_f32, widen
from synth import normal, randint, to_bf16
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _silu_check(g, u, dtype, what):
    y = gbe.silu_mul(to_dev(g), to_dev(u))
    got = to_f32(y)
    assert not np.isnan(got).any()
    assert_rel(got, oracle.get().silu_mul(widen(g), widen(u)), dtype, what)
    return y


def test_silu_tiny_saturation():
    a, p = W.cases(W.TINY)["silu_mul"]()
    y = to_f32(_silu_check(a["gate"], a["up"], "f32", "tiny silu"))
    g, u = a["gate"], a["up"]
    assert y[0, 0] == 0 and np.signbit(y[0, 0]) == (u[0, 0] > 0)   # silu(-1e4) = -0, times up
    assert y[0, 1] == np.float32(1e4) * u[0, 1]                     # large gate: g * u
    assert y[1, 0] == 0 and not np.signbit(y[1, 0])                  # -0 * (negative up) = +0
    assert y[1, 1] == np.float32(100.0) * u[1, 1]
    assert y[1, 2] == 0


@pytest.mark.parametrize("workload", [W.DECODE, W.PREFILL])
def test_silu_workload_full(workload):
    a, p = W.cases(workload)["silu_mul"]()
    _silu_check(a["gate"], a["up"], "bf16", f"silu {workload}")


def test_silu_dense_sweep_of_the_f32_range():
    """Every 64th f32 bit pattern of the gate over [-104, 90] (about 35
    million values, up = 1): the hardware exponential and reciprocal stay
    within the f32 bar of the oracle's libm quotient everywhere, including
    the exponent overflow edge near g = -88.7 where the exact value is
    tiny (the bar's 1e-30 floor) and beyond it, where both give -0."""
    neg = np.arange(0, np.float32(104.0).view(np.uint32), 64, dtype=np.uint32) | np.uint32(0x80000000)
    pos = np.arange(0, np.float32(90.0).view(np.uint32), 64, dtype=np.uint32)
    g = np.concatenate([neg, pos]).view(np.float32)
    u = np.ones_like(g)
    got = to_f32(gbe.silu_mul(to_dev(g), to_dev(u)))
    want = oracle.get().silu_mul(g, u)
    assert not np.isnan(got).any()
    assert_rel(got, want, "f32", "silu sweep")
    w = np.asarray(want, np.float64)
    big = np.abs(w) > 1e-30
    worst = np.max(np.abs(np.asarray(got, np.float64)[big] - w[big]) / np.abs(w[big]))
    print(f"silu f32 sweep: {g.size} gates, largest relative error {worst:.3g}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 3, 7, 8, 9, 1000, 1023, 4096 * 4 + 5, 1 << 20])
def test_silu_and_add_ragged(dtype, n):
    g = normal(9, f"t.silu.g.{n}", (n,), 0.0, 20.0)
    u = normal(9, f"t.silu.u.{n}", (n,), 0.0, 2.0)
    if dtype == "bf16":
        g, u = to_bf16(g), to_bf16(u)
    _silu_check(g, u, dtype, f"silu n={n}")
    y = gbe.add(to_dev(g), to_dev(u))
    s = oracle.get().add(widen(g), widen(u))
    want = oracle.get().bf16_round(s) if dtype == "bf16" else s.view(np.uint32)
    assert np.array_equal(bits(y), want), f"add n={n}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pointwise_aliases_and_unaligned(dtype):
    n = 10007
    g = normal(10, "t.pw.g", (n,), 0.0, 3.0)
    u = normal(10, "t.pw.u", (n,), 0.0, 3.0)
    if dtype == "bf16":
        g, u = to_bf16(g), to_bf16(u)
    ref_s = gbe.silu_mul(to_dev(g), to_dev(u))
    ref_a = gbe.add(to_dev(g), to_dev(u))
    gd, ud = to_dev(g), to_dev(u)
    gbe.gbe_silu_mul(gd, ud, gd)                  # y == gate
    assert np.array_equal(bits(gd), bits(ref_s))
    gd = to_dev(g)
    gbe.gbe_silu_mul(gd, ud, ud)                  # y == up
    assert np.array_equal(bits(ud), bits(ref_s))
    ud = to_dev(u)
    gbe.gbe_add(gd, ud, gd)                       # y == a
    assert np.array_equal(bits(gd), bits(ref_a))
    # element-offset views take the scalar path with the same bits
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    bg = torch.empty(n + 1, dtype=tdt, device="cuda")[1:]
    bu = torch.empty(n + 1, dtype=tdt, device="cuda")[1:]
    by = torch.empty(n + 1, dtype=tdt, device="cuda")[1:]
    bg.copy_(to_dev(g))
    bu.copy_(to_dev(u))
    gbe.gbe_silu_mul(bg, bu, by)
    assert np.array_equal(bits(by), bits(ref_s))
    gbe.gbe_add(bg, bu, by)
    assert np.array_equal(bits(by), bits(ref_a))


def test_add_prefill_full():
    a, p = W.cases(W.PREFILL)["add"]()
    y = gbe.add(to_dev(a["a"]), to_dev(a["b"]))
    o = oracle.get()
    assert np.array_equal(bits(y), o.bf16_round(o.add(widen(a["a"]), widen(a["b"]))))


def test_embedding_tiny():
    a, p = W.cases(W.TINY)["embedding"]()
    y = gbe.embedding(to_dev(a["table"]), to_dev(a["ids"]))
    assert np.array_equal(to_f32(y), oracle.get().embedding(a["table"], a["ids"]))


def test_embedding_prefill_full():
    a, p = W.cases(W.PREFILL)["embedding"]()
    table = to_dev(a["table"])
    y = gbe.embedding(table, to_dev(a["ids"]))
    want = oracle.get().embedding(widen(a["table"]), a["ids"])
    assert np.array_equal(to_f32(y).view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [1, 5, 8, 64, 130, 4096, 40000])
def test_embedding_shapes_repeats_and_bad_ids(dtype, d):
    V = 300
    table = normal(12, f"t.emb.{d}", (V, d), 0.0, 1.0)
    if dtype == "bf16":
        table = to_bf16(table)
    ids = np.array([7, 7, 0, 299, 3, 7, 12, 150] * 5, np.int32)
    y = gbe.embedding(to_dev(table), to_dev(ids))
    assert np.array_equal(bits(y), table[ids].view(bits(y).dtype))
    bad = ids.copy()
    bad[[1, 5, 9]] = [-1, 300, 1 << 30]
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = gbe.embedding(to_dev(table), to_dev(bad), bad_id_count=cnt)
    got = bits(y)
    assert int(cnt.item()) == 3
    ok = np.ones(len(bad), bool)
    ok[[1, 5, 9]] = False
    assert np.array_equal(got[ok], table[bad[ok]].view(got.dtype))
    assert np.all(got[~ok] == 0)
