"""RoPE on the GPU against the oracle, through the C ABI: both layouts,
partial rotary width, attention scaling, in place and out of place, the
vector and scalar paths, and the full-size workloads (positions up to 2^20)."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import assert_rope_close, bits, to_dev, to_f32, widen
from synth import normal, randint, to_bf16
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _run_case(a, p, in_place=None):
    x = a["x"]
    xd = to_dev(x)
    pos, om = to_dev(a["pos"]), to_dev(a["inv_freq"])
    ip = p["in_place"] if in_place is None else in_place
    y = gbe.rope(xd, pos, om, p["r"], p["mu"], p["layout"], in_place=ip)
    want = oracle.get().rope(widen(x), a["pos"], a["inv_freq"], p["r"], p["mu"], p["layout"])
    got = to_f32(y)
    assert_rope_close(got, want, widen(x), p["r"], p["mu"], p["layout"], p["dtype"],
                      f"rope layout {p['layout']} r={p['r']}")
    # entries past r pass through bit for bit
    assert np.array_equal(bits(y)[..., p["r"]:], x[..., p["r"]:].view(bits(y).dtype))
    return y


@pytest.mark.parametrize("name", ["rope_q"])
def test_tiny(name):
    a, p = W.cases(W.TINY)[name]()
    for layout in (0, 1):
        p2 = dict(p, layout=layout)
        _run_case(a, p2)


@pytest.mark.parametrize("name", ["rope_q", "rope_k"])
def test_decode_bf16(name):
    a, p = W.cases(W.DECODE)[name]()
    _run_case(a, p)


@pytest.mark.parametrize("name", ["rope_q", "rope_k", "rope_q_interleaved", "rope_k_interleaved"])
def test_prefill_bf16_full(name):
    a, p = W.cases(W.PREFILL)[name]()
    _run_case(a, p)


@pytest.mark.parametrize("name", ["rope_q", "rope_k"])
def test_rope_variants_f32_full_in_place(name):
    a, p = W.cases(W.ROPE_VARIANTS)[name]()
    y = _run_case(a, p)  # in place, as the workload says
    # the same call out of place gives the same bits
    y2 = gbe.rope(to_dev(a["x"]), to_dev(a["pos"]), to_dev(a["inv_freq"]), p["r"], p["mu"], p["layout"])
    assert np.array_equal(bits(y), bits(y2))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("T,H,D,r", [(1, 1, 2, 2), (5, 3, 10, 6), (7, 2, 128, 64), (33, 4, 64, 64),
                                     (17, 5, 96, 32), (3, 2, 130, 128), (9, 1, 12, 0), (40, 8, 128, 128)])
def test_shapes(dtype, layout, T, H, D, r):
    x = normal(5, f"t.rope.{T}.{H}.{D}", (T, H, D), 0.0, 1.0)
    if dtype == "bf16":
        x = to_bf16(x)
    pos = randint(5, f"t.rope.pos.{T}", (T,), 0, 1 << 20)
    om = (10000.0 ** (-2.0 * np.arange(max(r // 2, 1)) / max(r, 2))).astype(np.float32)
    for mu in (1.0, 1.2):
        _run_case({"x": x, "pos": pos, "inv_freq": om},
                  {"dtype": dtype, "r": r, "mu": mu, "layout": layout, "in_place": False})
        _run_case({"x": x, "pos": pos, "inv_freq": om},
                  {"dtype": dtype, "r": r, "mu": mu, "layout": layout, "in_place": True})


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_position_zero_is_identity_and_mu2_doubles(dtype):
    x = normal(6, "t.rope.id", (6, 4, 64), 0.0, 1.0)
    if dtype == "bf16":
        x = to_bf16(x)
    om = (10000.0 ** (-2.0 * np.arange(32) / 64)).astype(np.float32)
    pos0 = np.zeros(6, np.int32)
    for layout in (0, 1):
        y = gbe.rope(to_dev(x), to_dev(pos0), to_dev(om), 64, 1.0, layout)
        assert np.array_equal(bits(y), x.view(bits(y).dtype))
    if dtype == "f32":
        pos = np.arange(6, dtype=np.int32) * 1000
        y1 = gbe.rope(to_dev(x), to_dev(pos), to_dev(om), 64, 1.0, 0)
        y2 = gbe.rope(to_dev(x), to_dev(pos), to_dev(om), 64, 2.0, 0)
        assert torch.equal(y2, y1 * 2)


def test_unaligned_path_same_bits():
    x = normal(7, "t.rope.u", (9, 4, 128), 0.0, 1.0)
    om = (500000.0 ** (-2.0 * np.arange(64) / 128)).astype(np.float32)
    pos = randint(7, "t.rope.u.pos", (9,), 0, 8192)
    xd = to_dev(x)
    for layout in (0, 1):
        y = gbe.rope(xd, to_dev(pos), to_dev(om), 128, 1.0, layout)
        buf = torch.empty(x.size + 1, dtype=torch.float32, device="cuda")
        xs = buf[1:].view(9, 4, 128)
        xs.copy_(xd)
        ys = torch.empty(x.size + 1, dtype=torch.float32, device="cuda")[1:].view(9, 4, 128)
        gbe.gbe_rope(xs, ys, to_dev(pos), to_dev(om), 128, 1.0, layout)
        assert np.array_equal(bits(ys), bits(y))
