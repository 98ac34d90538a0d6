"""LayerNorm on the GPU against the oracle, through the C ABI: ragged widths,
both storage types, with and without bias, the unaligned path (same bits),
in place, and batch invariance.

Bar: |y - y_oracle| <= rtol * (max over the row of |y_oracle - b| + |b|),
rtol 1e-5 (f32) / 1e-2 (bf16): x - mean can cancel to nearly zero, so the
error is bounded against the row's scale rather than each entry."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import RTOL, bits, to_dev, to_f32, widen
from synth import normal, to_bf16, uniform

pytestmark = pytest.mark.gpu


def _case(rows, d, dtype, bias=True, seed=21):
    x = normal(seed, f"ln.x.{rows}.{d}", (rows, d), 0.5, 2.0)
    g = uniform(seed, f"ln.g.{d}", (d,), 0.5, 1.5)
    b = normal(seed, f"ln.b.{d}", (d,), 0.0, 0.3) if bias else None
    if dtype == "bf16":
        x, g = to_bf16(x), to_bf16(g)
        b = to_bf16(b) if bias else None
    return x, g, b


def _check(x, g, b, y_dev, dtype, what):
    gw = widen(g)
    bw = None if b is None else widen(b)
    want = oracle.get().layernorm(widen(x), gw, bw, 1e-5).astype(np.float64)
    got = to_f32(y_dev).astype(np.float64)
    bb = 0.0 if bw is None else np.abs(bw.astype(np.float64))
    centred = want - (0.0 if bw is None else bw)
    tol = RTOL[dtype] * (np.abs(centred).max(axis=-1, keepdims=True) + bb) + 1e-30
    bad = np.abs(got - want) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} entries off, first {np.argwhere(bad)[0].tolist()}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [1, 3, 8, 64, 100, 1000, 4096, 4100, 16384, 20000])
@pytest.mark.parametrize("bias", [True, False])
def test_layernorm_shapes(dtype, d, bias):
    rows = 23 if d <= 4100 else 4
    x, g, b = _case(rows, d, dtype, bias)
    y = gbe.layernorm(to_dev(x), to_dev(g), None if b is None else to_dev(b), 1e-5)
    _check(x, g, b, y, dtype, f"layernorm {dtype} d={d} bias={bias}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_layernorm_unaligned_in_place_and_batches(dtype):
    d = 4096
    x, g, b = _case(64, d, dtype)
    xd, gd, bd = to_dev(x), to_dev(g), to_dev(b)
    ref = gbe.layernorm(xd, gd, bd, 1e-5)
    buf = torch.empty(64 * d + 1, dtype=xd.dtype, device="cuda")
    xs = buf[1:].view(64, d)
    xs.copy_(xd)
    ys = torch.empty(64 * d + 1, dtype=xd.dtype, device="cuda")[1:].view(64, d)
    gbe.gbe_layernorm(xs, gd, bd, ys, 1e-5)
    assert np.array_equal(bits(ys), bits(ref)), "unaligned path"
    for n in (1, 5, 33, 64):
        assert np.array_equal(bits(gbe.layernorm(xd[:n].contiguous(), gd, bd, 1e-5)), bits(ref[:n])), n
    xi = xd.clone()
    gbe.gbe_layernorm(xi, gd, bd, xi, 1e-5)
    assert np.array_equal(bits(xi), bits(ref)), "in place"


def test_constant_row_gives_bias():
    d = 256
    x = torch.full((3, d), 2.5, device="cuda")
    g = torch.rand(d, device="cuda") + 0.5
    b = torch.randn(d, device="cuda")
    y = gbe.layernorm(x, g, b, 1e-5)
    assert torch.equal(y, b.expand(3, d))
