"""Multi-axis RoPE (gbe_rope_multi) on the GPU against the oracle, through
the C ABI: video-style splits of head_dim (uneven slices too), both
layouts and storage types, in place; one axis equals gbe_rope bit for bit."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import RTOL, bits, to_dev, to_f32, widen
from synth import normal, randint, to_bf16

pytestmark = pytest.mark.gpu


def _om(dims, bases):
    return np.concatenate([(b ** (-2.0 * np.arange(d // 2) / d)) for d, b in zip(dims, bases)]).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("dims,D", [([44, 42, 42], 128), ([16, 24, 24], 128), ([32, 32], 72), ([8], 8)])
def test_against_oracle(dtype, layout, dims, D):
    T, H = 37, 6
    x = normal(31, f"rm.x.{D}.{len(dims)}", (T, H, D), 0.0, 1.0)
    if dtype == "bf16":
        x = to_bf16(x)
    A = len(dims)
    pos = randint(31, f"rm.pos.{A}", (T, A), 0, 4096)
    om = _om(dims, [10000.0, 20000.0, 30000.0][:A])
    for in_place in (False, True):
        xd = to_dev(x)
        y = xd if in_place else torch.empty_like(xd)
        gbe.gbe_rope_multi(xd, y, to_dev(pos), dims, to_dev(om), 1.05, layout)
        want = oracle.get().rope_multi(widen(x), pos, dims, om, 1.05, layout)
        got = to_f32(y)
        scale = 1.05 * np.abs(widen(x)).max(axis=-1, keepdims=True) * 1.5
        assert np.all(np.abs(got - want) <= RTOL[dtype] * scale), (dims, in_place)
        rot = sum(dims)
        assert np.array_equal(bits(y)[..., rot:], x[..., rot:].view(bits(y).dtype)), "tail passes through"


def test_one_axis_equals_rope():
    x = normal(32, "rm.one", (20, 4, 64), 0.0, 1.0)
    pos = randint(32, "rm.one.pos", (20,), 0, 9000)
    om = (10000.0 ** (-2.0 * np.arange(32) / 64)).astype(np.float32)
    for layout in (0, 1):
        y1 = torch.empty(20, 4, 64, device="cuda")
        gbe.gbe_rope_multi(to_dev(x), y1, to_dev(pos), [64], to_dev(om), 1.0, layout)
        y2 = gbe.rope(to_dev(x), to_dev(pos), to_dev(om), 64, 1.0, layout)
        assert np.array_equal(bits(y1), bits(y2))


def test_bad_axes_are_refused():
    L = gbe.lib()
    import ctypes
    s = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(4, 2, 16, device="cuda")
    pos = torch.zeros(8, dtype=torch.int32, device="cuda")
    om = torch.ones(8, device="cuda")
    dims = (ctypes.c_int64 * 2)(10, 8)  # 18 > D = 16
    assert L.gbe_rope_multi(x.data_ptr(), x.data_ptr(), pos.data_ptr(), 4, 2, 16, 2, ctypes.cast(dims, ctypes.c_void_p),
                            om.data_ptr(), 1.0, 0, 0, s) == 6
    dims = (ctypes.c_int64 * 2)(7, 8)  # odd
    assert L.gbe_rope_multi(x.data_ptr(), x.data_ptr(), pos.data_ptr(), 4, 2, 16, 2, ctypes.cast(dims, ctypes.c_void_p),
                            om.data_ptr(), 1.0, 0, 0, s) == 6
    assert L.gbe_rope_multi(x.data_ptr(), x.data_ptr(), pos.data_ptr(), 4, 2, 16, 9, None, om.data_ptr(), 1.0, 0, 0,
                            s) == 2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("H", [6, 24, 12, 7])
def test_vector_path_equals_scalar(dtype, layout, H):
    """The (t, h, w) = (32, 48, 48) split of head_dim 128 takes the 16-byte
    vector kernel (at 24 and 12 heads, bf16 half layout: three heads a thread
    and four head chunks sharing the angles; at 6 and 7 heads, or f32: four
    heads and two chunks, or none); the same data one element off alignment
    takes the scalar one: the two agree bit for bit, in place and out of
    place."""
    T, D, dims = 50, 128, [32, 48, 48]
    x = normal(33, f"rm.vec.{H}", (T, H, D), 0.0, 1.0)
    if dtype == "bf16":
        x = to_bf16(x)
    pos = randint(33, "rm.vec.pos", (T, 3), 0, 300)
    om = _om(dims, [10000.0, 10000.0, 10000.0])
    xd, pd, od = to_dev(x), to_dev(pos), to_dev(om)
    y = torch.empty_like(xd)
    gbe.gbe_rope_multi(xd, y, pd, dims, od, 1.0, layout)
    buf = torch.empty(T * H * D + 1, dtype=xd.dtype, device="cuda")
    xs = buf[1:].view(T, H, D)
    xs.copy_(xd)
    ys = torch.empty(T * H * D + 1, dtype=xd.dtype, device="cuda")[1:].view(T, H, D)
    gbe.gbe_rope_multi(xs, ys, pd, dims, od, 1.0, layout)
    assert np.array_equal(bits(ys), bits(y)), "scalar path"
    gbe.gbe_rope_multi(xs, xs, pd, dims, od, 1.0, layout)
    assert np.array_equal(bits(xs), bits(y)), "in place"
    want = oracle.get().rope_multi(widen(x), pos, dims, om, 1.0, layout)
    scale = np.abs(widen(x)).max(axis=-1, keepdims=True) * 1.5
    assert np.all(np.abs(to_f32(y) - want) <= RTOL[dtype] * scale)
