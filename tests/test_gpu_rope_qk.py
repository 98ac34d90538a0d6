"""RoPE of q and k in one launch (gbe_rope_qk) on the GPU, through the C ABI:
equal bit for bit to two gbe_rope calls, correct on q/k slices of a fused
QKV buffer (v untouched), the cos/sin table against the oracle's, and
table-driven rotation equal bit for bit to formed angles (also for positions
past the table)."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import assert_rope_close, bits, to_dev, to_f32, widen
from synth import normal, randint, to_bf16
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _om(r, base=10000.0):
    return (base ** (-2.0 * np.arange(r // 2) / r)).astype(np.float32)


def _x(seed, name, shape, dtype):
    x = normal(seed, name, shape, 0.0, 1.0)
    return to_bf16(x) if dtype == "bf16" else x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("T,Hq,Hk,D,r", [(7, 4, 2, 64, 64), (33, 32, 8, 128, 128), (5, 3, 1, 128, 64),
                                         (9, 2, 2, 10, 6), (1, 1, 1, 2, 2)])
def test_fused_equals_separate(dtype, layout, T, Hq, Hk, D, r):
    q = _x(1, f"qk.q.{T}.{D}", (T, Hq, D), dtype)
    k = _x(1, f"qk.k.{T}.{D}", (T, Hk, D), dtype)
    pos = to_dev(randint(1, f"qk.pos.{T}", (T,), 0, 1 << 20))
    om = to_dev(_om(r))
    yq = gbe.rope(to_dev(q), pos, om, r, 1.2, layout)
    yk = gbe.rope(to_dev(k), pos, om, r, 1.2, layout)
    qd, kd = to_dev(q), to_dev(k)
    qo, ko = torch.empty_like(qd), torch.empty_like(kd)
    gbe.gbe_rope_qk(qd, qo, kd, ko, pos, om, r, 1.2, layout)
    assert np.array_equal(bits(qo), bits(yq)) and np.array_equal(bits(ko), bits(yk))
    gbe.gbe_rope_qk(qd, qd, kd, kd, pos, om, r, 1.2, layout)  # in place
    assert np.array_equal(bits(qd), bits(yq)) and np.array_equal(bits(kd), bits(yk))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_qkv_buffer_in_place(dtype, layout):
    """q and k are column slices of one [T, (Hq + 2 Hk) D] buffer; v is untouched."""
    T, Hq, Hk, D, r = 64, 32, 8, 128, 128
    qkv = _x(2, "qk.qkv", (T, (Hq + 2 * Hk) * D), dtype)
    pos = randint(2, "qk.qkv.pos", (T,), 0, 8192)
    om = _om(r, 500000.0)
    buf = to_dev(qkv)
    q = buf[:, :Hq * D].view(T, Hq, D)
    k = buf[:, Hq * D:(Hq + Hk) * D].view(T, Hk, D)
    gbe.gbe_rope_qk(q, q, k, k, to_dev(pos), to_dev(om), r, 1.0, layout)
    got = bits(buf)
    v0 = (Hq + Hk) * D
    assert np.array_equal(got[:, v0:], qkv[:, v0:].view(got.dtype)), "v must be untouched"
    o = oracle.get()
    src = widen(qkv)
    for lo, H in ((0, Hq), (Hq * D, Hk)):
        x = np.ascontiguousarray(src[:, lo:lo + H * D].reshape(T, H, D))
        want = o.rope(x, pos, om, r, 1.0, layout)
        have = to_f32(buf[:, lo:lo + H * D].reshape(T, H, D))
        assert_rope_close(have, want, x, r, 1.0, layout, dtype, f"qkv slice at {lo}")


def test_qkv_unaligned_stride_takes_scalar_path_same_bits():
    """A token stride that breaks 16-byte alignment runs the scalar path, same bits."""
    T, H, D, r = 17, 3, 16, 16
    x = _x(3, "qk.sc", (T, H, D), "f32")
    pos = to_dev(randint(3, "qk.sc.pos", (T,), 0, 5000))
    om = to_dev(_om(r))
    ref = gbe.rope(to_dev(x), pos, om, r, 1.0, 0)
    stride = H * D + 1  # 49 f32 = 196 bytes: not a multiple of 16
    buf = torch.zeros(T * stride, dtype=torch.float32, device="cuda")
    view = buf.as_strided((T, H, D), (stride, D, 1))
    view.copy_(to_dev(x))
    gbe.gbe_rope_qk(view, view, None, None, pos, om, r, 1.0, 0)
    assert np.array_equal(bits(view.contiguous()), bits(ref))
    pad = buf.view(T, stride)[:, H * D:]
    assert torch.all(pad == 0), "padding between tokens untouched"


@pytest.mark.parametrize("r", [2, 16, 64, 128])
def test_cos_sin_table_against_oracle(r):
    om = _om(r, 500000.0)
    L = 4096
    tab = gbe.rope_cos_sin(to_dev(om), r, L).cpu().numpy()
    want = oracle.get().rope_cos_sin(om, r, L)
    assert np.all(np.abs(tab.astype(np.float64) - want) <= 4e-7), np.abs(tab - want).max()
    assert np.all(tab[0, :, 0] == 1.0) and np.all(tab[0, :, 1] == 0.0)


def test_cos_sin_of_large_angles_against_oracle():
    """Angles up to 2^23 rad: frequencies 1 and 8 at every position below
    2^20 + 3 (the quarter-turn reduction up to 2^22, sincosf whole beyond),
    plus frequencies whose products land on and near multiples of pi/2."""
    om = np.array([1.0, 8.0, 0.7853982, 1.5707964], np.float32)
    r, L = 8, (1 << 20) + 3
    tab = gbe.rope_cos_sin(to_dev(om), r, L).cpu().numpy()
    want = oracle.get().rope_cos_sin(om, r, L)
    err = np.abs(tab.astype(np.float64) - want)
    assert np.all(err <= 4e-7), (err.max(), np.unravel_index(err.argmax(), err.shape))
    assert np.all(tab[0, :, 0] == 1.0) and np.all(tab[0, :, 1] == 0.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_cached_equals_formed(dtype, layout):
    T, Hq, Hk, D, r = 40, 8, 2, 128, 64
    q = _x(4, "qk.c.q", (T, Hq, D), dtype)
    k = _x(4, "qk.c.k", (T, Hk, D), dtype)
    pos = randint(4, "qk.c.pos", (T,), 0, 3000)
    pos[:5] = [0, 1, 2047, 2048, 2999]  # the last two lie past a 2048-entry table
    om = to_dev(_om(r))
    table = gbe.rope_cos_sin(om, r, 2048)
    outs = []
    for cache in (None, table):
        qd, kd = to_dev(q), to_dev(k)
        gbe.gbe_rope_qk(qd, qd, kd, kd, to_dev(pos), om, r, 1.0, layout, cos_sin=cache)
        outs.append((bits(qd), bits(kd)))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_prefill_q_and_k_in_one_launch_against_oracle():
    cases = W.cases(W.PREFILL)
    aq, p = cases["rope_q"]()
    ak, _ = cases["rope_k"]()
    qd, kd = to_dev(aq["x"]), to_dev(ak["x"])
    gbe.gbe_rope_qk(qd, qd, kd, kd, to_dev(aq["pos"]), to_dev(aq["inv_freq"]), p["r"], p["mu"], p["layout"])
    o = oracle.get()
    for a, y, what in ((aq, qd, "q"), (ak, kd, "k")):
        x = widen(a["x"])
        want = o.rope(x, a["pos"], a["inv_freq"], p["r"], p["mu"], p["layout"])
        assert_rope_close(to_f32(y), want, x, p["r"], p["mu"], p["layout"], "bf16", f"prefill {what}")


def test_overlapping_outputs_are_refused():
    L = gbe.lib()
    s = torch.cuda.current_stream().cuda_stream
    T, H, D = 8, 2, 16
    buf = torch.zeros(T * 3 * H * D, dtype=torch.float32, device="cuda")
    pos = torch.zeros(T, dtype=torch.int32, device="cuda")
    om = torch.ones(D // 2, dtype=torch.float32, device="cuda")
    stride = 3 * H * D
    base = buf.data_ptr()
    # q_out overlapping k's columns
    st = L.gbe_rope_qk(base, base + 4 * D, stride, H, base + 4 * H * D, base + 4 * H * D, stride, H,
                       pos.data_ptr(), T, D, D, om.data_ptr(), None, 0, 1.0, 0, 0, s)
    assert st == 8
    # disjoint interleaved columns in one buffer are accepted
    st = L.gbe_rope_qk(base, base, stride, H, base + 4 * H * D, base + 4 * H * D, stride, H,
                       pos.data_ptr(), T, D, D, om.data_ptr(), None, 0, 1.0, 0, 0, s)
    assert st == 0
    # a token stride shorter than a row is refused
    st = L.gbe_rope_qk(base, base, H * D - 1, H, None, None, 0, 0, pos.data_ptr(), T, D, D, om.data_ptr(),
                       None, 0, 1.0, 0, 0, s)
    assert st == 2
    torch.cuda.synchronize()
