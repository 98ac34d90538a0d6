"""QK-norm then RoPE in one pass (gbe_qk_norm_rope) on the GPU, through the
C ABI: equal bit for bit to the unfused composition through the same
library (gbe_rmsnorm over head rows, then gbe_rope_qk), within tolerance of
the oracle's composition, correct on QKV slices, and the same bits on the
unaligned path and with the cos/sin table."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import assert_rope_close, bits, to_dev, to_f32, widen
from synth import normal, randint, to_bf16, uniform

pytestmark = pytest.mark.gpu


def _case(seed, T, Hq, Hk, D, r, dtype):
    q = normal(seed, f"qkn.q.{T}.{D}", (T, Hq, D), 0.0, 2.0)
    k = normal(seed, f"qkn.k.{T}.{D}", (T, Hk, D), 0.0, 2.0)
    gq = uniform(seed, f"qkn.gq.{D}", (D,), 0.5, 1.5)
    gk = uniform(seed, f"qkn.gk.{D}", (D,), 0.5, 1.5)
    if dtype == "bf16":
        q, k, gq, gk = to_bf16(q), to_bf16(k), to_bf16(gq), to_bf16(gk)
    pos = randint(seed, f"qkn.pos.{T}", (T,), 0, 1 << 16)
    om = (1e6 ** (-2.0 * np.arange(max(r // 2, 1)) / max(r, 2))).astype(np.float32)
    return q, k, gq, gk, pos, om


def _unfused(q, k, gq, gk, pos, om, r, mu, layout, eps=1e-6):
    T, Hq, D = q.shape
    Hk = k.shape[1]
    qn = gbe.rmsnorm(to_dev(q).view(T * Hq, D), to_dev(gq), eps).view(T, Hq, D)
    kn = gbe.rmsnorm(to_dev(k).view(T * Hk, D), to_dev(gk), eps).view(T, Hk, D)
    gbe.gbe_rope_qk(qn, qn, kn, kn, to_dev(pos), to_dev(om), r, mu, layout)
    return qn, kn


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("T,Hq,Hk,D,r", [(9, 32, 8, 128, 128), (5, 4, 2, 64, 32), (3, 3, 1, 16, 16),
                                         (4, 2, 2, 8, 8), (17, 16, 4, 96, 64),
                                         # more chunks of head rows than warps of a token's CTA
                                         (3, 160, 9, 128, 128), (2, 300, 20, 128, 128),
                                         # four-pass items of 4 lanes a row (f32 head_dim 32, bf16 64),
                                         # head counts ragged in 16-row items
                                         (7, 20, 5, 32, 32), (6, 33, 3, 64, 64),
                                         # wide heads: up to 64 chunks (256 f32 / 512 bf16)
                                         (2, 4, 2, 256, 256), (3, 5, 3, 128, 96), (3, 3, 2, 200, 160),
                                         (2, 2, 1, 512, 512), (2, 3, 2, 384, 320)])
@pytest.mark.parametrize("mu", [1.0, 1.1])
def test_equals_unfused_composition(dtype, layout, T, Hq, Hk, D, r, mu):
    q, k, gq, gk, pos, om = _case(1, T, Hq, Hk, D, r, dtype)
    if dtype == "f32" and D > 256:  # past 64 chunks: refused before anything runs
        qd = to_dev(q)
        with pytest.raises(gbe.GbeError) as e:
            gbe.gbe_qk_norm_rope(qd, qd, to_dev(gq), None, None, None, 1e-6, to_dev(pos), to_dev(om), r, mu, layout)
        assert e.value.status == 2
        return
    qn, kn = _unfused(q, k, gq, gk, pos, om, r, mu, layout)
    qd, kd = to_dev(q), to_dev(k)
    gbe.gbe_qk_norm_rope(qd, qd, to_dev(gq), kd, kd, to_dev(gk), 1e-6, to_dev(pos), to_dev(om), r, mu, layout)
    assert np.array_equal(bits(qd), bits(qn)), "q"
    assert np.array_equal(bits(kd), bits(kn)), "k"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_against_oracle(dtype, layout):
    T, Hq, Hk, D, r = 64, 32, 8, 128, 128
    q, k, gq, gk, pos, om = _case(2, T, Hq, Hk, D, r, dtype)
    qd, kd = to_dev(q), to_dev(k)
    qo, ko = torch.empty_like(qd), torch.empty_like(kd)
    gbe.gbe_qk_norm_rope(qd, qo, to_dev(gq), kd, ko, to_dev(gk), 1e-6, to_dev(pos), to_dev(om), r, 1.0, layout)
    o = oracle.get()
    for x, g, y, what in ((q, gq, qo, "q"), (k, gk, ko, "k")):
        xw, gw = widen(x), widen(g)
        want = o.qk_norm_rope(xw, gw, 1e-6, pos, om, r, 1.0, layout, n_bf16=(dtype == "bf16"))
        n = o.rmsnorm(xw.reshape(-1, D), gw, 1e-6).reshape(xw.shape)
        assert_rope_close(to_f32(y), want, n, r, 1.0, layout, dtype, what)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_wide_heads_against_oracle_slices_and_cache(dtype, layout):
    """Head rows of 33 to 64 chunks (f32 head_dim 256, bf16 512): against the
    oracle; on QKV slices with a token stride off the 16-byte grid (the
    scalar path) and with the cos/sin table, equal to the composition."""
    D = 256 if dtype == "f32" else 512
    T, Hq, Hk, r = 6, 4, 2, D
    q, k, gq, gk, pos, om = _case(4, T, Hq, Hk, D, r, dtype)
    qd, kd = to_dev(q), to_dev(k)
    qo, ko = torch.empty_like(qd), torch.empty_like(kd)
    gbe.gbe_qk_norm_rope(qd, qo, to_dev(gq), kd, ko, to_dev(gk), 1e-6, to_dev(pos), to_dev(om), r, 1.0, layout)
    o = oracle.get()
    for x, g, y, what in ((q, gq, qo, "q"), (k, gk, ko, "k")):
        xw, gw = widen(x), widen(g)
        want = o.qk_norm_rope(xw, gw, 1e-6, pos, om, r, 1.0, layout, n_bf16=(dtype == "bf16"))
        n = o.rmsnorm(xw.reshape(-1, D), gw, 1e-6).reshape(xw.shape)
        assert_rope_close(to_f32(y), want, n, r, 1.0, layout, dtype, what)
    qn, kn = _unfused(q, k, gq, gk, pos, om, r, 1.0, layout)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    for extra in (0, 1):
        stride = (Hq + Hk) * D + extra
        buf = torch.zeros(T * stride, dtype=tdt, device="cuda")
        buf.view(T, stride)[:, :Hq * D] = to_dev(q).view(T, Hq * D)
        buf.view(T, stride)[:, Hq * D:(Hq + Hk) * D] = to_dev(k).view(T, Hk * D)
        qv = buf.as_strided((T, Hq, D), (stride, D, 1))
        kv = buf.as_strided((T, Hk, D), (stride, D, 1), Hq * D)
        cache = gbe.rope_cos_sin(to_dev(om), r, 1 << 15) if extra == 0 else None
        gbe.gbe_qk_norm_rope(qv, qv, to_dev(gq), kv, kv, to_dev(gk), 1e-6, to_dev(pos), to_dev(om), r, 1.0, layout,
                             cos_sin=cache)
        assert np.array_equal(bits(qv.contiguous()), bits(qn)), extra
        assert np.array_equal(bits(kv.contiguous()), bits(kn)), extra


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_qkv_slices_cache_and_unaligned(dtype, layout):
    T, Hq, Hk, D, r = 33, 8, 2, 64, 64
    q, k, gq, gk, pos, om = _case(3, T, Hq, Hk, D, r, dtype)
    qn, kn = _unfused(q, k, gq, gk, pos, om, r, 1.0, layout)
    width = (Hq + 2 * Hk) * D
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    for extra in (0, 1):  # extra = 1: token stride not a multiple of 16 bytes -> scalar path
        stride = width + extra
        buf = torch.zeros(T * stride, dtype=tdt, device="cuda")
        rows = buf.view(T, stride)
        rows[:, :Hq * D] = to_dev(q).view(T, Hq * D)
        rows[:, Hq * D:(Hq + Hk) * D] = to_dev(k).view(T, Hk * D)
        rows[:, (Hq + Hk) * D:width] = 7.0
        qv = buf.as_strided((T, Hq, D), (stride, D, 1))
        kv = buf.as_strided((T, Hk, D), (stride, D, 1), Hq * D)
        cache = gbe.rope_cos_sin(to_dev(om), r, 1 << 15) if extra == 0 else None  # some positions past it
        gbe.gbe_qk_norm_rope(qv, qv, to_dev(gq), kv, kv, to_dev(gk), 1e-6, to_dev(pos), to_dev(om), r, 1.0, layout,
                             cos_sin=cache)
        assert np.array_equal(bits(qv.contiguous()), bits(qn)), extra
        assert np.array_equal(bits(kv.contiguous()), bits(kn)), extra
        assert torch.all(rows[:, (Hq + Hk) * D:width] == 7.0), "v untouched"


def test_head_dim_limit():
    L = gbe.lib()
    s = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(2 * 4 * 512, device="cuda")
    g = torch.ones(512, device="cuda")
    pos = torch.zeros(2, dtype=torch.int32, device="cuda")
    om = torch.ones(256, device="cuda")
    st = L.gbe_qk_norm_rope(x.data_ptr(), x.data_ptr(), 4 * 512, 4, g.data_ptr(), None, None, 0, 0, None, 1e-6,
                            pos.data_ptr(), 2, 512, 512, om.data_ptr(), None, 0, 1.0, 0, 0, s)
    assert st == 2  # 512 f32 entries = 128 chunks > 64


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hk,D,mu,cached,extra", [(32, 8, 128, 1.0, False, 0), (12, 3, 64, 1.1, True, 0),
                                                     (8, 2, 128, 1.0, True, 8)])
def test_many_tokens_equal_unfused_composition(dtype, Hq, Hk, D, mu, cached, extra):
    """Many tokens (20011) in the half-layout, whole-head case: equal bit for
    bit to the composition, with ragged head counts, mu != 1, the cos/sin
    table and q, k as slices of one buffer (a token stride past the heads)."""
    T, r = 20011, D
    q, k, gq, gk, pos, om = _case(5, T, Hq, Hk, D, r, dtype)
    qn, kn = _unfused(q, k, gq, gk, pos, om, r, mu, 0)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    stride = (Hq + Hk) * D + extra
    buf = torch.full((T * stride,), 7.0, dtype=tdt, device="cuda")
    rows = buf.view(T, stride)
    rows[:, :Hq * D] = to_dev(q).view(T, Hq * D)
    rows[:, Hq * D:(Hq + Hk) * D] = to_dev(k).view(T, Hk * D)
    qv = buf.as_strided((T, Hq, D), (stride, D, 1))
    kv = buf.as_strided((T, Hk, D), (stride, D, 1), Hq * D)
    cache = gbe.rope_cos_sin(to_dev(om), r, 1 << 15) if cached else None  # some positions past it
    gbe.gbe_qk_norm_rope(qv, qv, to_dev(gq), kv, kv, to_dev(gk), 1e-6, to_dev(pos), to_dev(om), r, mu, 0,
                         cos_sin=cache)
    assert np.array_equal(bits(qv.contiguous()), bits(qn)), "q"
    assert np.array_equal(bits(kv.contiguous()), bits(kn)), "k"
    assert torch.all(rows[:, (Hq + Hk) * D:] == 7.0), "past the heads untouched"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_special_values_equal_unfused_composition(dtype):
    """Head rows of zeros (1/rms = 1/sqrt(eps)), with an infinity, with a NaN,
    and of values near the top of the range, in the whole-head half layout
    (four-pass items) and at a partial r: the fused call gives the
    composition's bits."""
    for T, Hq, Hk, D, r in ((9, 32, 8, 128, 128), (5, 8, 2, 64, 32)):
        q, k, gq, gk, pos, om = _case(6, T, Hq, Hk, D, r, dtype)
        q, k = widen(q).copy(), widen(k).copy()
        q[0, 3] = 0.0
        q[1, 5, 7] = np.inf
        k[2, 1, 0] = np.nan
        q[3, 0] = 1.0e30
        k[4, 0] = -2.0e-30
        if dtype == "bf16":
            q, k = to_bf16(q), to_bf16(k)
        else:
            q, k = q.astype(np.float32), k.astype(np.float32)
        for eps in (1e-6, 0.0):  # eps = 0: the zero head's 1/rms is infinite, its output NaN
            qn, kn = _unfused(q, k, gq, gk, pos, om, r, 1.0, 0, eps=eps)
            qd, kd = to_dev(q), to_dev(k)
            gbe.gbe_qk_norm_rope(qd, qd, to_dev(gq), kd, kd, to_dev(gk), eps, to_dev(pos), to_dev(om), r, 1.0, 0)
            assert np.array_equal(bits(qd), bits(qn)), (T, D, r, eps, "q")
            assert np.array_equal(bits(kd), bits(kn)), (T, D, r, eps, "k")

