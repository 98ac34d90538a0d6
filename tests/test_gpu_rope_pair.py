"""gbe_rope_pair on the GPU: two RoPE operands in one launch, each with its
own rotated width, frequencies, scale and layout ("Elementwise kernels in C",
sections 2.2 and 4; "Operations", section 3).  Each operand's result must
equal gbe_rope of that operand alone, bit for bit, and the oracle within the
RoPE bar; the refusals of the per-operand checks."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import assert_rope_close, bits, to_dev, to_f32, widen
from synth import normal, randint, to_bf16
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _freqs(r, base):
    return (base ** (-2.0 * np.arange(r // 2) / max(r, 1))).astype(np.float32)


def _x(dtype, tag, shape):
    x = normal(71, f"t.pair.{tag}", shape, 0.0, 1.0)
    return to_bf16(x) if dtype == "bf16" else x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("la,lb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("T,D,Ha,Hb,ra,rb", [(37, 128, 32, 8, 64, 128), (5, 64, 3, 2, 64, 32), (64, 128, 4, 4, 0, 96),
                                             (300, 96, 2, 1, 48, 96)])
@pytest.mark.parametrize("in_place", [False, True])
def test_equals_two_single_calls(dtype, la, lb, T, D, Ha, Hb, ra, rb, in_place):
    xa, xb = _x(dtype, f"a{T}.{D}", (T, Ha, D)), _x(dtype, f"b{T}.{D}", (T, Hb, D))
    pos = to_dev(randint(71, f"t.pair.pos{T}", (T,), 0, 1 << 20).astype(np.int32))
    fa, fb = to_dev(_freqs(ra, 10000.0)), to_dev(_freqs(rb, 500000.0))
    a, b = to_dev(xa), to_dev(xb)
    ya, yb = (a.clone(), b.clone()) if in_place else (torch.empty_like(a), torch.empty_like(b))
    ia = ya if in_place else a
    ib = yb if in_place else b
    gbe.gbe_rope_pair((ia, ya, fa, ra, 1.0, la), (ib, yb, fb, rb, 1.2, lb), pos)
    ref_a, ref_b = torch.empty_like(a), torch.empty_like(b)
    gbe.gbe_rope(a, ref_a, pos, fa, ra, 1.0, la)
    gbe.gbe_rope(b, ref_b, pos, fb, rb, 1.2, lb)
    assert np.array_equal(bits(ya), bits(ref_a)), "first operand"
    assert np.array_equal(bits(yb), bits(ref_b)), "second operand"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_slices_of_one_qkv_buffer_and_the_scalar_path(dtype):
    """q and k as column slices of a fused QKV buffer (token stride > H * D),
    in place, mixed layouts; and the same with a token stride that leaves
    rows off the 16-byte grid (the scalar path) -- the same bits."""
    T, Hq, Hk, D = 33, 4, 2, 64
    for pad in (0, 1):
        Wd = (Hq + 2 * Hk) * D + pad
        qkv = to_dev(_x(dtype, f"qkv{pad}", (T, Wd)))
        ref = qkv.clone()
        pos = to_dev(randint(71, "t.pair.qkvpos", (T,), 0, 4096).astype(np.int32))
        fq, fk = to_dev(_freqs(32, 10000.0)), to_dev(_freqs(64, 10000.0))
        q = qkv[:, :Hq * D].view(T, Hq, D) if pad == 0 else qkv[:, :Hq * D].unflatten(1, (Hq, D))
        k = qkv[:, Hq * D:(Hq + Hk) * D].unflatten(1, (Hk, D))
        gbe.gbe_rope_pair((q, q, fq, 32, 1.0, 1), (k, k, fk, 64, 0.9, 0), pos)
        rq = ref[:, :Hq * D].unflatten(1, (Hq, D)).contiguous()
        rk = ref[:, Hq * D:(Hq + Hk) * D].unflatten(1, (Hk, D)).contiguous()
        oq, ok = torch.empty_like(rq), torch.empty_like(rk)
        gbe.gbe_rope(rq, oq, pos, fq, 32, 1.0, 1)
        gbe.gbe_rope(rk, ok, pos, fk, 64, 0.9, 0)
        assert np.array_equal(bits(q.contiguous()), bits(oq)), pad
        assert np.array_equal(bits(k.contiguous()), bits(ok)), pad
        assert torch.equal(qkv[:, (Hq + Hk) * D:], ref[:, (Hq + Hk) * D:]), "v untouched"


def test_rope_variants_workload_in_one_launch():
    """The f32 RoPE-variants workload at full size: q [4096, 32, 128]
    interleaved r = 64 and k [4096, 8, 128] half r = 128 mu = 1.2, in place,
    in one launch: each equals its single call bit for bit, the pass-through
    entries are untouched, and 64 tokens match the oracle."""
    cases = W.cases(W.ROPE_VARIANTS)
    (aq, pq), (ak, pk) = cases["rope_q"](), cases["rope_k"]()
    q, k = to_dev(aq["x"]), to_dev(ak["x"])
    pos = to_dev(aq["pos"])
    fq, fk = to_dev(aq["inv_freq"]), to_dev(ak["inv_freq"])
    q1, k1 = q.clone(), k.clone()
    gbe.gbe_rope_pair((q, q, fq, pq["r"], pq["mu"], pq["layout"]), (k, k, fk, pk["r"], pk["mu"], pk["layout"]), pos)
    gbe.gbe_rope(q1, q1, pos, fq, pq["r"], pq["mu"], pq["layout"])
    gbe.gbe_rope(k1, k1, pos, fk, pk["r"], pk["mu"], pk["layout"])
    assert torch.equal(q.view(torch.int32), q1.view(torch.int32))
    assert torch.equal(k.view(torch.int32), k1.view(torch.int32))
    assert np.array_equal(bits(q)[..., pq["r"]:], aq["x"][..., pq["r"]:].view(np.uint32))
    o = oracle.get()
    sel = np.arange(0, 4096, 64)
    for got, a, p in ((q, aq, pq), (k, ak, pk)):
        want = o.rope(a["x"][sel], a["pos"][sel], a["inv_freq"], p["r"], p["mu"], p["layout"])
        assert_rope_close(to_f32(got)[sel], want, a["x"][sel], p["r"], p["mu"], p["layout"], "f32")


def test_refusals():
    L = gbe.lib()
    s = torch.cuda.current_stream().cuda_stream
    x = torch.ones(4, 2, 16, device="cuda")
    pos = torch.zeros(4, dtype=torch.int32, device="cuda")
    f = torch.ones(8, device="cuda")
    op = lambda **kw: gbe.binding.RopeOperand(**{**dict(x=x.data_ptr(), y=x.data_ptr(), stride=32, H=2, r=16,
                                                        inv_freq=f.data_ptr(), mu=1.0, layout=0), **kw})
    import ctypes
    call = lambda a, b: L.gbe_rope_pair(ctypes.cast(ctypes.byref(a), ctypes.c_void_p) if a is not None else None,
                                        ctypes.cast(ctypes.byref(b), ctypes.c_void_p) if b is not None else None,
                                        pos.data_ptr(), 4, 16, 0, s)
    assert call(None, op()) == 1
    assert call(op(), op(layout=2)) == 4
    assert call(op(), op(r=15)) == 6 and call(op(r=18), None) == 6 and call(op(), op(mu=float("nan"))) == 6
    assert call(op(), op(stride=31)) == 2
    y = torch.empty_like(x)
    assert call(op(), op(y=y.data_ptr())) == 8              # two outputs in one buffer
    assert call(op(y=y.data_ptr()), None) == 0
    assert call(op(y=pos.data_ptr(), x=y.data_ptr()), None) == 8  # an output over the positions
    torch.cuda.synchronize()
