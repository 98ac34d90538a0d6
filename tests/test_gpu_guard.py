"""Guard regions around every output, through the C ABI.

Each output of each entry point is placed inside a larger device buffer
whose 256 bytes before and after it (and, for q/k slices of a fused QKV
buffer, the v columns between the rows) hold a sentinel pattern.  The calls
run at ragged shapes -- widths that are not a multiple of the 16-byte vector,
odd counts, r < D, strided token rows, rows not a multiple of a CTA's rows --
and on both the aligned (vector) and the off-grid (scalar) path.  After each
call the sentinels must be untouched and the output must still match the
oracle.  This is the stand-in for an address sanitizer: torch's caching
allocator pads allocations, so a kernel writing one vector past a tensor
would otherwise go unnoticed."""
import math

import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import assert_rel, assert_rope_close, bits, to_dev, to_f32, widen
from synth import normal, randint, to_bf16, uniform

pytestmark = pytest.mark.gpu

PAD = 256
SENT = 0xA5
TD = {"f32": torch.float32, "bf16": torch.bfloat16}
ES = {"f32": 4, "bf16": 2}


class Guarded:
    """An output of `shape` and `dtype` inside a device buffer with PAD
    sentinel bytes before and after it; `shift` extra bytes before it put it
    off the 16-byte grid (the scalar path)."""

    def __init__(self, shape, dtype, shift=0):
        es = torch.empty((), dtype=dtype).element_size()
        self.nbytes = math.prod(shape) * es
        self.lo = PAD + shift
        self.raw = torch.full((self.lo + self.nbytes + PAD,), SENT, dtype=torch.uint8, device="cuda")
        self.t = self.raw[self.lo:self.lo + self.nbytes].view(dtype).view(shape)

    def assert_intact(self, what):
        torch.cuda.synchronize()
        r = self.raw.cpu().numpy()
        before, after = r[:self.lo], r[self.lo + self.nbytes:]
        assert (before == SENT).all(), f"{what}: {int((before != SENT).sum())} bytes written before the output"
        assert (after == SENT).all(), f"{what}: {int((after != SENT).sum())} bytes written after the output"


def _gen(dtype, tag, shape, std=1.0):
    x = normal(61, f"t.guard.{tag}", shape, 0.0, std)
    return to_bf16(x) if dtype == "bf16" else x


def _shifts(dtype):
    return (0, ES[dtype])


def _placed(a: np.ndarray, dtype, shift):
    """An input array placed at the same offset from the 16-byte grid as the
    outputs of the call (so the call takes the path the shift selects)."""
    g = Guarded(a.shape, TD[dtype], shift)
    g.t.copy_(to_dev(a))
    return g.t


@pytest.mark.parametrize("dtype,rows,d", [("bf16", 7, 1000), ("bf16", 5, 4104), ("f32", 3, 33),
                                          ("f32", 2, 16388), ("bf16", 9, 8)])
def test_rmsnorm_add_rmsnorm_layernorm(dtype, rows, d):
    o = oracle.get()
    x, r = _gen(dtype, f"x{d}", (rows, d)), _gen(dtype, f"r{d}", (rows, d))
    w = uniform(61, f"t.guard.w{d}", (d,), 0.5, 1.5)
    b = normal(61, f"t.guard.b{d}", (d,), 0.0, 0.3)
    if dtype == "bf16":
        w, b = to_bf16(w), to_bf16(b)
    for shift in _shifts(dtype):
        xd, rd, wd, bd = (_placed(a, dtype, shift) for a in (x, r, w, b))
        y = Guarded((rows, d), TD[dtype], shift)
        gbe.gbe_rmsnorm(xd, wd, y.t, 1e-5)
        y.assert_intact(f"rmsnorm {dtype} [{rows},{d}] shift {shift}")
        assert_rel(to_f32(y.t), o.rmsnorm(widen(x), widen(w), 1e-5), dtype, "rmsnorm")
        y, h = Guarded((rows, d), TD[dtype], shift), Guarded((rows, d), TD[dtype], shift)
        gbe.gbe_add_rmsnorm(xd, rd, wd, y.t, h.t, 1e-5)
        y.assert_intact("add_rmsnorm y")
        h.assert_intact("add_rmsnorm h")
        yo, ho = o.add_rmsnorm(widen(x), widen(r), widen(w), 1e-5, h_bf16=dtype == "bf16")
        want_h = o.bf16_round(ho) if dtype == "bf16" else ho.view(np.uint32)
        assert np.array_equal(bits(h.t), want_h)
        assert_rel(to_f32(y.t), yo, dtype, "add_rmsnorm y")
        y = Guarded((rows, d), TD[dtype], shift)
        gbe.gbe_layernorm(xd, wd, bd, y.t, 1e-5)
        y.assert_intact("layernorm")
        want = o.layernorm(widen(x), widen(w), widen(b), 1e-5)
        scale = np.abs(want - widen(b)).max(axis=1, keepdims=True) + np.abs(widen(b))
        assert np.all(np.abs(to_f32(y.t) - want) <= {"f32": 1e-5, "bf16": 1e-2}[dtype] * scale + 1e-30)


def _freqs(r, base=10000.0):
    return (base ** (-2.0 * np.arange(r // 2) / max(r, 1))).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", [0, 1])
def test_rope_and_rope_multi(dtype, layout):
    o = oracle.get()
    T, H, D, r = 5, 3, 72, 40
    x = _gen(dtype, f"rope{layout}", (T, H, D))
    pos = randint(61, "t.guard.pos", (T,), 0, 5000).astype(np.int32)
    om = _freqs(r)
    for shift in _shifts(dtype):
        xd = _placed(x, dtype, shift)
        y = Guarded((T, H, D), TD[dtype], shift)
        gbe.gbe_rope(xd, y.t, to_dev(pos), to_dev(om), r, 1.2, layout)
        y.assert_intact(f"rope {dtype} layout {layout} shift {shift}")
        want = o.rope(widen(x), pos, om, r, 1.2, layout)
        got = to_f32(y.t)
        assert_rope_close(got, want, widen(x), r, 1.2, layout, dtype, "rope")
        assert np.array_equal(bits(y.t)[..., r:], x[..., r:].view(bits(y.t).dtype))
        dims = (16, 24)
        pm = randint(61, "t.guard.pm", (T, 2), 0, 300).astype(np.int32)
        fm = np.concatenate([_freqs(dd) for dd in dims])
        y = Guarded((T, H, D), TD[dtype], shift)
        gbe.gbe_rope_multi(xd, y.t, to_dev(pm), dims, to_dev(fm), 1.0, layout)
        y.assert_intact("rope_multi")
        want = o.rope_multi(widen(x), pm, dims, fm, 1.0, layout)
        assert np.all(np.abs(to_f32(y.t) - want) <= {"f32": 2e-5, "bf16": 2e-2}[dtype] * (np.abs(widen(x)).max() + 1))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rope_qk_and_qk_norm_rope_in_a_guarded_qkv_buffer(dtype):
    """q and k outputs are column slices of a fused QKV output buffer whose v
    columns hold the sentinel too: strided writes must leave them alone."""
    o = oracle.get()
    T, Hq, Hk, D, r = 7, 4, 2, 64, 48
    W = (Hq + 2 * Hk) * D
    qkv = _gen(dtype, "qkv", (T, W))
    pos = randint(61, "t.guard.qkpos", (T,), 0, 9000).astype(np.int32)
    om = _freqs(r)
    gq = uniform(61, "t.guard.gq", (D,), 0.5, 1.5)
    gk = uniform(61, "t.guard.gk", (D,), 0.5, 1.5)
    if dtype == "bf16":
        gq, gk = to_bf16(gq), to_bf16(gk)
    src = to_dev(qkv)
    q_in = src[:, :Hq * D].view(T, Hq, D)
    k_in = src[:, Hq * D:(Hq + Hk) * D].view(T, Hk, D)
    for fused in (False, True):
        out = Guarded((T, W), TD[dtype])
        q_out = out.t[:, :Hq * D].view(T, Hq, D)
        k_out = out.t[:, Hq * D:(Hq + Hk) * D].view(T, Hk, D)
        if fused:
            gbe.gbe_qk_norm_rope(q_in, q_out, to_dev(gq), k_in, k_out, to_dev(gk), 1e-6, to_dev(pos), to_dev(om),
                                 r, 1.0, 1)
        else:
            gbe.gbe_rope_qk(q_in, q_out, k_in, k_out, to_dev(pos), to_dev(om), r, 1.0, 0)
        out.assert_intact(f"qkv fused={fused}")
        ob = out.raw[out.lo:out.lo + out.nbytes].cpu().numpy().reshape(T, W * ES[dtype])
        assert (ob[:, (Hq + Hk) * D * ES[dtype]:] == SENT).all(), "the v columns were written"
        x32 = widen(qkv)
        qx, kx = x32[:, :Hq * D].reshape(T, Hq, D), x32[:, Hq * D:(Hq + Hk) * D].reshape(T, Hk, D)
        if fused:
            wq = o.qk_norm_rope(qx, widen(gq), 1e-6, pos, om, r, 1.0, 1, n_bf16=dtype == "bf16")
            wk = o.qk_norm_rope(kx, widen(gk), 1e-6, pos, om, r, 1.0, 1, n_bf16=dtype == "bf16")
            tol = {"f32": 1e-5, "bf16": 1e-2}[dtype]
            for got, want in ((to_f32(q_out), wq), (to_f32(k_out), wk)):
                assert np.all(np.abs(got - want) <= tol * (np.abs(want).max() + 1))
        else:
            assert_rope_close(to_f32(q_out), o.rope(qx, pos, om, r, 1.0, 0), qx, r, 1.0, 0, dtype, "q")
            assert_rope_close(to_f32(k_out), o.rope(kx, pos, om, r, 1.0, 0), kx, r, 1.0, 0, dtype, "k")


def test_rope_cos_sin_table():
    o = oracle.get()
    r, L = 40, 37
    om = _freqs(r)
    tab = Guarded((L, r // 2, 2), torch.float32)
    gbe.gbe_rope_cos_sin(tab.t, to_dev(om), r)
    tab.assert_intact("cos/sin table")
    assert np.all(np.abs(to_f32(tab.t) - o.rope_cos_sin(om, r, L)) <= 4e-7)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 7, 1001, 4096 * 4 + 5])
def test_silu_mul_and_add(dtype, n):
    o = oracle.get()
    g, u = _gen(dtype, f"g{n}", (n,), 3.0), _gen(dtype, f"u{n}", (n,))
    for shift in _shifts(dtype):
        gd, ud = _placed(g, dtype, shift), _placed(u, dtype, shift)
        y = Guarded((n,), TD[dtype], shift)
        gbe.gbe_silu_mul(gd, ud, y.t)
        y.assert_intact(f"silu_mul {dtype} n={n} shift {shift}")
        assert_rel(to_f32(y.t), o.silu_mul(widen(g), widen(u)), dtype, "silu_mul")
        y = Guarded((n,), TD[dtype], shift)
        gbe.gbe_add(gd, ud, y.t)
        y.assert_intact("add")
        s = o.add(widen(g), widen(u))
        assert np.array_equal(bits(y.t), o.bf16_round(s) if dtype == "bf16" else s.view(np.uint32))


@pytest.mark.parametrize("dtype,d", [("bf16", 1000), ("bf16", 4096), ("f32", 33), ("f32", 512)])
def test_embedding(dtype, d):
    o = oracle.get()
    V, n = 300, 9
    table = _gen(dtype, f"tab{d}", (V, d))
    ids = randint(61, f"t.guard.ids{d}", (n,), 0, V).astype(np.int32)
    ids[4] = V + 3  # a bad id: a zero row and one count
    for shift in _shifts(dtype):
        td = _placed(table, dtype, shift)
        out = Guarded((n, d), TD[dtype], shift)
        cnt = Guarded((1,), torch.int32)
        cnt.t.zero_()
        gbe.gbe_embedding(td, to_dev(ids), out.t, cnt.t)
        out.assert_intact(f"embedding {dtype} d={d} shift {shift}")
        cnt.assert_intact("embedding counter")
        assert int(cnt.t.item()) == 1
        good = np.delete(np.arange(n), 4)
        want = o.embedding(widen(table), ids[good])
        got = to_f32(out.t)
        assert np.array_equal(got[good].view(np.uint32), want.view(np.uint32))
        assert np.all(got[4] == 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_sample_and_uniforms(dtype):
    """argmax against the oracle; the sampling outputs (whose parity with the
    oracle the sampling tests hold) against the same calls into plain
    buffers, bit for bit; the uniforms against the oracle's stream."""
    o = oracle.get()
    rows, n = 13, 1003
    x = _gen(dtype, "am", (rows, n), 3.0)
    for shift in _shifts(dtype):
        xd = _placed(x, dtype, shift)
        out = Guarded((rows,), torch.int32)
        gbe.gbe_argmax(xd, out.t)
        out.assert_intact(f"argmax {dtype} shift {shift}")
        assert np.array_equal(out.t.cpu().numpy(), o.argmax(widen(x)))
        u = torch.from_numpy(o.pcg64_uniforms(1, 0, rows)).cuda()
        for method, kw in (("temperature", dict(temperature=0.8)), ("top_k", dict(temperature=1.0, top_k=20)),
                           ("top_p", dict(temperature=1.0, p=0.9)), ("min_p", dict(temperature=1.0, p=0.1))):
            out = Guarded((rows,), torch.int32)
            gbe.gbe_sample(xd, u, out.t, method, **kw)
            out.assert_intact(f"sample {method}")
            assert torch.equal(out.t, gbe.sample(xd, u, method, **kw))
            out = Guarded((rows,), torch.int32)
            gbe.gbe_sample_seeded(xd, out.t, method, 1, 0, **kw)
            out.assert_intact(f"sample_seeded {method}")
            assert torch.equal(out.t, gbe.sample(xd, u, method, **kw))
    for n_u in (1, 31, 77):
        uu = Guarded((n_u,), torch.float32)
        gbe.gbe_pcg64_uniforms(uu.t, 9, 5)
        uu.assert_intact(f"uniforms n={n_u}")
        assert np.array_equal(uu.t.cpu().numpy().view(np.uint32), o.pcg64_uniforms(9, 5, n_u).view(np.uint32))
