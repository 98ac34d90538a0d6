"""RMSNorm and fused add+RMSNorm on the GPU against the oracle, through the
C ABI: small shapes spanning several tiles and ragged widths, both storage
types, the aligned and unaligned paths, in-place calls, the full-size
workloads, and batch invariance (a row's bits do not depend on the batch)."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import assert_bf16_within_ulp, assert_rel, bits, to_dev, to_f32, widen
from synth import normal, to_bf16, uniform
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(rows, d, dtype, seed=11):
    x = normal(seed, f"t.rms.x.{rows}.{d}", (rows, d), 0.0, 1.0)
    w = uniform(seed, f"t.rms.w.{d}", (d,), 0.5, 1.5)
    if dtype == "bf16":
        return to_bf16(x), to_bf16(w)
    return x, w


def _check_rms(x, w, eps, y_dev, dtype, what):
    want = oracle.get().rmsnorm(widen(x), widen(w), eps)
    assert_rel(to_f32(y_dev), want, dtype, what)
    if dtype == "bf16":
        assert_bf16_within_ulp(bits(y_dev), want, what)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [1, 3, 8, 33, 64, 100, 128, 1000, 4096, 4100, 5000, 16384, 20000, 40000])
def test_rmsnorm_shapes(dtype, d):
    rows = 37 if d <= 5000 else 5
    x, w = _inputs(rows, d, dtype)
    y = gbe.rmsnorm(to_dev(x), to_dev(w), 1e-5)
    _check_rms(x, w, 1e-5, y, dtype, f"rmsnorm {dtype} d={d}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 4096, 12000, 16384, 30000])
def test_rmsnorm_unaligned_path_same_bits(dtype, d):
    """An element-offset view takes the scalar path; its bits equal the vector path's."""
    x, w = _inputs(9, d, dtype)
    xd, wd = to_dev(x), to_dev(w)
    y_vec = gbe.rmsnorm(xd, wd, 1e-5)
    buf = torch.empty(9 * d + 1, dtype=xd.dtype, device="cuda")
    xs = buf[1:].view(9, d)
    xs.copy_(xd)
    out = torch.empty(9 * d + 1, dtype=xd.dtype, device="cuda")[1:].view(9, d)
    gbe.gbe_rmsnorm(xs, wd, out, 1e-5)
    assert np.array_equal(bits(out), bits(y_vec))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rmsnorm_in_place_and_zero_rows(dtype):
    x, w = _inputs(20, 256, dtype)
    x[4] = 0
    xd = to_dev(x)
    y_ref = gbe.rmsnorm(xd, to_dev(w), 1e-5)
    gbe.gbe_rmsnorm(xd, to_dev(w), xd, 1e-5)
    assert np.array_equal(bits(xd), bits(y_ref))
    got = to_f32(y_ref)
    assert np.all(got[4] == 0) and not np.isnan(got).any()


def test_rmsnorm_tiny_workload():
    a, p = W.cases(W.TINY)["rmsnorm"]()
    y = gbe.rmsnorm(to_dev(a["x"]), to_dev(a["w"]), p["eps"])
    _check_rms(a["x"], a["w"], p["eps"], y, "f32", "tiny rmsnorm")
    assert np.all(to_f32(y)[3] == 0)


def test_rmsnorm_wide_f32_workload_full():
    a, p = W.cases(W.WIDE)["rmsnorm"]()
    y = gbe.rmsnorm(to_dev(a["x"]), to_dev(a["w"]), p["eps"])
    _check_rms(a["x"], a["w"], p["eps"], y, "f32", "rmsnorm [1024,16384] f32")


def test_rmsnorm_prefill_bf16_workload_full():
    a, p = W.cases(W.PREFILL)["rmsnorm"]()
    y = gbe.rmsnorm(to_dev(a["x"]), to_dev(a["w"]), p["eps"])
    _check_rms(a["x"], a["w"], p["eps"], y, "bf16", "rmsnorm [8192,4096] bf16")


@pytest.mark.parametrize("workload", [W.DECODE, W.PREFILL])
def test_add_rmsnorm_workload_full(workload):
    a, p = W.cases(workload)["add_rmsnorm"]()
    xd, rd, wd = to_dev(a["x"]), to_dev(a["residual"]), to_dev(a["w"])
    y, h = gbe.add_rmsnorm(xd, rd, wd, p["eps"])
    o = oracle.get()
    yo, ho = o.add_rmsnorm(widen(a["x"]), widen(a["residual"]), widen(a["w"]), p["eps"], h_bf16=True)
    assert np.array_equal(bits(h), o.bf16_round(ho)), "h must be the rounded sum, bit for bit"
    assert_rel(to_f32(y), yo, "bf16", f"add_rmsnorm y {workload}")
    assert_bf16_within_ulp(bits(y), yo, "add_rmsnorm y")
    # the fused call equals the unfused composition through the same library, bit for bit
    h2 = gbe.add(xd, rd)
    y2 = gbe.rmsnorm(h2, wd, p["eps"])
    assert np.array_equal(bits(h2), bits(h)) and np.array_equal(bits(y2), bits(y))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [5, 64, 1000, 4096, 12000, 16384, 20000, 30000])
def test_add_rmsnorm_shapes_and_aliases(dtype, d):
    x, w = _inputs(13, d, dtype, seed=3)
    r, _ = _inputs(13, d, dtype, seed=4)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    y, h = gbe.add_rmsnorm(xd, rd, wd, 1e-5)
    o = oracle.get()
    yo, ho = o.add_rmsnorm(widen(x), widen(r), widen(w), 1e-5, h_bf16=(dtype == "bf16"))
    if dtype == "bf16":
        assert np.array_equal(bits(h), o.bf16_round(ho))
    else:
        assert np.array_equal(bits(h), ho.view(np.uint32))
    assert_rel(to_f32(y), yo, dtype, f"add_rmsnorm {dtype} d={d}")
    # h == residual and y == x in place
    gbe.gbe_add_rmsnorm(xd, rd, wd, xd, rd, 1e-5)
    assert np.array_equal(bits(rd), bits(h)) and np.array_equal(bits(xd), bits(y))


def _invariance(fn_full, fn_part, rows, what):
    ref = fn_full()
    for b in range(1, rows + 1):
        part = fn_part(b)
        if not torch.equal(part.view(torch.int16 if part.dtype == torch.bfloat16 else torch.int32),
                           ref[:b].view(torch.int16 if ref.dtype == torch.bfloat16 else torch.int32)):
            raise AssertionError(f"{what}: batch of {b} rows differs from the full batch")


def test_batch_invariance_wide_f32():
    """[1024, 16384] f32: the first b rows alone give the same bits, b = 1..1024."""
    a, p = W.cases(W.WIDE)["rmsnorm"]()
    xd, wd = to_dev(a["x"]), to_dev(a["w"])
    out = torch.empty_like(xd)
    _invariance(lambda: gbe.rmsnorm(xd, wd, p["eps"]),
                lambda b: (gbe.gbe_rmsnorm(xd[:b], wd, out[:b], p["eps"]), out[:b])[1], 1024,
                "rmsnorm f32 d=16384")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_wide_rows_batch_invariant(dtype):
    """Wide rows (f32: 1024 threads a row, bf16: 512) give the same bits in
    any batch, for RMSNorm and the fused add (both outputs)."""
    rows, d = 200, 16384
    x, w = _inputs(rows, d, dtype, seed=13)
    r, _ = _inputs(rows, d, dtype, seed=14)
    xd, wd, rd = to_dev(x), to_dev(w), to_dev(r)
    ref = gbe.rmsnorm(xd, wd, 1e-5)
    yf, hf = gbe.add_rmsnorm(xd, rd, wd, 1e-5)
    _check_rms(x[:3], w, 1e-5, ref[:3], dtype, f"rmsnorm {dtype} wide")
    iv = torch.int32 if dtype == "f32" else torch.int16
    for b in (1, 5, 40, 76, 77, 150, 152, 153, 200):
        y = gbe.rmsnorm(xd[:b].contiguous(), wd, 1e-5)
        assert torch.equal(y.view(iv), ref[:b].view(iv)), b
        ya, ha = gbe.add_rmsnorm(xd[:b].contiguous(), rd[:b].contiguous(), wd, 1e-5)
        assert torch.equal(ya.view(iv), yf[:b].view(iv)), ("add y", b)
        assert torch.equal(ha.view(iv), hf[:b].view(iv)), ("add h", b)


@pytest.mark.parametrize("dtype,d", [("f32", 16384), ("f32", 16000), ("bf16", 32768), ("bf16", 31000)])
def test_rows_of_1024_threads_many_rows(dtype, d):
    """Rows of 1024 threads in a batch of more rows than two per SM (700):
    the whole batch and slices of it small enough to take the kernel that
    keeps rows in registers give the same bits; some rows match the oracle."""
    rows = 700
    x, w = _inputs(rows, d, dtype, seed=17)
    xd, wd = to_dev(x), to_dev(w)
    ref = gbe.rmsnorm(xd, wd, 1e-5)
    iv = torch.int32 if dtype == "f32" else torch.int16
    for r0, r1 in ((0, 100), (299, 400), (600, 700), (699, 700)):
        y = gbe.rmsnorm(xd[r0:r1].contiguous(), wd, 1e-5)
        assert torch.equal(y.view(iv), ref[r0:r1].view(iv)), (r0, r1)
    pick = [0, 151, 152, 350, 699]
    _check_rms(x[pick], w, 1e-5, ref[pick], dtype, f"rmsnorm {dtype} d={d} many rows")
    y2 = xd.clone()
    gbe.gbe_rmsnorm(y2, wd, y2, 1e-5)  # in place
    assert torch.equal(y2.view(iv), ref.view(iv)), "in place"
    # rows of zeros, with an infinity, with a NaN and of huge values: the same
    # bits in the large batch as alone
    x2 = widen(x).copy()
    x2[3] = 0.0
    x2[310, 17] = np.inf
    x2[460, 5] = np.nan
    x2[611] = 3.0e38
    x2 = to_bf16(x2) if dtype == "bf16" else x2.astype(np.float32)
    xd2 = to_dev(x2)
    ref2 = gbe.rmsnorm(xd2, wd, 1e-5)
    for r in (3, 310, 460, 611):
        y = gbe.rmsnorm(xd2[r:r + 1].contiguous(), wd, 1e-5)
        assert torch.equal(y.view(iv), ref2[r:r + 1].view(iv)), r
    assert torch.all(ref2[3] == 0), "a zero row stays zero"


def test_batch_invariance_prefill_bf16():
    """[8192, 4096] bf16: batches b = 1..4096 and rows placed at other offsets."""
    a, p = W.cases(W.PREFILL)["add_rmsnorm"]()
    xd, rd, wd = to_dev(a["x"]), to_dev(a["residual"]), to_dev(a["w"])
    out = torch.empty_like(xd)
    _invariance(lambda: gbe.rmsnorm(xd, wd, p["eps"]),
                lambda b: (gbe.gbe_rmsnorm(xd[:b], wd, out[:b], p["eps"]), out[:b])[1], 4096,
                "rmsnorm bf16 d=4096")
    ref = gbe.rmsnorm(xd, wd, p["eps"])
    for off, b in [(1, 7), (4095, 1), (100, 4000), (8191, 1), (3, 2048)]:
        y = gbe.rmsnorm(xd[off:off + b].contiguous(), wd, p["eps"])
        assert torch.equal(y.view(torch.int16), ref[off:off + b].view(torch.int16)), (off, b)
    # fused add+norm: batches of the first rows
    yf, hf = gbe.add_rmsnorm(xd, rd, wd, p["eps"])
    yo, ho = torch.empty_like(xd), torch.empty_like(xd)
    for b in list(range(1, 65)) + [100, 1000, 2047, 4096]:
        gbe.gbe_add_rmsnorm(xd[:b], rd[:b], wd, yo[:b], ho[:b], p["eps"])
        assert torch.equal(yo[:b].view(torch.int16), yf[:b].view(torch.int16)), b
        assert torch.equal(ho[:b].view(torch.int16), hf[:b].view(torch.int16)), b


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_add_rmsnorm_wide_rows_unaligned_same_bits(dtype):
    """Fused add+RMSNorm on rows of 1024 threads (d = 16384 f32 / 30000
    bf16): the scalar path gives the vector path's y and h bits."""
    d = 16384 if dtype == "f32" else 30000
    x, w = _inputs(5, d, dtype, seed=7)
    r, _ = _inputs(5, d, dtype, seed=8)
    xd, rd, wd = to_dev(x), to_dev(r), to_dev(w)
    y, h = gbe.add_rmsnorm(xd, rd, wd, 1e-5)

    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")[1:].view(t.shape)
        buf.copy_(t)
        return buf
    xs, rs = shifted(xd), shifted(rd)
    ys, hs = shifted(torch.zeros_like(xd)), shifted(torch.zeros_like(xd))
    gbe.gbe_add_rmsnorm(xs, rs, wd, ys, hs, 1e-5)
    assert np.array_equal(bits(ys), bits(y)) and np.array_equal(bits(hs), bits(h))
