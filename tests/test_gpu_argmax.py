"""Greedy argmax on the GPU against the oracle, bit exact, through the C ABI:
planted ties and NaN, rows with no number, -inf rows, signed zeros, +inf,
every cluster split of the row, the scalar path, and the full workloads."""
import numpy as np
import pytest

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import to_dev, widen
from synth import normal, to_bf16, units
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _check(x, what):
    got = gbe.argmax(to_dev(x)).cpu().numpy()
    want = oracle.get().argmax(widen(x))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{what}: rows {bad[:8].tolist()} got {got[bad[:8]]} want {want[bad[:8]]}"
    return got


def test_tiny_planted():
    a, p = W.cases(W.TINY)["argmax"]()
    got = _check(a["x"], "tiny")
    assert got[2] == -1 and got[3] == 0


def test_decode_bf16():
    a, p = W.cases(W.DECODE)["argmax"]()
    _check(a["x"], "decode [64,128256] bf16")


def test_wide_f32_full():
    a, p = W.cases(W.WIDE)["argmax"]()
    got = _check(a["x"], "[1024,152064] f32")
    x = a["x"]
    tied = np.nonzero((x == np.float32(30.0)).sum(axis=1) == 2)[0]
    assert tied.size > 20
    for r in tied:
        assert got[r] == np.nonzero(x[r] == np.float32(30.0))[0][0]


def test_prefill_bf16_full():
    a, p = W.cases(W.PREFILL)["argmax"]()
    _check(a["x"], "[8192,128256] bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,n", [(1, 1), (1, 7), (3, 8), (5, 1000), (2, 4097), (64, 128256), (1, 152064),
                                    (300, 5000), (2000, 777), (17, 65536 + 3)])
def test_shapes_and_splits(dtype, rows, n):
    x = normal(21, f"t.am.{rows}.{n}", (rows, n), 0.0, 4.0)
    u = units(21, f"t.am.nan.{rows}.{n}", rows * n).reshape(rows, n)
    x[u < 0.02] = np.nan
    if rows > 2:
        x[1] = np.nan
        x[2] = -np.inf
    if dtype == "bf16":
        x = to_bf16(x)
        if rows > 4:  # coarse values: many exact ties at the top
            x[4] = to_bf16(np.round(widen(x[4:5]) * 0.5)[0] * 2)
    got = _check(x, f"{dtype} [{rows},{n}]")
    if rows > 2:
        assert got[1] == -1 and got[2] == 0


def test_special_values():
    rows = [
        [0.0, -0.0, -1.0],
        [-0.0, 0.0, -1.0],
        [np.nan, np.inf, np.inf, 1.0],
        [-np.inf, np.nan, -np.inf],
        [np.nan, np.nan, np.nan, 3.0],
        [5.0, 5.0, 5.0, 5.0],
    ]
    n = max(len(r) for r in rows)
    x = np.full((len(rows), n), np.nan, np.float32)
    for i, r in enumerate(rows):
        x[i, :len(r)] = r
    got = _check(x, "special values")
    assert got.tolist() == [0, 0, 1, 0, 3, 0]
