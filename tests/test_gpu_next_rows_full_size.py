"""The rows beyond the step at the full prefill shapes that
`bench.py --isolated --extra` times, on the inputs the bench itself builds
and launched the way it launches them:

  * QK-norm + RoPE on q [8192, 32, 128] + k [8192, 8, 128] bf16: bit for bit
    against the unfused composition through the same library (gbe_rmsnorm
    over every head row, then gbe_rope_qk) over every token, and against the
    oracle on 64 tokens spread over the batch;
  * LayerNorm [8192, 4096] bf16 with gain and bias: the oracle on 64 rows;
  * multi-axis RoPE x [8192, 24, 128] bf16, axes 32 / 48 / 48: the oracle on
    64 tokens, and the entries past the slices unchanged;
  * RoPE of q and k driven by the cos/sin table of 8192 positions: bit for
    bit against the same call forming its angles itself (the table holds the
    same values), and the table against the oracle's.

Bars as in the smaller tests (RTOL 1e-2 for bf16, relative to the row's or
the pair's scale)."""
import numpy as np
import pytest
import torch

import bench
import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import RTOL, assert_rope_close, bits, to_dev, to_f32, widen

pytestmark = pytest.mark.gpu

T_FULL = 8192


@pytest.fixture(scope="module")
def extra():
    return bench.build_extra_inputs(T_FULL, ops=("qk_norm_rope", "rope_qk_half_cached", "layernorm", "rope_multi"))


def _spread(n_total, n=64):
    return np.linspace(0, n_total - 1, n).astype(np.int64)


def test_qk_norm_rope_full_size(extra):
    a, p = extra["qk_norm_rope"]
    q, k = to_dev(a["q"]), to_dev(a["k"])
    gq, gk = to_dev(a["gq"]), to_dev(a["gk"])
    pos, om = to_dev(a["pos"]), to_dev(a["inv_freq"])
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    bench.run_op(gbe, "qk_norm_rope", p, {"q": q, "k": k, "gq": gq, "gk": gk, "pos": pos, "inv_freq": om}, (qo, ko))
    T, Hq, D = q.shape
    Hk = k.shape[1]
    assert T == T_FULL
    qn = gbe.rmsnorm(q.reshape(T * Hq, D), gq, p["eps"]).view(T, Hq, D)
    kn = gbe.rmsnorm(k.reshape(T * Hk, D), gk, p["eps"]).view(T, Hk, D)
    gbe.gbe_rope_qk(qn, qn, kn, kn, pos, om, p["r"], p["mu"], p["layout"])
    assert np.array_equal(bits(qo), bits(qn)), "q against the unfused composition"
    assert np.array_equal(bits(ko), bits(kn)), "k against the unfused composition"
    o = oracle.get()
    t = _spread(T)
    for x, g, y, what in ((a["q"], a["gq"], qo, "q"), (a["k"], a["gk"], ko, "k")):
        xs, gw = widen(x[t]), widen(g)
        want = o.qk_norm_rope(xs, gw, p["eps"], a["pos"][t], a["inv_freq"], p["r"], p["mu"], p["layout"],
                              n_bf16=True)
        n = o.rmsnorm(xs.reshape(-1, D), gw, p["eps"]).reshape(xs.shape)
        assert_rope_close(to_f32(y)[t], want, n, p["r"], p["mu"], p["layout"], "bf16", what)


def test_layernorm_full_size(extra):
    a, p = extra["layernorm"]
    x, g, b = to_dev(a["x"]), to_dev(a["g"]), to_dev(a["b"])
    y = torch.empty_like(x)
    bench.run_op(gbe, "layernorm", p, {"x": x, "g": g, "b": b}, y)
    assert x.shape[0] == T_FULL
    rows = _spread(x.shape[0])
    bw = widen(a["b"]).astype(np.float64)
    want = oracle.get().layernorm(widen(a["x"][rows]), widen(a["g"]), widen(a["b"]), p["eps"]).astype(np.float64)
    got = to_f32(y)[rows].astype(np.float64)
    tol = RTOL["bf16"] * (np.abs(want - bw).max(axis=-1, keepdims=True) + np.abs(bw)) + 1e-30
    bad = np.abs(got - want) > tol
    assert not bad.any(), f"{int(bad.sum())} entries off, first {np.argwhere(bad)[0].tolist()}"


def test_rope_multi_full_size(extra):
    a, p = extra["rope_multi"]
    x, pos, om = to_dev(a["x"]), to_dev(a["pos"]), to_dev(a["inv_freq"])
    y = torch.empty_like(x)
    bench.run_op(gbe, "rope_multi", p, {"x": x, "pos": pos, "inv_freq": om}, y)
    assert x.shape[0] == T_FULL
    t = _spread(x.shape[0])
    xs = widen(a["x"][t])
    want = oracle.get().rope_multi(xs, a["pos"][t], p["dims"], a["inv_freq"], p["mu"], p["layout"])
    got = to_f32(y)[t]
    scale = abs(p["mu"]) * np.abs(xs).max(axis=-1, keepdims=True) * 1.5
    assert np.all(np.abs(got - want) <= RTOL["bf16"] * scale)
    rot = sum(p["dims"])
    if rot < x.shape[-1]:
        assert np.array_equal(bits(y)[..., rot:], bits(x)[..., rot:]), "entries past the slices pass through"


def test_rope_qk_from_the_table_full_size(extra):
    a, p = extra["rope_qk_half_cached"]
    q, k = to_dev(a["q"]), to_dev(a["k"])
    pos, om = to_dev(a["pos"]), to_dev(a["inv_freq"])
    table = gbe.rope_cos_sin(om, p["r"], p["cache_len"])
    want_table = oracle.get().rope_cos_sin(a["inv_freq"], p["r"], p["cache_len"])
    diff = np.abs(table.cpu().numpy().astype(np.float64) - want_table)
    assert np.all(diff <= 4e-7), ("cos/sin table", float(diff.max()))
    qa, ka = torch.empty_like(q), torch.empty_like(k)
    bench.run_op(gbe, "rope_qk_half_cached", p, {"q": q, "k": k, "pos": pos, "inv_freq": om, "cos_sin": table},
                 (qa, ka))
    qb, kb = torch.empty_like(q), torch.empty_like(k)
    gbe.gbe_rope_qk(q, qb, k, kb, pos, om, p["r"], p["mu"], p["layout"])
    assert q.shape[0] == T_FULL
    assert np.array_equal(bits(qa), bits(qb)), "q: table against formed angles"
    assert np.array_equal(bits(ka), bits(kb)), "k: table against formed angles"
