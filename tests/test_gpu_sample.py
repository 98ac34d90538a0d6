"""Sampling on the GPU against the oracle, through the C ABI.

The oracle evaluates the definition in f32 (running sums in the
distribution's order); the kernel sums fixed-point weights exactly (per
entry for top-k / top-p, per unit of 4 or 8 consecutive entries summed in
f32 for temperature / min-p).  Both are
the inverse CDF at the same u, so they pick the same entry except where u
lies within rounding of a boundary between two entries, or an entry sits
within rounding of a top-p / min-p cut.  The bar:
  * every row where the two differ is such a case: u lies within DELTA of
    the boundary between them in the float64 distribution (written from the
    definition in pins.sampling_probs_f64, independently of both), or the
    row has a keep/cut decision within DELTA of its threshold, and then the
    kernel's pick is still an entry the float64 distribution keeps;
  * such rows are few (MAX_MISS of the rows);
  * on flat rows of 152k entries, where the oracle's f32 running sums drift
    across boundaries, every draw is held to the float64 distribution within
    2e-6 (the kernel's sums are exact; its weights carry a few f32 roundings
    of the exponent, log2(e) / t among them, which shift the whole CDF by at
    most |x - max| / t * 1e-7 of the mass);
  * exact limits: top_k = 1 and top_p = 0 give the argmax; min_p = 0 gives
    the temperature draw; a row with no number, or with +inf, gives -1.
DELTA = 1e-5 of the kept mass covers the f32 running sums of rows of up to
152k entries in the oracle and the f32 rounding of x / t in both."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import to_dev, widen
from pins import sampling_probs_f64
from synth import normal, to_bf16, units
from synth import workloads as W

pytestmark = pytest.mark.gpu

DELTA = 1e-5
MAX_MISS = 0.05

METHODS = [("temperature", dict(temperature=0.8)), ("top_k", dict(temperature=1.3, top_k=50)),
           ("top_p", dict(temperature=0.9, p=0.9)), ("min_p", dict(temperature=1.0, p=0.05))]


def _oracle(x32, u, method, kw):
    okw = dict(temperature=kw.get("temperature", 1.0), top_k=kw.get("top_k", 1))
    if method == "top_p":
        okw["top_p"] = kw["p"]
    if method == "min_p":
        okw["min_p"] = kw["p"]
    return oracle.get().sample(x32, method, u, **okw)


def _interval(x_row, method, kw, idx):
    """(lo, hi) of entry idx in the float64 CDF, and the row's cut margin."""
    pr, order, margin = sampling_probs_f64(x_row, method, t=kw.get("temperature", 1.0), k=kw.get("top_k", 1),
                                           p=kw.get("p", 1.0))
    c = np.cumsum(pr[order])
    pos = np.nonzero(order == idx)[0]
    if idx < 0 or pos.size == 0 or pr[idx] <= 0:
        return None, margin
    hi = c[pos[0]]
    return (hi - pr[idx], hi), margin


def _valid_draw(x_row, u, method, kw, idx, delta):
    """idx is the float64 inverse CDF at u up to delta: u lies within delta of
    idx's interval; where a keep/cut decision of the row lies within delta of
    its threshold, idx need only be a number of the row."""
    g, m = _interval(x_row, method, kw, idx)
    if m < delta:
        return 0 <= idx < len(x_row) and not np.isnan(x_row[idx])
    return g is not None and g[0] - delta <= u <= g[1] + delta


def _check(x, u, method, kw, what, max_miss=MAX_MISS):
    xd = to_dev(x)
    ud = torch.from_numpy(np.ascontiguousarray(u, np.float32)).cuda()
    got = gbe.sample(xd, ud, method, **kw).cpu().numpy()
    x32 = widen(x)
    want = _oracle(x32, u, method, kw)
    miss = np.nonzero(got != want)[0]
    for r in miss:
        assert _valid_draw(x32[r], float(u[r]), method, kw, int(got[r]), DELTA), (
            f"{what}: row {r} u={u[r]} drew {got[r]}, oracle {want[r]}: not within rounding of a boundary")
    assert miss.size <= max(1, max_miss * len(got)), f"{what}: {miss.size} of {len(got)} rows differ"
    return got


def _logits(rows, n, dtype, seed=31, std=4.0, nan_frac=0.0, tag="s"):
    x = normal(seed, f"t.smp.{tag}.{rows}.{n}", (rows, n), 0.0, std)
    if nan_frac:
        v = units(seed, f"t.smp.nan.{tag}.{rows}.{n}", rows * n).reshape(rows, n)
        x[v < nan_frac] = np.nan
    return to_bf16(x) if dtype == "bf16" else x


def _u(rows, tag, seed=31):
    return units(seed, f"t.smp.u.{tag}.{rows}", rows).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("method,kw", METHODS)
@pytest.mark.parametrize("rows,n", [(1, 1), (3, 7), (9, 1000), (4, 4097), (16, 32000), (2, 65536 + 3)])
def test_shapes(dtype, method, kw, rows, n):
    x = _logits(rows, n, dtype, nan_frac=0.01)
    u = _u(rows, f"{rows}.{n}")
    _check(x, u, method, kw, f"{method} {dtype} [{rows},{n}]")


@pytest.mark.parametrize("method,kw", METHODS)
def test_decode_logits(method, kw):
    """The decode workload's logits: 64 rows of a 128256-entry vocabulary, bf16."""
    a, _ = W.cases(W.DECODE)["argmax"]()
    x = a["x"]
    u = _u(x.shape[0], "decode")
    _check(x, u, method, kw, f"{method} decode")


@pytest.mark.parametrize("method,kw", [("temperature", dict(temperature=1.0)),
                                       ("top_k", dict(temperature=0.7, top_k=1000)),
                                       ("top_p", dict(temperature=1.0, p=0.5)),
                                       ("min_p", dict(temperature=0.6, p=0.001))])
def test_flat_wide_rows(method, kw):
    """Flat logits over 152064 entries, f32, with NaN and exact ties: every
    entry carries mass, so boundaries lie ~1e-5 apart and the oracle's f32
    running sums drift across several of them.  Here every draw is held to
    the float64 distribution itself, within 2e-6 of the kept mass."""
    x = _logits(24, 152064, "f32", std=0.5, nan_frac=0.001, tag="flat")
    x[:, 100:200] = x[:, 1000:1100]
    u = _u(24, f"flat.{method}")
    got = gbe.sample(to_dev(x), torch.from_numpy(u).cuda(), method, **kw).cpu().numpy()
    for r in range(24):
        assert _valid_draw(x[r], float(u[r]), method, kw, int(got[r]), 2e-6), (method, r, u[r], got[r])


def test_draws_in_proportion():
    """Inverse CDF on the GPU: over a grid of 4000 u, each index of a short
    row is drawn 4000 * p_i times (+-2.5), p_i from the float64 definition."""
    rng = np.random.default_rng(7)
    for trial in range(4):
        x = (rng.standard_normal(60) * 2.0).astype(np.float32)
        x[[5, 17]] = x[3]
        x[11] = np.nan
        for method, kw in (("temperature", dict(temperature=0.8)), ("top_k", dict(temperature=1.3, top_k=7)),
                           ("top_p", dict(temperature=0.9, p=0.6)), ("min_p", dict(temperature=1.0, p=0.2))):
            pr, _, margin = sampling_probs_f64(x, method, t=kw["temperature"], k=kw.get("top_k", 1),
                                               p=kw.get("p", 1.0))
            if margin < 1e-4:
                continue
            u = ((np.arange(4000) + 0.5) / 4000).astype(np.float32)
            rows = torch.from_numpy(np.repeat(x.reshape(1, -1), 4000, axis=0)).cuda()
            got = gbe.sample(rows, torch.from_numpy(u).cuda(), method, **kw).cpu().numpy()
            counts = np.bincount(got, minlength=60)
            assert np.all(np.abs(counts - 4000 * pr) <= 2.5), (trial, method, np.abs(counts - 4000 * pr).max())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_limits(dtype):
    x = _logits(40, 5000, dtype, nan_frac=0.02, tag="lim")
    x32 = widen(x)
    x32[3] = np.nan
    x32[4, :] = -np.inf
    x32[5, 77] = np.inf
    x32[6, 10] = x32[6, 4000] = 60.0  # tie at the maximum
    x = to_bf16(x32) if dtype == "bf16" else x32
    xd = to_dev(x)
    u = torch.from_numpy(_u(40, "lim")).cuda()
    want = gbe.argmax(xd).cpu().numpy()
    g = lambda m, **kw: gbe.sample(xd, u, m, **kw).cpu().numpy()
    got_k1 = g("top_k", temperature=0.7, top_k=1)
    got_p0 = g("top_p", temperature=1.0, p=0.0)
    greedy = gbe.sample(xd, None, "greedy").cpu().numpy()
    assert np.array_equal(greedy, want)
    for got in (got_k1, got_p0):
        assert np.array_equal(np.delete(got, [4, 5]), np.delete(want, [4, 5]))
        assert got[4] == -1 and got[5] == -1
    assert got_k1[6] == 10
    for m, kw in METHODS:
        got = g(m, **kw)
        assert got[3] == -1 and got[4] == -1 and got[5] == -1, m
    assert np.array_equal(g("min_p", temperature=0.9, p=0.0), g("temperature", temperature=0.9))
    # min_p = 1 keeps only the entries equal to the maximum
    got = g("min_p", temperature=1.0, p=1.0)
    assert np.array_equal(np.delete(got, [4, 5, 6]), np.delete(want, [4, 5, 6]))
    assert got[6] in (10, 4000)
    # x / t overflowing to +inf leaves no finite maximum
    big = torch.full((1, 64), 3e38, device="cuda")
    assert gbe.sample(big, u[:1], "temperature", temperature=0.5).item() == -1


def test_u_edges_and_top_k_past_n():
    x = _logits(8, 3000, "f32", tag="edge")
    xd = to_dev(x)
    for uu, pick in ((0.0, "first"), (np.nextafter(np.float32(1), np.float32(0)), "last"), (-3.0, "first"),
                     (7.0, "last")):
        u = torch.full((8,), float(uu), device="cuda")
        got = gbe.sample(xd, u, "top_k", temperature=1.0, top_k=10).cpu().numpy()
        for r in range(8):
            order = sorted(range(3000), key=lambda i: (-x[r, i], i))[:10]
            assert got[r] == (order[0] if pick == "first" else order[-1]), (uu, r)
    u = torch.from_numpy(_u(8, "edge")).cuda()
    a = gbe.sample(xd, u, "top_k", temperature=1.0, top_k=3000).cpu().numpy()
    b = gbe.sample(xd, u, "top_k", temperature=1.0, top_k=1 << 40).cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("method,kw", METHODS)
def test_unaligned_and_batch_invariant(dtype, method, kw):
    """The scalar path (rows not 16-byte aligned) draws what the vector path
    does, and a row's draw does not depend on the rows around it."""
    rows, n = 12, 8192
    x = _logits(rows, n, dtype, nan_frac=0.01, tag="inv")
    xd = to_dev(x)
    u = torch.from_numpy(_u(rows, "inv")).cuda()
    ref = gbe.sample(xd, u, method, **kw).cpu().numpy()
    buf = torch.empty(rows * n + 1, dtype=xd.dtype, device="cuda")
    xs = buf[1:].view(rows, n)
    xs.copy_(xd)
    assert np.array_equal(gbe.sample(xs, u, method, **kw).cpu().numpy(), ref)
    for r0, r1 in ((0, 1), (3, 7), (11, 12)):
        got = gbe.sample(xd[r0:r1].contiguous(), u[r0:r1].contiguous(), method, **kw).cpu().numpy()
        assert np.array_equal(got, ref[r0:r1]), (r0, r1)


@pytest.mark.parametrize("method,kw", METHODS)
def test_prefill_logits_sampled_rows(method, kw):
    """All 8192 rows of the prefill logits [8192, 128256] bf16 in one launch;
    64 of them checked against the oracle."""
    a, _ = W.cases(W.PREFILL)["argmax"]()
    x = a["x"]
    u = _u(x.shape[0], "prefill")
    got = gbe.sample(to_dev(x), torch.from_numpy(u).cuda(), method, **kw).cpu().numpy()
    pick = np.linspace(0, x.shape[0] - 1, 64).astype(np.int64)
    sub = _check(x[pick], u[pick], method, kw, f"{method} prefill rows")
    assert np.array_equal(got[pick], sub)


@pytest.mark.parametrize("method,kw", METHODS + [("top_k", dict(temperature=0.7, top_k=300))])
def test_draws_do_not_depend_on_the_split(method, kw):
    """Batches too small to fill the GPU split each row over a cluster of 2, 4
    or 8 CTAs; large ones take one CTA a row.  The same rows give the same
    draws in a batch of 320 (one CTA a row), 48, 16 and 1 (clusters), NaN
    entries included; a few rows are also checked against the oracle."""
    rows, n = 320, 131072
    x = _logits(rows, n, "bf16", nan_frac=0.001, tag="split")
    xd = to_dev(x)
    u = torch.from_numpy(_u(rows, "split")).cuda()
    ref = gbe.sample(xd, u, method, **kw).cpu().numpy()
    for r0, r1 in ((0, 48), (100, 116), (7, 8), (319, 320)):
        got = gbe.sample(xd[r0:r1].contiguous(), u[r0:r1].contiguous(), method, **kw).cpu().numpy()
        assert np.array_equal(got, ref[r0:r1]), (r0, r1)
    _check(x[:8], u[:8].cpu().numpy(), method, kw, f"{method} split rows", max_miss=1.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rows_without_a_maximum_in_a_split_batch(dtype):
    """A small batch of wide rows is split over clusters (eight CTAs a row
    for temperature and min-p at this size): a row of NaN, a row of -inf
    and a row holding +inf still give -1, every CTA of their clusters
    leaving together, and the other rows draw what they draw in a batch of
    one CTA a row."""
    n = 131072
    x32 = widen(_logits(4, n, dtype, nan_frac=0.001, tag="split.lim"))
    x32[1] = np.nan
    x32[2, :] = -np.inf
    x32[3, 5] = np.inf
    x = to_bf16(x32) if dtype == "bf16" else x32
    xd = to_dev(x)
    big = torch.cat([xd] * 80)  # 320 rows: one CTA a row
    u = torch.from_numpy(_u(4, "split.lim")).cuda()
    ub = torch.cat([u] * 80)
    for m, kw in METHODS:
        got = gbe.sample(xd, u, m, **kw).cpu().numpy()
        assert got[1] == -1 and got[2] == -1 and got[3] == -1, (m, got)
        ref = gbe.sample(big, ub, m, **kw).cpu().numpy()
        assert np.array_equal(got, ref[:4]), (m, got, ref[:4])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rows_walked_by_resident_ctas(dtype):
    """A batch larger than the resident CTAs (1500 rows: several waves),
    with rows of NaN, of -inf, holding +inf, of equal logits and with one
    dominant entry in among them: every row draws what it draws alone or in
    a small batch, the rows without a maximum give -1, and some are checked
    against the oracle."""
    rows, n = 1500, 8192
    x32 = widen(_logits(rows, n, dtype, nan_frac=0.002, tag="resident"))
    x32[5] = np.nan
    x32[306, :] = -np.inf
    x32[457, 17] = np.inf
    x32[700] = 1.5
    x32[1499, 4000] = 60.0
    x = to_bf16(x32) if dtype == "bf16" else x32
    xd = to_dev(x)
    u = torch.from_numpy(_u(rows, "resident")).cuda()
    for m, kw in METHODS + [("top_k", dict(temperature=0.7, top_k=300))]:
        got = gbe.sample(xd, u, m, **kw).cpu().numpy()
        assert got[5] == -1 and got[306] == -1 and got[457] == -1, (m, got[[5, 306, 457]])
        assert got[1499] == 4000, m
        for r0, r1 in ((0, 1), (5, 6), (300, 320), (699, 701), (1490, 1500)):
            ref = gbe.sample(xd[r0:r1].contiguous(), u[r0:r1].contiguous(), m, **kw).cpu().numpy()
            assert np.array_equal(got[r0:r1], ref), (m, r0, r1)
        pick = np.array([0, 1, 303, 304, 455, 456, 700, 1200])
        sub = _check(x[pick], u[pick].cpu().numpy(), m, kw, f"{m} resident rows", max_miss=1.0)
        assert np.array_equal(got[pick], sub), m


def test_top_p_rows_past_the_first_gather():
    """Top-p 0.9 at t = 0.7 on the first 512 rows of the prefill logits (the
    bench's setting): in about 2 % of them the first, narrow gather of the
    row's top holds less than the cut's mass, and a wider round (or the exact
    search) decides.  Every draw is held to the float64 distribution within
    2e-6, and every difference from the oracle is a boundary case."""
    kw = dict(temperature=0.7, p=0.9)
    a, _ = W.cases(W.PREFILL)["argmax"](rows=(0, 512))
    x = a["x"]
    u = _u(x.shape[0], "topp.rounds")
    got = _check(x, u, "top_p", kw, "top_p prefill rows", max_miss=1.0)
    x32 = widen(x)
    for r in range(x.shape[0]):
        assert _valid_draw(x32[r], float(u[r]), "top_p", kw, int(got[r]), 2e-6), (r, u[r], got[r])


def test_refusals_on_device():
    x = torch.randn(4, 1000, device="cuda")
    u = torch.rand(4, device="cuda")
    out = torch.empty(4, dtype=torch.int32, device="cuda")
    L = gbe.lib()
    # out inside x: an alias
    assert L.gbe_sample(x.data_ptr(), u.data_ptr(), x.data_ptr() + 64, 4, 1000, 1, 1.0, 1, 1.0, 0, None) == 8
    # u in pageable host memory
    uh = torch.rand(4)
    assert L.gbe_sample(x.data_ptr(), uh.data_ptr(), out.data_ptr(), 4, 1000, 1, 1.0, 1, 1.0, 0, None) == 10
    # u NULL: refused except for greedy, which does not read it
    assert L.gbe_sample(x.data_ptr(), None, out.data_ptr(), 4, 1000, 1, 1.0, 1, 1.0, 0, None) == 1
    assert L.gbe_sample(x.data_ptr(), None, out.data_ptr(), 4, 1000, 0, 0.0, 0, 9.0, 0, None) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, gbe.argmax(x))
    with pytest.raises(gbe.GbeError):
        gbe.sample(x, u, "top_k", temperature=1.0, top_k=0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_search_paths(dtype):
    """The less common routes of the descending search: top-k past the
    gather limit (the full histogram, split by the next digits), top-p with
    p = 1 and p = 0.999 (the cut past the head of the row), groups of more
    equal logits than the gather limit (walked in index order), and a row of
    a few repeated values.  Over tens of thousands of equal probabilities the
    oracle's f32 running sums drift by more than one entry, so here any row
    may differ from it, and every draw is held to the float64 distribution
    (within DELTA of a boundary)."""
    rows, n = 6, 65536
    x = _logits(rows, n, dtype, std=1.0, tag="paths")
    x32 = widen(x)
    x32[2] = 0.75                                              # one value: a single group of n
    x32[3] = np.floor(units(31, "paths.rep", n) * 3) / 8.0     # three values, ~n/3 each
    x32[4, : n // 2] = 0.5                                     # half tied at the top
    x = to_bf16(x32) if dtype == "bf16" else x32
    u = _u(rows, "paths")
    for method, kw in (("top_k", dict(temperature=1.0, top_k=20000)), ("top_k", dict(temperature=0.5, top_k=5000)),
                       ("top_k", dict(temperature=1.0, top_k=3)), ("top_p", dict(temperature=1.0, p=1.0)),
                       ("top_p", dict(temperature=0.8, p=0.999)), ("top_p", dict(temperature=1.0, p=0.5)),
                       ("top_p", dict(temperature=2.0, p=0.2))):
        _check(x, u, method, kw, f"{method} {kw} {dtype}", max_miss=1.0)


def test_equal_logits_exact():
    """8192 equal logits (a group larger than the gather limit): every
    method reduces to a uniform draw over a prefix in index order, and with a
    power-of-two count the oracle's f32 sums are exact, so the draws match
    exactly."""
    n = 8192
    x = np.full((8, n), 1.5, np.float32)
    u = _u(8, "equal")
    xd = to_dev(x)
    ud = torch.from_numpy(u).cuda()
    for method, kw, m in (("temperature", dict(temperature=1.0), n), ("top_k", dict(temperature=1.0, top_k=4096), 4096),
                          ("top_p", dict(temperature=1.0, p=0.5), 4096), ("min_p", dict(temperature=1.0, p=0.5), n)):
        got = gbe.sample(xd, ud, method, **kw).cpu().numpy()
        want = np.floor(u.astype(np.float64) * m).astype(np.int64)
        assert np.array_equal(got, want), (method, got, want)
        assert np.array_equal(got, _oracle(x, u, method, kw)), method


@pytest.mark.parametrize("method,kw", [("top_k", dict(temperature=1.0, top_k=1)),
                                       ("top_k", dict(temperature=0.8, top_k=16)),
                                       ("top_k", dict(temperature=1.0, top_k=100)),
                                       ("top_k", dict(temperature=1.0, top_k=300)),
                                       ("top_k", dict(temperature=1.2, top_k=512)),
                                       ("top_p", dict(temperature=0.5, p=0.95)),
                                       ("top_p", dict(temperature=1.0, p=0.8)),
                                       ("top_p", dict(temperature=2.0, p=0.6))])
def test_candidate_counts(method, kw):
    """The decode logits with k and temperatures that gather from a few to a
    few thousand candidates: the one-warp register sort (up to 256), the
    block sort (up to 4096) and the exact search past that.  Every draw is
    held to the float64 distribution within 2e-6.  Against the oracle every
    difference must be a boundary case, but their number is not capped: at
    higher temperatures the cut falls among hundreds to thousands of small
    entries, and the oracle's f32 running sum drifts across several of them
    (as on the flat rows above)."""
    a, _ = W.cases(W.DECODE)["argmax"]()
    x = a["x"]
    u = _u(x.shape[0], f"cand.{method}.{kw.get('top_k', kw.get('p'))}")
    got = _check(x, u, method, kw, f"{method} {kw} decode", max_miss=1.0)
    x32 = widen(x)
    for r in range(x.shape[0]):
        assert _valid_draw(x32[r], float(u[r]), method, kw, int(got[r]), 2e-6), (method, kw, r, u[r], got[r])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_signed_zeros_are_equal_logits(dtype):
    """-0 and +0 are equal logits, ordered by index like any other equal
    logits ("Operations" section 8 sorts descending; equal logits keep index
    order, and -0 equals +0 as in the argmax rule of "Elementwise kernels in
    C" section 2.4).  Rows whose largest entries are zeros of both signs, -0
    at lower indices than +0: top-k cuts between them and top-p walks across
    them.  The weights of the zeros are exactly 2^40 each and every other
    entry is far below them, so the draw is the floor(u * m)-th kept zero in
    index order, exactly, for m kept zeros; the oracle must agree."""
    rows, n = 16, 4096
    x = normal(37, f"t.smp.zero.{n}", (rows, n), -40.0, 1.0)
    x = np.minimum(x, -30.0).astype(np.float32)
    zeros = []
    for r in range(rows):
        pos = np.sort(np.unique((units(37, f"t.smp.zero.pos.{r}", 8) * n).astype(np.int64)))[:6]
        assert len(pos) == 6
        sign = np.array([-0.0, -0.0, 0.0, -0.0, 0.0, 0.0], np.float32)
        if r % 2:
            sign = -sign  # +0 first on odd rows
        x[r, pos] = sign
        zeros.append(pos)
    assert np.signbit(x[0, zeros[0][0]]) and not np.signbit(x[0, zeros[0][2]])
    xx = to_bf16(x) if dtype == "bf16" else x
    xd = to_dev(xx)
    u = _u(rows, "zero")
    ud = torch.from_numpy(u).cuda()
    x32 = widen(xx)
    for method, kw, m in (("top_k", dict(temperature=1.0, top_k=1), 1),
                          ("top_k", dict(temperature=1.0, top_k=3), 3),
                          ("top_k", dict(temperature=0.7, top_k=5), 5),
                          ("top_p", dict(temperature=1.0, p=0.6), 3),
                          ("top_p", dict(temperature=1.0, p=0.4), 2)):
        got = gbe.sample(xd, ud, method, **kw).cpu().numpy()
        want = np.array([zeros[r][int(np.floor(np.float64(u[r]) * m))] for r in range(rows)])
        assert np.array_equal(got, want), (method, kw, got, want)
        assert np.array_equal(got, _oracle(x32, u, method, kw)), (method, kw)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_many_signed_zeros_take_the_exact_search(dtype):
    """2000 zeros of random sign among 8192 entries far below them: top-k
    with k = 600 (past the gathered paths, so the exact radix search) and
    top-p with p = 0.3001 (600 of 2000 equal weights) keep the first 600
    zeros in index order, whatever their signs."""
    rows, n, nz = 4, 8192, 2000
    x = np.minimum(normal(41, "t.smp.zeros.many", (rows, n), -40.0, 1.0), -30.0).astype(np.float32)
    zeros = []
    for r in range(rows):
        perm = np.argsort(units(41, f"t.smp.zeros.perm.{r}", n))
        pos = np.sort(perm[:nz])
        sgn = units(41, f"t.smp.zeros.sign.{r}", nz) < 0.5
        x[r, pos] = np.where(sgn, np.float32(-0.0), np.float32(0.0))
        zeros.append(pos)
    xx = to_bf16(x) if dtype == "bf16" else x
    xd = to_dev(xx)
    u = _u(rows, "zeros.many")
    ud = torch.from_numpy(u).cuda()
    for method, kw in (("top_k", dict(temperature=1.0, top_k=600)), ("top_p", dict(temperature=1.0, p=0.3001))):
        got = gbe.sample(xd, ud, method, **kw).cpu().numpy()
        want = np.array([zeros[r][int(np.floor(np.float64(u[r]) * 600))] for r in range(rows)])
        assert np.array_equal(got, want), (method, got, want)
        assert np.array_equal(got, _oracle(widen(xx), u, method, kw)), method


# ---- the seeded draw ("Operations" section 8: sample_categorical with a
# seeded PCG generator; same seed, same distribution, same draw) -----------------

@pytest.mark.parametrize("seed,offset,n", [(0, 0, 1), (42, 0, 100003), (7, (1 << 40) + 3, 4097),
                                           ((1 << 64) - 1, (1 << 64) - 50, 1000), (3, 12345, 31)])
def test_pcg64_uniforms_match_the_oracle(seed, offset, n):
    """The device stream equals the oracle's bit for bit, including draws
    past 2^64 and ragged warps."""
    got = gbe.pcg64_uniforms(n, seed, offset).cpu().numpy()
    want = oracle.get().pcg64_uniforms(seed, offset, n)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("method,kw", METHODS)
@pytest.mark.parametrize("rows,n", [(3, 1000), (16, 32000), (200, 4097)])
def test_seeded_draws_are_the_draws_at_the_streams_uniforms(dtype, method, kw, rows, n):
    """Row r of a seeded call draws exactly what gbe_sample draws at the
    uniform of stream draw offset + r (the kernel forms that uniform itself);
    against the oracle's seeded sampler, the usual boundary rule."""
    x = _logits(rows, n, dtype, nan_frac=0.01, tag="seeded")
    xd = to_dev(x)
    for seed, offset in ((11, 0), (11, 1 << 33), ((1 << 64) - 2, 17)):
        got = gbe.sample_seeded(xd, method, seed, offset, **kw).cpu().numpy()
        u = oracle.get().pcg64_uniforms(seed, offset, rows)
        ref = gbe.sample(xd, torch.from_numpy(u).cuda(), method, **kw).cpu().numpy()
        assert np.array_equal(got, ref), (method, seed, offset)
        _check(x, u, method, kw, f"seeded {method} {dtype} [{rows},{n}]")


@pytest.mark.parametrize("method,kw", METHODS)
def test_seeded_reproducible_and_batch_invariant(method, kw):
    """The same seed and offset give the same draws; rows [r0, r1) drawn
    alone at offset + r0 equal those rows of the whole batch; another seed
    gives other draws."""
    rows, n = 64, 32000
    x = _logits(rows, n, "bf16", tag="seeded.inv")
    xd = to_dev(x)
    a = gbe.sample_seeded(xd, method, 5, 1000, **kw).cpu().numpy()
    assert np.array_equal(a, gbe.sample_seeded(xd, method, 5, 1000, **kw).cpu().numpy())
    for r0, r1 in ((0, 1), (7, 30), (63, 64)):
        part = gbe.sample_seeded(xd[r0:r1], method, 5, 1000 + r0, **kw).cpu().numpy()
        assert np.array_equal(part, a[r0:r1]), (r0, r1)
    b = gbe.sample_seeded(xd, method, 6, 1000, **kw).cpu().numpy()
    assert (a != b).sum() > rows // 4, method


def test_seeded_greedy_and_refusals():
    x = to_dev(_logits(4, 1000, "f32", tag="seeded.g"))
    assert torch.equal(gbe.sample_seeded(x, "greedy", 1, 0), gbe.argmax(x))
    with pytest.raises(gbe.GbeError) as e:
        gbe.sample_seeded(x, "top_k", 1, 0, top_k=0)
    assert e.value.status == 12
    L = gbe.lib()
    s = torch.cuda.current_stream().cuda_stream
    u = torch.full((8,), 7.0, device="cuda")
    assert L.gbe_pcg64_uniforms(u.data_ptr(), -1, 1, 0, s) == 2
    assert L.gbe_pcg64_uniforms(None, 8, 1, 0, s) == 1
    assert L.gbe_pcg64_uniforms(u.data_ptr(), 0, 1, 0, s) == 0
    torch.cuda.synchronize()
    assert torch.all(u == 7.0)
