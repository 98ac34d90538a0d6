"""The C ABI on the host, no GPU needed: the library loads, exports every
function include/*.h declares, and rejects invalid arguments before any CUDA
call (only checks that return before touching the device are exercised)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import elementwise_row_rmsnorm_gb300 as gbe
    gbe.build()
    return gbe.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gbe_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_ops():
    names = declared_functions()
    for op in ("gbe_rmsnorm", "gbe_add_rmsnorm", "gbe_rope", "gbe_rope_qk", "gbe_rope_cos_sin", "gbe_rope_multi", "gbe_qk_norm_rope", "gbe_silu_mul",
               "gbe_add", "gbe_embedding", "gbe_argmax", "gbe_sample", "gbe_layernorm", "gbe_status_string", "gbe_version",
               "gbe_last_cuda_error", "gbe_sample_seeded", "gbe_pcg64_uniforms"):
        assert op in names


def test_library_exports_every_declared_function(L):
    import elementwise_row_rmsnorm_gb300.binding as b
    out = subprocess.run(["nm", "-D", "--defined-only", b.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(gbe_\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_status_strings_and_version(L):
    import elementwise_row_rmsnorm_gb300 as gbe
    assert L.gbe_version() == 10100
    for st in range(13):
        assert gbe.status_string(st) and gbe.status_string(st) != "unknown status"
    assert gbe.status_string(99) == "unknown status"


NULL = None
S = None  # default stream handle; never reached by these calls


def test_rejects_bad_sizes_and_scalars(L):
    assert L.gbe_rmsnorm(NULL, NULL, NULL, 4, 0, 1e-5, 0, S) == 2          # d <= 0
    assert L.gbe_rmsnorm(NULL, NULL, NULL, -1, 8, 1e-5, 0, S) == 2         # rows < 0
    assert L.gbe_rmsnorm(NULL, NULL, NULL, 4, 8, 1e-5, 7, S) == 3          # dtype
    assert L.gbe_rmsnorm(NULL, NULL, NULL, 4, 8, -1.0, 0, S) == 5          # eps < 0
    assert L.gbe_rmsnorm(NULL, NULL, NULL, 4, 8, float("nan"), 1, S) == 5  # eps NaN
    assert L.gbe_rmsnorm(NULL, NULL, NULL, 4, 8, float("inf"), 1, S) == 5
    assert L.gbe_rmsnorm(NULL, NULL, NULL, 0, 8, 1e-5, 0, S) == 0          # empty: no-op
    assert L.gbe_add_rmsnorm(NULL, NULL, NULL, NULL, NULL, 2, 8, -3.0, 0, S) == 5
    assert L.gbe_add_rmsnorm(NULL, NULL, NULL, NULL, NULL, 0, 8, 1e-5, 0, S) == 0
    assert L.gbe_layernorm(NULL, NULL, NULL, NULL, 4, 0, 1e-5, 0, S) == 2
    assert L.gbe_layernorm(NULL, NULL, NULL, NULL, 4, 8, float("nan"), 0, S) == 5
    assert L.gbe_layernorm(NULL, NULL, NULL, NULL, 4, 8, 1e-5, 3, S) == 3
    assert L.gbe_layernorm(NULL, NULL, NULL, NULL, 0, 8, 1e-5, 1, S) == 0
    # rope: layout, width, scaling, shapes
    assert L.gbe_rope(NULL, NULL, NULL, 4, 2, 16, 8, NULL, 1.0, 2, 0, S) == 4
    assert L.gbe_rope(NULL, NULL, NULL, 4, 2, 16, 7, NULL, 1.0, 0, 0, S) == 6   # odd r
    assert L.gbe_rope(NULL, NULL, NULL, 4, 2, 16, 18, NULL, 1.0, 0, 0, S) == 6  # r > D
    assert L.gbe_rope(NULL, NULL, NULL, 4, 2, 16, -2, NULL, 1.0, 0, 0, S) == 6
    assert L.gbe_rope(NULL, NULL, NULL, 4, 2, 16, 8, NULL, float("inf"), 0, 0, S) == 6
    assert L.gbe_rope(NULL, NULL, NULL, 4, 2, 0, 0, NULL, 1.0, 0, 0, S) == 2
    assert L.gbe_rope(NULL, NULL, NULL, -4, 2, 16, 8, NULL, 1.0, 0, 0, S) == 2
    assert L.gbe_rope(NULL, NULL, NULL, 0, 2, 16, 8, NULL, 1.0, 0, 0, S) == 0
    assert L.gbe_rope(NULL, NULL, NULL, 4, 0, 16, 8, NULL, 1.0, 0, 1, S) == 0
    # pointwise
    assert L.gbe_silu_mul(NULL, NULL, NULL, -1, 0, S) == 2
    assert L.gbe_silu_mul(NULL, NULL, NULL, 0, 1, S) == 0
    assert L.gbe_add(NULL, NULL, NULL, 5, 2, S) == 3
    assert L.gbe_add(NULL, NULL, NULL, 0, 0, S) == 0
    # embedding
    assert L.gbe_embedding(NULL, NULL, NULL, 3, 0, 10, NULL, 0, S) == 2
    assert L.gbe_embedding(NULL, NULL, NULL, 3, 4, -1, NULL, 0, S) == 2
    assert L.gbe_embedding(NULL, NULL, NULL, 0, 4, 10, NULL, 1, S) == 0
    # argmax: rows of length 0 are rejected, no rows is a no-op
    assert L.gbe_argmax(NULL, NULL, 3, 0, 0, S) == 7
    assert L.gbe_argmax(NULL, NULL, 0, 0, 0, S) == 0
    assert L.gbe_argmax(NULL, NULL, 3, 1 << 31, 0, S) == 2
    assert L.gbe_argmax(NULL, NULL, 3, 10, 5, S) == 3


def test_rope_qk_and_table_reject_bad_arguments(L):
    def call(T=4, D=32, r=32, layout=0, mu=1.0, dtype=0, qs=64, ks=32, hq=2, hk=1, cache=None, clen=0):
        return L.gbe_rope_qk(NULL, NULL, qs, hq, NULL, NULL, ks, hk, NULL, T, D, r, NULL, cache, clen, mu,
                             layout, dtype, S)
    assert call(layout=3) == 4
    assert call(dtype=9) == 3
    assert call(r=31) == 6 and call(r=34) == 6 and call(mu=float("nan")) == 6
    assert call(D=0) == 2 and call(T=-1) == 2 and call(hq=-1) == 2
    assert call(qs=63) == 2            # token stride shorter than Hq * D
    assert call(ks=31) == 2
    assert call(cache=1, clen=-1) == 2
    assert call(T=0) == 0              # nothing to do
    assert call(hq=0, hk=0) == 0
    assert L.gbe_rope_cos_sin(NULL, -1, 8, NULL, S) == 2
    assert L.gbe_rope_cos_sin(NULL, 10, 7, NULL, S) == 6
    assert L.gbe_rope_cos_sin(NULL, 0, 8, NULL, S) == 0
    assert L.gbe_rope_cos_sin(NULL, 10, 0, NULL, S) == 0


def test_qk_norm_rope_rejects_bad_arguments(L):
    def call(T=4, D=128, r=128, layout=0, eps=1e-6, mu=1.0, dtype=1, qs=1024, hq=8, ks=256, hk=2):
        return L.gbe_qk_norm_rope(NULL, NULL, qs, hq, NULL, NULL, NULL, ks, hk, NULL, eps, NULL, T, D, r, NULL,
                                  NULL, 0, mu, layout, dtype, S)
    assert call(layout=2) == 4 and call(dtype=5) == 3
    assert call(eps=-1.0) == 5 and call(eps=float("inf")) == 5
    assert call(D=520, qs=8 * 520, ks=2 * 520, r=520) == 2     # bf16 head rows of more than 64 chunks
    assert call(D=264, dtype=0, qs=8 * 264, ks=2 * 264, r=264) == 2   # f32: 66 chunks
    assert call(r=130) == 6 and call(r=7) == 6
    assert call(qs=1000) == 2
    assert call(T=0) == 0 and call(hq=0, hk=0) == 0


def test_sample_rejects_bad_arguments(L):
    def call(rows=4, n=100, method=1, t=1.0, k=5, p=0.5, dtype=1):
        return L.gbe_sample(NULL, NULL, NULL, rows, n, method, t, k, p, dtype, S)
    assert call(method=5) == 12 and call(method=-1) == 12
    assert call(t=0.0) == 12 and call(t=-1.0) == 12 and call(t=float("nan")) == 12 and call(t=float("inf")) == 12
    assert call(method=2, k=0) == 12 and call(method=2, k=-3) == 12
    for m in (3, 4):
        assert call(method=m, p=-0.1) == 12 and call(method=m, p=1.5) == 12 and call(method=m, p=float("nan")) == 12
    assert call(dtype=4) == 3
    assert call(n=(1 << 23) + 1) == 2 and call(rows=-1) == 2 and call(n=-1) == 2
    assert call(n=0) == 7
    assert call(rows=0) == 0 and call(rows=0, n=0) == 0


def test_rejects_size_overflow(L):
    big = 1 << 62
    assert L.gbe_silu_mul(NULL, NULL, NULL, big, 0, S) == 2
    assert L.gbe_rmsnorm(NULL, NULL, NULL, 1 << 31, 1 << 31, 1e-5, 0, S) == 2
    assert L.gbe_rope(NULL, NULL, NULL, 1 << 31, 1 << 20, 1 << 20, 2, NULL, 1.0, 0, 0, S) == 2


# Fake, never-dereferenced addresses: the overlap checks are address
# arithmetic and run before any driver call, so a layout whose outputs
# overlap is refused with GBE_ERR_ALIAS (8) on any machine; a layout that
# passes them goes on to the driver checks, which refuse these addresses
# (GBE_ERR_POINTER on a GPU machine, GBE_ERR_CUDA without a device).  No
# call below can reach a launch.
BASE, POS, FREQ = 0x7F0000000000, 0x7F1000000000, 0x7F2000000000
PASSES_OVERLAP_CHECKS = (10, 11)


def _rope_qk(L, q, qo, qs, hq, k, ko, ks, hk, T=16, D=128, dtype=1):
    return L.gbe_rope_qk(q, qo, qs, hq, k, ko, ks, hk, POS, T, D, D, FREQ, NULL, 0, 1.0, 0, dtype, S)


def _qk_norm_rope(L, q, qo, qs, hq, k, ko, ks, hk, T=16, D=128, dtype=1):
    return L.gbe_qk_norm_rope(q, qo, qs, hq, FREQ + 4096, k, ko, ks, hk, FREQ + 8192, 1e-6, POS, T, D, D, FREQ,
                              NULL, 0, 1.0, 0, dtype, S)


@pytest.mark.parametrize("call", [_rope_qk, _qk_norm_rope])
def test_strided_slice_overlap_rules(L, call):
    es, D, Hq, Hk = 2, 128, 32, 8
    stride = (Hq + 2 * Hk) * D          # one token row of a fused QKV buffer: [q | k | v]
    q, k = BASE, BASE + Hq * D * es
    out = BASE + (1 << 30)              # a second QKV buffer for out-of-place results
    qo, ko = out, out + Hq * D * es
    # q and k slices of one QKV row, in place: their rows interleave without sharing a byte
    assert call(L, q, q, stride, Hq, k, k, stride, Hk) in PASSES_OVERLAP_CHECKS
    # out of place, into the slices of another QKV buffer
    assert call(L, q, qo, stride, Hq, k, ko, stride, Hk) in PASSES_OVERLAP_CHECKS
    # k ahead of q in the row (negative distance from q to k)
    assert call(L, BASE + Hk * D * es, BASE + Hk * D * es, stride, Hq, BASE, BASE, stride, Hk) \
        in PASSES_OVERLAP_CHECKS
    # k's output shifted one element back: its first entry is q's last, in every row
    assert call(L, q, q, stride, Hq, k, k - es, stride, Hk) == 8
    # q's output shifted one element forward into k
    assert call(L, q, q + es, stride, Hq, k, k, stride, Hk) == 8
    assert call(L, q, q, stride, Hq, k, q + stride * es, stride, Hk, T=16) == 8
    # ... unless there is only one token
    assert call(L, q, q, stride, Hq, k, q + stride * es, stride, Hk, T=1) in PASSES_OVERLAP_CHECKS
    # different token strides whose extents overlap: not resolvable row by row, refused
    assert call(L, q, q, stride, Hq, k, k, stride + 8, Hk) == 8
    # an output that shares bytes with its own input without being it
    assert call(L, q, q + stride * es, stride, Hq, k, k, stride, Hk, T=4) == 8
    # an output overlapping the positions
    assert call(L, q, POS, stride, Hq, k, k, stride, Hk) == 8


def test_contiguous_overlap_rules_before_driver(L):
    n, es = 1024, 4
    a, b = BASE, BASE + n * es
    assert L.gbe_add(a, b, a, n, 0, S) in PASSES_OVERLAP_CHECKS        # y == a
    assert L.gbe_add(a, b, b, n, 0, S) in PASSES_OVERLAP_CHECKS        # y == b
    assert L.gbe_add(a, b, a + es, n, 0, S) == 8                       # shifted by one element
    assert L.gbe_add(a, b, b - es, n, 0, S) == 8
    assert L.gbe_rmsnorm(a, b, a, 4, 256, 1e-5, 0, S) in PASSES_OVERLAP_CHECKS
    assert L.gbe_rmsnorm(a, a + 768 * es, b, 4, 256, 1e-5, 0, S) in PASSES_OVERLAP_CHECKS  # w inside x: inputs may overlap
    assert L.gbe_rmsnorm(a, b - 64 * es, b - 1024 * es, 4, 256, 1e-5, 0, S) == 8  # y == x, but y holds w
    assert L.gbe_embedding(a, POS, a + (1 << 20), 4, 64, 100, NULL, 0, S) in PASSES_OVERLAP_CHECKS
    assert L.gbe_embedding(a, POS, a + 64 * es, 4, 64, 100, NULL, 0, S) == 8  # out inside the table


def test_rope_pair_rejects_bad_operands(L):
    """gbe_rope_pair checks each operand as gbe_rope_qk does; none of these
    calls reaches the driver (fake addresses, refused by the argument or the
    overlap checks)."""
    import ctypes

    from elementwise_row_rmsnorm_gb300.binding import RopeOperand

    def op(**kw):
        d = dict(x=BASE, y=BASE, stride=64, H=2, r=32, inv_freq=FREQ, mu=1.0, layout=0)
        d.update(kw)
        return RopeOperand(**d)

    def call(a, b, T=4, D=32, dtype=0):
        ref = lambda o: ctypes.cast(ctypes.byref(o), ctypes.c_void_p) if o is not None else None
        return L.gbe_rope_pair(ref(a), ref(b), POS, T, D, dtype, S)
    assert call(None, op()) == 1
    assert call(op(), op(layout=3)) == 4 and call(op(layout=-1), None) == 4
    assert call(op(), op(r=31)) == 6 and call(op(r=34), None) == 6 and call(op(), op(mu=float("inf"))) == 6
    assert call(op(), op(stride=63)) == 2 and call(op(H=-1), None) == 2
    assert call(op(), None, dtype=7) == 3
    assert call(op(), None, T=0) == 0 and call(op(H=0), op(H=0)) == 0
    second = BASE + (1 << 20)
    # two operands in place in separate buffers pass the overlap checks
    assert call(op(), op(x=second, y=second)) in PASSES_OVERLAP_CHECKS
    # the second operand writing over the first one's rows
    assert call(op(), op(x=second, y=BASE + 8)) == 8
