"""Python binding of the C ABI (include/gbe_elementwise.h).

Argument marshalling only: each ``gbe_*`` function takes torch tensors that
live on the current CUDA device (or in pinned host memory, which the kernels
then read and write in place over the host link), checks that their shapes and dtypes
agree with one another, and passes their pointers, sizes and the current
stream to the C entry point of the same name.  Every step of every op runs
in the CUDA library; there is no other code path.  If the library is not
built, the first call raises :class:`LibraryMissing`.

The functions without the ``gbe_`` prefix (``rmsnorm``, ``rope``, ...) are
conveniences that allocate the outputs with torch and call the ``gbe_``
function.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libgbe_elementwise.so")

GBE_F32, GBE_BF16 = 0, 1
_DTYPES = {torch.float32: GBE_F32, torch.bfloat16: GBE_BF16}

_lib = None
_lock = threading.Lock()


class LibraryMissing(RuntimeError):
    pass


class GbeError(RuntimeError):
    def __init__(self, op: str, status: int, message: str, cuda_error: int = 0):
        super().__init__(f"{op}: status {status} ({message})"
                         + (f", cudaError {cuda_error}" if cuda_error else ""))
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded C library (raises LibraryMissing when it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryMissing(
                    f"{LIB_PATH} is not built; run elementwise_row_rmsnorm_gb300.build() "
                    "(nvcc, sm_103a) first")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
            u64 = ctypes.c_uint64
            sigs = {
                "gbe_rmsnorm": [vp, vp, vp, i64, i64, f32, i32, vp],
                "gbe_add_rmsnorm": [vp, vp, vp, vp, vp, i64, i64, f32, i32, vp],
                "gbe_layernorm": [vp, vp, vp, vp, i64, i64, f32, i32, vp],
                "gbe_rope": [vp, vp, vp, i64, i64, i64, i64, vp, f32, i32, i32, vp],
                "gbe_rope_qk": [vp, vp, i64, i64, vp, vp, i64, i64, vp, i64, i64, i64, vp, vp, i64, f32, i32,
                                i32, vp],
                "gbe_rope_cos_sin": [vp, i64, i64, vp, vp],
                "gbe_rope_pair": [vp, vp, vp, i64, i64, i32, vp],
                "gbe_rope_multi": [vp, vp, vp, i64, i64, i64, i64, vp, vp, f32, i32, i32, vp],
                "gbe_qk_norm_rope": [vp, vp, i64, i64, vp, vp, vp, i64, i64, vp, f32, vp, i64, i64, i64, vp, vp,
                                     i64, f32, i32, i32, vp],
                "gbe_silu_mul": [vp, vp, vp, i64, i32, vp],
                "gbe_add": [vp, vp, vp, i64, i32, vp],
                "gbe_embedding": [vp, vp, vp, i64, i64, i64, vp, i32, vp],
                "gbe_argmax": [vp, vp, i64, i64, i32, vp],
                "gbe_sample": [vp, vp, vp, i64, i64, i32, f32, i64, f32, i32, vp],
                "gbe_sample_seeded": [vp, vp, i64, i64, i32, f32, i64, f32, u64, u64, i32, vp],
                "gbe_pcg64_uniforms": [vp, i64, u64, u64, vp],
                "gbe_version": [],
                "gbe_last_cuda_error": [],
                "gbe_status_string": [i32],
            }
            for name, args in sigs.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_char_p if name == "gbe_status_string" else ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gbe_status_string(status).decode()


def _check(op: str, st: int):
    if st != 0:
        L = lib()
        raise GbeError(op, st, status_string(st), L.gbe_last_cuda_error() if st == 11 else 0)


# The current stream's handle without building a torch Stream object per
# call (the private accessors torch's own extensions use; the public path
# where they are absent).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None and _cur_device is not None:
            return _raw_stream(_cur_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dt(*ts) -> int:
    dt = ts[0].dtype
    for t in ts:
        if t.dtype != dt:
            raise TypeError(f"all float tensors of one call share a dtype ({dt} vs {t.dtype})")
    if dt not in _DTYPES:
        raise TypeError(f"unsupported dtype {dt} (float32 or bfloat16)")
    return _DTYPES[dt]


def _on_device(t) -> bool:
    """CUDA tensors, and pinned host tensors (mapped at the same address on the
    device, so kernels read and write them in place: zero-copy)."""
    return t.is_cuda or t.is_pinned()


def _dev(*ts):
    for t in ts:
        if not _on_device(t):
            raise ValueError("tensors must be on the CUDA device or in pinned host memory")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


# ---- the C entry points, one to one -----------------------------------------------

def gbe_rmsnorm(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, eps: float, stream=None) -> None:
    _dev(x, w, y)
    d = x.shape[-1]
    if y.shape != x.shape or w.numel() != d:
        raise ValueError("rmsnorm: y must match x and w must have x.shape[-1] entries")
    _check("gbe_rmsnorm", lib().gbe_rmsnorm(_ptr(x), _ptr(w), _ptr(y), x.numel() // d if d else 0, d,
                                            eps, _dt(x, w, y), _stream(stream)))


def gbe_layernorm(x, g, b, y, eps: float, stream=None) -> None:
    """b may be None (no bias)."""
    _dev(*[t for t in (x, g, b, y) if t is not None])
    d = x.shape[-1]
    if y.shape != x.shape or g.numel() != d or (b is not None and b.numel() != d):
        raise ValueError("layernorm: y matches x; g and b have x.shape[-1] entries")
    floats = [t for t in (x, g, b, y) if t is not None]
    _check("gbe_layernorm", lib().gbe_layernorm(_ptr(x), _ptr(g), _ptr(b), _ptr(y), x.numel() // d if d else 0, d,
                                                eps, _dt(*floats), _stream(stream)))


def gbe_add_rmsnorm(x, residual, w, y, h, eps: float, stream=None) -> None:
    _dev(x, residual, w, y, h)
    d = x.shape[-1]
    if not (residual.shape == y.shape == h.shape == x.shape) or w.numel() != d:
        raise ValueError("add_rmsnorm: x, residual, y, h must share a shape; w has x.shape[-1] entries")
    _check("gbe_add_rmsnorm", lib().gbe_add_rmsnorm(
        _ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(h), x.numel() // d if d else 0, d, eps,
        _dt(x, residual, w, y, h), _stream(stream)))


def gbe_rope(x, y, pos, inv_freq, r: int, mu: float = 1.0, layout: int = 0, stream=None) -> None:
    _dev(x, y, pos, inv_freq)
    if x.dim() != 3 or y.shape != x.shape:
        raise ValueError("rope: x is [T, H, D] and y matches it")
    T, H, D = x.shape
    if pos.dtype != torch.int32 or pos.numel() != T:
        raise ValueError("rope: pos is int32[T]")
    if inv_freq.dtype != torch.float32 or inv_freq.numel() < r // 2:
        raise ValueError("rope: inv_freq is float32[r/2]")
    _check("gbe_rope", lib().gbe_rope(_ptr(x), _ptr(y), _ptr(pos), T, H, D, r, _ptr(inv_freq), mu, layout,
                                      _dt(x, y), _stream(stream)))


def _rows_view(t: torch.Tensor, D: int):
    """(T, H, token stride) of a [T, H, D] view whose heads and entries are
    contiguous but whose tokens may be strided (a slice of a QKV buffer)."""
    shape, st = t.shape, t.stride()  # one query each (the per-call host cost matters at decode sizes)
    if len(shape) != 3 or shape[2] != D or st[2] != 1 or (shape[1] > 1 and st[1] != D):
        raise ValueError("rope_qk: operands are [T, H, D] views with contiguous heads")
    return shape[0], shape[1], st[0] if shape[0] > 1 else shape[1] * D


def gbe_rope_qk(q, q_out, k, k_out, pos, inv_freq, r: int, mu: float = 1.0, layout: int = 0,
                cos_sin=None, stream=None) -> None:
    """q, k (and their outputs, which may be the same views): [T, H, D] views
    of one storage type whose token stride may exceed H * D."""
    ts = [t for t in (q, q_out, k, k_out, pos, inv_freq) if t is not None]
    for t in ts:
        if not _on_device(t):
            raise ValueError("tensors must be on the CUDA device or in pinned host memory")
    D = (q if q is not None else k).shape[2]
    T = (q if q is not None else k).shape[0]
    sides = []
    for x, y in ((q, q_out), (k, k_out)):
        if x is None:
            sides.append((None, None, 0, 0))
            continue
        Tx, H, sx = _rows_view(x, D)
        _, _, sy = _rows_view(y, D)
        if Tx != T or y.shape != x.shape or sx != sy:
            raise ValueError("rope_qk: an output has its input's shape and token stride")
        sides.append((x.data_ptr(), y.data_ptr(), sx, H))
    if pos.dtype != torch.int32 or pos.numel() != T or not pos.is_contiguous():
        raise ValueError("rope_qk: pos is int32[T]")
    if inv_freq.dtype != torch.float32 or inv_freq.numel() < r // 2:
        raise ValueError("rope_qk: inv_freq is float32[r/2]")
    cache_len = 0
    if cos_sin is not None:
        if cos_sin.dtype != torch.float32 or not cos_sin.is_contiguous() or (r and cos_sin.numel() % r):
            raise ValueError("rope_qk: cos_sin is float32[cache_len, r/2, 2]")
        cache_len = cos_sin.numel() // r if r else 0
    floats = [t for t in (q, q_out, k, k_out) if t is not None]
    (qx, qy, qs, hq), (kx, ky, ks, hk) = sides
    _check("gbe_rope_qk", lib().gbe_rope_qk(qx, qy, qs, hq, kx, ky, ks, hk, _ptr(pos), T, D, r, _ptr(inv_freq),
                                            _ptr(cos_sin), cache_len, mu, layout, _dt(*floats), _stream(stream)))


class RopeOperand(ctypes.Structure):
    """gbe_rope_operand of the C header."""
    _fields_ = [("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("stride", ctypes.c_int64), ("H", ctypes.c_int64),
                ("r", ctypes.c_int64), ("inv_freq", ctypes.c_void_p), ("mu", ctypes.c_float), ("layout", ctypes.c_int)]


def gbe_rope_pair(a, b, pos, stream=None) -> None:
    """RoPE of two operands in one launch.  a and b (b may be None) are
    tuples (x, y, inv_freq, r, mu, layout): x and y [T, H, D] views with
    contiguous heads whose token stride may exceed H * D (y is x: in place),
    inv_freq float32[r/2]; the operands share pos (int32[T]), T, D and dtype."""
    ops, floats = [], []
    T = D = None
    for o in (a, b):
        if o is None:
            ops.append(None)
            continue
        x, y, inv_freq, r, mu, layout = o
        for t in (x, y, inv_freq):
            if not _on_device(t):
                raise ValueError("tensors must be on the CUDA device or in pinned host memory")
        D = x.shape[2] if D is None else D
        Tx, H, sx = _rows_view(x, D)
        _, _, sy = _rows_view(y, D)
        T = Tx if T is None else T
        if Tx != T or y.shape != x.shape or sx != sy:
            raise ValueError("rope_pair: the operands share T and D; an output has its input's shape and stride")
        if inv_freq.dtype != torch.float32 or inv_freq.numel() < r // 2 or not inv_freq.is_contiguous():
            raise ValueError("rope_pair: inv_freq is float32[r/2]")
        ops.append(RopeOperand(x.data_ptr(), y.data_ptr(), sx, H, r, inv_freq.data_ptr(), mu, layout))
        floats += [x, y]
    if ops[0] is None:
        raise ValueError("rope_pair: the first operand is required")
    if pos.dtype != torch.int32 or pos.numel() != T or not pos.is_contiguous() or not _on_device(pos):
        raise ValueError("rope_pair: pos is int32[T]")
    pa = ctypes.byref(ops[0])
    pb = ctypes.byref(ops[1]) if ops[1] is not None else None
    _check("gbe_rope_pair", lib().gbe_rope_pair(ctypes.cast(pa, ctypes.c_void_p), ctypes.cast(pb, ctypes.c_void_p)
                                                if pb is not None else None, _ptr(pos), T, D, _dt(*floats),
                                                _stream(stream)))


def gbe_qk_norm_rope(q, q_out, gq, k, k_out, gk, eps: float, pos, inv_freq, r: int, mu: float = 1.0,
                     layout: int = 0, cos_sin=None, stream=None) -> None:
    """QK-norm (per-head RMSNorm with gains gq / gk of head_dim entries), then
    RoPE; q, k and outputs as for gbe_rope_qk."""
    for t in (q, q_out, k, k_out, gq, gk, pos, inv_freq, cos_sin):
        if t is not None and not _on_device(t):
            raise ValueError("tensors must be on the CUDA device or in pinned host memory")
    ref = q if q is not None else k
    T, D = ref.shape[0], ref.shape[2]
    sides = []
    for x, y, g in ((q, q_out, gq), (k, k_out, gk)):
        if x is None:
            sides.append((None, None, None, 0, 0))
            continue
        Tx, H, sx = _rows_view(x, D)
        _, _, sy = _rows_view(y, D)
        if Tx != T or y.shape != x.shape or sx != sy:
            raise ValueError("qk_norm_rope: an output has its input's shape and token stride")
        if g is None or g.numel() != D or not g.is_contiguous() or g.dtype != x.dtype:
            raise ValueError("qk_norm_rope: each gain has head_dim entries of the operand's dtype")
        sides.append((x.data_ptr(), y.data_ptr(), g.data_ptr(), sx, H))
    if pos.dtype != torch.int32 or pos.numel() != T or not pos.is_contiguous():
        raise ValueError("qk_norm_rope: pos is int32[T]")
    if inv_freq.dtype != torch.float32 or inv_freq.numel() < r // 2:
        raise ValueError("qk_norm_rope: inv_freq is float32[r/2]")
    cache_len = 0
    if cos_sin is not None:
        if cos_sin.dtype != torch.float32 or not cos_sin.is_contiguous() or (r and cos_sin.numel() % r):
            raise ValueError("qk_norm_rope: cos_sin is float32[cache_len, r/2, 2]")
        cache_len = cos_sin.numel() // r if r else 0
    floats = [t for t in (q, q_out, k, k_out, gq, gk) if t is not None]
    (qx, qy, qg, qs, hq), (kx, ky, kg, ks, hk) = sides
    _check("gbe_qk_norm_rope", lib().gbe_qk_norm_rope(qx, qy, qs, hq, qg, kx, ky, ks, hk, kg, eps, _ptr(pos), T, D,
                                                      r, _ptr(inv_freq), _ptr(cos_sin), cache_len, mu, layout,
                                                      _dt(*floats), _stream(stream)))


def gbe_rope_multi(x, y, pos, dims, inv_freq, mu: float = 1.0, layout: int = 0, stream=None) -> None:
    """x, y: [T, H, D]; pos: int32 [T, A]; dims: A even slice widths (a host
    sequence); inv_freq: float32, the axes' frequencies concatenated."""
    _dev(x, y, pos, inv_freq)
    if x.dim() != 3 or y.shape != x.shape:
        raise ValueError("rope_multi: x is [T, H, D] and y matches it")
    T, H, D = x.shape
    dims_arr = (ctypes.c_int64 * max(1, len(dims)))(*[int(v) for v in dims])
    A = len(dims)
    if pos.dtype != torch.int32 or pos.numel() != T * A:
        raise ValueError("rope_multi: pos is int32[T, A]")
    if inv_freq.dtype != torch.float32 or inv_freq.numel() < sum(int(v) for v in dims) // 2:
        raise ValueError("rope_multi: inv_freq holds sum(dims)/2 float32 entries")
    _check("gbe_rope_multi", lib().gbe_rope_multi(_ptr(x), _ptr(y), _ptr(pos), T, H, D, A,
                                                  ctypes.cast(dims_arr, ctypes.c_void_p), _ptr(inv_freq), mu, layout,
                                                  _dt(x, y), _stream(stream)))


def gbe_rope_cos_sin(cos_sin, inv_freq, r: int, stream=None) -> None:
    _dev(cos_sin, inv_freq)
    if cos_sin.dtype != torch.float32 or (r and cos_sin.numel() % r) or inv_freq.dtype != torch.float32:
        raise ValueError("rope_cos_sin: cos_sin is float32[cache_len, r/2, 2], inv_freq float32[r/2]")
    cache_len = cos_sin.numel() // r if r else 0
    _check("gbe_rope_cos_sin", lib().gbe_rope_cos_sin(_ptr(cos_sin), cache_len, r, _ptr(inv_freq),
                                                      _stream(stream)))


def gbe_silu_mul(gate, up, y, stream=None) -> None:
    _dev(gate, up, y)
    if not (gate.shape == up.shape == y.shape):
        raise ValueError("silu_mul: gate, up, y must share a shape")
    _check("gbe_silu_mul", lib().gbe_silu_mul(_ptr(gate), _ptr(up), _ptr(y), gate.numel(),
                                              _dt(gate, up, y), _stream(stream)))


def gbe_add(a, b, y, stream=None) -> None:
    _dev(a, b, y)
    if not (a.shape == b.shape == y.shape):
        raise ValueError("add: a, b, y must share a shape")
    _check("gbe_add", lib().gbe_add(_ptr(a), _ptr(b), _ptr(y), a.numel(), _dt(a, b, y), _stream(stream)))


def gbe_embedding(table, ids, out, bad_id_count=None, stream=None) -> None:
    _dev(table, ids, out)
    if bad_id_count is not None:
        _dev(bad_id_count)
        if bad_id_count.dtype != torch.int32 or bad_id_count.numel() != 1:
            raise ValueError("embedding: bad_id_count is one int32")
    if table.dim() != 2 or ids.dtype != torch.int32:
        raise ValueError("embedding: table is [V, d], ids int32")
    V, d = table.shape
    if out.shape != (ids.numel(), d):
        raise ValueError("embedding: out is [n, d]")
    _check("gbe_embedding", lib().gbe_embedding(_ptr(table), _ptr(ids), _ptr(out), ids.numel(), d, V,
                                                _ptr(bad_id_count), _dt(table, out), _stream(stream)))


def gbe_argmax(x, out, stream=None) -> None:
    _dev(x, out)
    n = x.shape[-1]
    rows = math.prod(x.shape[:-1])
    if out.dtype != torch.int32 or out.numel() != rows:
        raise ValueError("argmax: out is int32 with one entry per row")
    _check("gbe_argmax", lib().gbe_argmax(_ptr(x), _ptr(out), rows, n, _dt(x), _stream(stream)))


SAMPLE_METHODS = {"greedy": 0, "temperature": 1, "top_k": 2, "top_p": 3, "min_p": 4}


def gbe_sample(x, u, out, method: str, temperature: float = 1.0, top_k: int = 1, p: float = 1.0,
               stream=None) -> None:
    """One draw per row of x [..., n] at the uniforms u (f32, one per row);
    `p` is top-p's mass or min-p's ratio.  u may be None for greedy."""
    if method not in SAMPLE_METHODS:
        raise ValueError(f"sample: method is one of {sorted(SAMPLE_METHODS)}")
    _dev(x, out)
    n = x.shape[-1]
    rows = math.prod(x.shape[:-1])
    if out.dtype != torch.int32 or out.numel() != rows:
        raise ValueError("sample: out is int32 with one entry per row")
    if u is not None:
        _dev(u)
        if u.dtype != torch.float32 or u.numel() != rows:
            raise ValueError("sample: u is float32 with one entry per row")
    _check("gbe_sample", lib().gbe_sample(_ptr(x), None if u is None else _ptr(u), _ptr(out), rows, n,
                                          SAMPLE_METHODS[method], temperature, top_k, p, _dt(x),
                                          _stream(stream)))


def gbe_sample_seeded(x, out, method: str, seed: int, offset: int = 0, temperature: float = 1.0, top_k: int = 1,
                      p: float = 1.0, stream=None) -> None:
    """One draw per row of x [..., n]; row r draws with the uniform of draw
    offset + r of the PCG64 stream seeded with `seed` (0 <= seed, offset < 2^64)."""
    if method not in SAMPLE_METHODS:
        raise ValueError(f"sample: method is one of {sorted(SAMPLE_METHODS)}")
    _dev(x, out)
    n = x.shape[-1]
    rows = math.prod(x.shape[:-1])
    if out.dtype != torch.int32 or out.numel() != rows:
        raise ValueError("sample: out is int32 with one entry per row")
    if not (0 <= seed < 1 << 64 and 0 <= offset < 1 << 64):
        raise ValueError("sample: seed and offset are unsigned 64-bit integers")
    _check("gbe_sample_seeded", lib().gbe_sample_seeded(_ptr(x), _ptr(out), rows, n, SAMPLE_METHODS[method],
                                                        temperature, top_k, p, seed, offset, _dt(x),
                                                        _stream(stream)))


def gbe_pcg64_uniforms(u, seed: int, offset: int = 0, stream=None) -> None:
    """u (float32, any shape) <- the uniforms of draws offset .. offset + u.numel() - 1."""
    _dev(u)
    if u.dtype != torch.float32:
        raise ValueError("pcg64_uniforms: u is float32")
    if not (0 <= seed < 1 << 64 and 0 <= offset < 1 << 64):
        raise ValueError("pcg64_uniforms: seed and offset are unsigned 64-bit integers")
    _check("gbe_pcg64_uniforms", lib().gbe_pcg64_uniforms(_ptr(u), u.numel(), seed, offset, _stream(stream)))


# ---- conveniences that allocate the outputs -------------------------------------------

def rmsnorm(x, w, eps: float = 1e-5, out=None, stream=None):
    y = torch.empty_like(x) if out is None else out
    gbe_rmsnorm(x, w, y, eps, stream)
    return y


def layernorm(x, g, b=None, eps: float = 1e-5, stream=None):
    y = torch.empty_like(x)
    gbe_layernorm(x, g, b, y, eps, stream)
    return y


def add_rmsnorm(x, residual, w, eps: float = 1e-5, stream=None):
    y, h = torch.empty_like(x), torch.empty_like(x)
    gbe_add_rmsnorm(x, residual, w, y, h, eps, stream)
    return y, h


def rope(x, pos, inv_freq, r: int, mu: float = 1.0, layout: int = 0, in_place: bool = False, stream=None):
    y = x if in_place else torch.empty_like(x)
    gbe_rope(x, y, pos, inv_freq, r, mu, layout, stream)
    return y


def rope_cos_sin(inv_freq, r: int, cache_len: int, stream=None):
    t = torch.empty((cache_len, r // 2, 2), dtype=torch.float32, device=inv_freq.device)
    gbe_rope_cos_sin(t, inv_freq, r, stream)
    return t


def silu_mul(gate, up, stream=None):
    y = torch.empty_like(gate)
    gbe_silu_mul(gate, up, y, stream)
    return y


def add(a, b, stream=None):
    y = torch.empty_like(a)
    gbe_add(a, b, y, stream)
    return y


def embedding(table, ids, bad_id_count=None, stream=None):
    out = torch.empty((ids.numel(), table.shape[1]), dtype=table.dtype, device=table.device)
    gbe_embedding(table, ids, out, bad_id_count, stream)
    return out


def argmax(x, stream=None):
    out = torch.empty(x.shape[:-1], dtype=torch.int32, device=x.device)
    gbe_argmax(x, out, stream)
    return out


def sample_seeded(x, method: str, seed: int, offset: int = 0, temperature: float = 1.0, top_k: int = 1,
                  p: float = 1.0, stream=None):
    out = torch.empty(x.shape[:-1], dtype=torch.int32, device=x.device)
    gbe_sample_seeded(x, out, method, seed, offset, temperature, top_k, p, stream)
    return out


def pcg64_uniforms(n: int, seed: int, offset: int = 0, device="cuda", stream=None):
    u = torch.empty(n, dtype=torch.float32, device=device)
    gbe_pcg64_uniforms(u, seed, offset, stream)
    return u


def sample(x, u, method: str, temperature: float = 1.0, top_k: int = 1, p: float = 1.0, stream=None):
    out = torch.empty(x.shape[:-1], dtype=torch.int32, device=x.device)
    gbe_sample(x, u, out, method, temperature, top_k, p, stream)
    return out
