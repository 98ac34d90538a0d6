"""Helpers of the GPU parity tests: moving generated arrays to the device,
reading results back in the oracle's terms, and the comparison rules.

Comparison rules (the bar the tests hold the CUDA path to):
  * argmax, embedding, add, the h output of add+RMSNorm, RoPE pass-through
    entries and the position-0 identity: bit equality;
  * RMSNorm y and SiLU-mul: |y - y_oracle| <= rtol * |y_oracle| (+1e-30 so
    that -0 against a value below 1e-30 at the exp overflow edge passes);
  * RoPE: per pair, |y - y_oracle| <= rtol * mu * |(a, b)|, since
    a cos - b sin can cancel to nearly zero;
  * rtol = 1e-5 for f32 and 1e-2 for bf16, the bf16 result (rounded once)
    against the oracle's unrounded f32 result.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

RTOL = {"f32": 1e-5, "bf16": 1e-2}
DEV = "cuda"


def to_dev(a: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a).to(DEV)


def to_f32(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> f32 numpy (bf16 widened exactly by the oracle's own rule)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return oracle.get().bf16_widen(t.view(torch.int16).numpy().view(np.uint16))
    return t.numpy().astype(np.float32, copy=False)


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.numpy()


def widen(a: np.ndarray) -> np.ndarray:
    """Generated input -> the f32 values the oracle computes on."""
    return oracle.get().bf16_widen(a) if a.dtype == np.uint16 else a


def assert_rel(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad_nan = np.isnan(got) != np.isnan(want)
    assert not bad_nan.any(), f"{what}: NaN mismatch at {np.argwhere(bad_nan)[:5]}"
    ok = np.isnan(want) | (np.abs(got - want) <= RTOL[dtype] * np.abs(want) + 1e-30)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        ratio = np.nanmax(np.abs(got - want) / np.maximum(np.abs(want), 1e-30))
        raise AssertionError(f"{what}: {int((~ok).sum())} entries off (max rel {ratio:.3g}); "
                             f"first at {idx.tolist()}: got {got[tuple(idx[0])]}, want {want[tuple(idx[0])]}")


def assert_bf16_within_ulp(got_bits: np.ndarray, want_f32: np.ndarray, what: str = ""):
    """The bf16 result lies within one bf16 step of the oracle's f32 result rounded."""
    ref = oracle.get().bf16_round(want_f32).astype(np.int32)
    g = got_bits.astype(np.int32)
    # same sign and magnitude order: bf16 bit patterns of one sign are monotone
    diff = np.abs(g - ref)
    finite = np.isfinite(want_f32)
    assert np.all(diff[finite] <= 1), f"{what}: {int((diff[finite] > 1).sum())} bf16 results beyond 1 ulp"


def assert_rope_close(got: np.ndarray, want: np.ndarray, x: np.ndarray, r: int, mu: float, layout: int,
                      dtype: str, what: str = ""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    x = np.asarray(x, np.float64)
    i = np.arange(r // 2)
    ia, ib = (i, i + r // 2) if layout == 0 else (2 * i, 2 * i + 1)
    norm = np.hypot(x[..., ia], x[..., ib])
    tol = RTOL[dtype] * abs(mu) * norm + 1e-30
    for idx in (ia, ib):
        err = np.abs(got[..., idx] - want[..., idx])
        if not np.all(err <= tol):
            k = np.argwhere(err > tol)[0]
            raise AssertionError(f"{what}: rotated entry off at {k.tolist()} "
                                 f"({err[tuple(k)]:.3g} > {tol[tuple(k)]:.3g})")
