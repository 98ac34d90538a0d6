"""GB300 (sm_103a) elementwise and row-wise transformer ops behind a C ABI.

RMSNorm (eps inside the root), fused residual add + RMSNorm, RoPE (half and
interleaved layouts, partial rotary width, attention scaling), SiLU-mul,
embedding gather, residual add, greedy argmax and sampling (with the
caller's uniforms or a seeded PCG64 stream) -- one hand-written CUDA
kernel each, in ``lib/libgbe_elementwise.so`` (declared in
``include/gbe_elementwise.h``).  This package is the binding: see
:mod:`elementwise_row_rmsnorm_gb300.binding`.
"""
from .binding import (GBE_BF16, GBE_F32, GbeError, LibraryMissing, add, add_rmsnorm, argmax, embedding,
                      gbe_add, gbe_add_rmsnorm, gbe_argmax, gbe_embedding, gbe_layernorm, gbe_pcg64_uniforms,
                      gbe_qk_norm_rope, gbe_rmsnorm, gbe_rope, gbe_rope_cos_sin, gbe_rope_multi, gbe_rope_pair, gbe_rope_qk,
                      gbe_sample, gbe_sample_seeded, gbe_silu_mul, layernorm, lib, pcg64_uniforms, rmsnorm, rope,
                      rope_cos_sin, sample, sample_seeded, silu_mul, status_string)


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (nvcc) if a source is newer than it."""
    from . import _build
    return _build.build(force=force)


__all__ = [
    "GBE_BF16", "GBE_F32", "GbeError", "LibraryMissing", "add", "add_rmsnorm", "argmax", "build",
    "embedding", "gbe_add", "gbe_add_rmsnorm", "gbe_argmax", "gbe_embedding", "gbe_layernorm",
    "gbe_pcg64_uniforms", "gbe_qk_norm_rope", "gbe_rmsnorm", "gbe_rope", "gbe_rope_cos_sin", "gbe_rope_multi", "gbe_rope_pair",
    "gbe_rope_qk", "gbe_sample", "gbe_sample_seeded", "gbe_silu_mul", "layernorm", "lib", "pcg64_uniforms",
    "rmsnorm", "rope", "rope_cos_sin", "sample", "sample_seeded", "silu_mul", "status_string",
]
