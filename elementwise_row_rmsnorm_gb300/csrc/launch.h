// launch.h -- internal launchers behind the C ABI (abi.cu validates every
// argument before any of these is called; they only pick a kernel variant
// and launch it on the caller's stream).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gbe {

// res == nullptr: RMSNorm; otherwise the fused residual add + RMSNorm, h = x + res.
cudaError_t launch_rmsnorm(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows,
                           int64_t d, float eps, int dtype, bool vec, cudaStream_t st);

// LayerNorm of each row with gain g and optional bias b (nullptr: none).
cudaError_t launch_layernorm(const void* x, const void* g, const void* b, void* y, int64_t rows, int64_t d,
                             float eps, int dtype, bool vec, cudaStream_t st);

// RoPE over one or two [T, H, D] operands (q and k) that share positions and
// head_dim; each operand has a token stride (elements) used for its input
// and its output, and its own rotated width, frequencies, scale and layout.
// cos_sin: NULL, or a [cache_len, r/2] table of (cos, sin), given only when
// both operands share r, inv_freq and layout.
struct RopeArgs {
    struct Side {
        const void* x;
        void* y;
        int64_t stride;
        int64_t H;
        int64_t r;
        const float* inv_freq;
        float mu;
        int layout;
    } side[2];
    const int32_t* pos;
    int64_t T, D;
    const float* cos_sin;
    int64_t cache_len;
};

cudaError_t launch_rope(const RopeArgs& a, int dtype, bool vec, cudaStream_t st);

cudaError_t launch_rope_cos_sin(float* cos_sin, int64_t len, int64_t r, const float* inv_freq, cudaStream_t st);

// Multi-axis RoPE: A <= 8 slices; slice a starts at entry off[a] and holds
// poff[a + 1] - poff[a] pairs; poff[A] is the number of rotated pairs.
constexpr int kMaxAxes = 8;
struct MultiAxis {
    int A;
    int off[kMaxAxes];
    int poff[kMaxAxes + 1];
};

cudaError_t launch_rope_multi(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D,
                              const MultiAxis& ax, const float* inv_freq, float mu, int layout, int dtype,
                              cudaStream_t st);

// QK-norm (per-head RMSNorm with a [D] gain per operand) followed by RoPE.
struct QkNormRopeArgs {
    struct Side {
        const void* x;
        void* y;
        const void* g;
        int64_t stride;
        int64_t H;
    } side[2];
    float eps;
    const int32_t* pos;
    int64_t T, D, r;
    const float* inv_freq;
    const float* cos_sin;
    int64_t cache_len;
    float mu;
    int layout;
};

cudaError_t launch_qk_norm_rope(const QkNormRopeArgs& a, int dtype, bool vec, cudaStream_t st);

cudaError_t launch_silu_mul(const void* gate, const void* up, void* y, int64_t n, int dtype, bool vec,
                            cudaStream_t st);

cudaError_t launch_add(const void* a, const void* b, void* y, int64_t n, int dtype, bool vec, cudaStream_t st);

cudaError_t launch_embedding(const void* table, const int32_t* ids, void* out, int64_t n, int64_t d, int64_t V,
                             int32_t* bad_id_count, int dtype, bool vec, cudaStream_t st);

cudaError_t launch_argmax(const void* x, int32_t* out, int64_t rows, int64_t n, int dtype, bool vec,
                          cudaStream_t st);

// The uniforms of a sampling launch: u[row] when u is given, else draw
// offset + row of the PCG64 stream seeded with `seed`.
struct Draws {
    const float* u;
    unsigned long long seed, offset;
};

cudaError_t launch_sample(const void* x, int32_t* out, int64_t rows, int64_t n, int method, float t, int64_t k,
                          float p, Draws d, int dtype, bool vec, cudaStream_t st);

// u[i] = the uniform of draw offset + i of the PCG64 stream seeded with `seed`.
cudaError_t launch_pcg64_uniforms(float* u, int64_t n, unsigned long long seed, unsigned long long offset,
                                  cudaStream_t st);

}  // namespace gbe
