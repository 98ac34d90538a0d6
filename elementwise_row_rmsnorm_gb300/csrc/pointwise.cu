// pointwise.cu -- SiLU-mul and residual add on sm_103a.
//
// SiLU-mul ("Elementwise kernels in C", section 2.3; "Operations", section 4,
// Silu and SwiGlu): y = g / (1 + e^-g) * u, silu first, then the product.
// Evaluated as g * (1 / (1 + 2^(-g log2 e))) * u with the hardware
// exponential and reciprocal (ex2.approx, rcp.approx): a few f32 roundings
// and two approximations, relative error within ~5e-6 over the f32 range
// (|g| log2 e times 2^-24 from the exponent's argument plus a few ulps),
// where an accurate expf and an IEEE division cost ~7 % of this op's time
// on GB300.  It saturates like the quotient: for g -> -inf, 2^(-g log2 e)
// overflows to +inf, its reciprocal is 0 and the product is -0 (no NaN);
// for g -> +inf the factor is 1 and the result is g.
// Add ("Operations", section 1; "Elementwise kernels in C", section 2.4):
// y = a + b, the residual connection.
//
// Both read two flat arrays of n elements and write one; y may be either
// input (exactly, not a partial overlap).  The math is f32; bf16 inputs are
// widened exactly and the result rounded to nearest-even once.
//
// Map: each thread owns U 16-byte vectors spaced one CTA-width apart (so
// every load instruction of a warp covers 512 contiguous bytes), issues all
// 2U loads before any use, then computes and stores; loads and stores carry
// the evict-first (.cs) hint, each byte being touched once.  One CTA covers
// 256 * U vectors; the last CTA also does the n mod V elements past the last
// whole vector.  U = 4 when that still gives at least two CTAs per SM, else
// U = 1 (small, decode-size arrays: more threads, each with less to do, so
// the launch fills the GPU).  Misaligned pointers take a scalar path with
// the same per-element arithmetic.
#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kThreads = 256;
constexpr int kU = 4;  // vectors per thread on large arrays

enum { kSiluMul = 0, kAdd = 1 };

__device__ __forceinline__ float ex2_approx(float a) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

__device__ __forceinline__ float rcp_approx(float a) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

template <int OP>
__device__ __forceinline__ float op1(float a, float b) {
    if (OP == kSiluMul) {
        const float e = ex2_approx(__fmul_rn(a, -1.44269502f));  // e^-g
        const float silu = __fmul_rn(a, rcp_approx(__fadd_rn(1.0f, e)));
        return __fmul_rn(silu, b);
    }
    return __fadd_rn(a, b);
}

template <int DT, int OP, int U>
__global__ void __launch_bounds__(kThreads)
pointwise_vec(const void* a, const void* b, void* y, int64_t n) {
    using S = Store<DT>;
    constexpr int V = S::V;
    pdl_begin();
    const int64_t nvec = n / V;
    const int64_t v0 = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x;
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    char* py = static_cast<char*>(y);
    Vec16 ra[U], rb[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t i = v0 + (int64_t)u * kThreads;
        if (i < nvec) {
            ra[u] = ld_once(pa + i * 16);
            rb[u] = ld_once(pb + i * 16);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t i = v0 + (int64_t)u * kThreads;
        if (i < nvec) {
            float fa[V], fb[V], fy[V];
            S::unpack(ra[u], fa);
            S::unpack(rb[u], fb);
#pragma unroll
            for (int e = 0; e < V; ++e) fy[e] = op1<OP>(fa[e], fb[e]);
            st_once(py + i * 16, S::pack(fy));
        }
    }
    if (blockIdx.x == gridDim.x - 1) {
        const int64_t tail0 = nvec * V;
        const int64_t i = tail0 + threadIdx.x;
        if (i < n) S::store1(y, i, op1<OP>(S::load1(a, i), S::load1(b, i)));
    }
}

template <int DT, int OP>
__global__ void __launch_bounds__(kThreads)
pointwise_scalar(const void* a, const void* b, void* y, int64_t n) {
    using S = Store<DT>;
    pdl_begin();
    const int64_t i0 = (int64_t)blockIdx.x * (kThreads * kU) + threadIdx.x;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int64_t i = i0 + (int64_t)u * kThreads;
        if (i < n) S::store1(y, i, op1<OP>(S::load1(a, i), S::load1(b, i)));
    }
}

template <int OP>
cudaError_t launch_pw(const void* a, const void* b, void* y, int64_t n, int dtype, bool vec, cudaStream_t st) {
    const int V = dtype == kF32 ? 4 : 8;
    const int64_t per_cta = (int64_t)kThreads * kU;
    if (vec) {
        const int64_t nvec = n / V;
        int64_t grid = (nvec + per_cta - 1) / per_cta;
        if (grid < 2 * (int64_t)sm_count()) {  // too few CTAs to fill the GPU: one vector per thread
            grid = (nvec + kThreads - 1) / kThreads;
            if (grid < 1) grid = 1;  // the tail alone (n < V) still needs one CTA
            if (dtype == kF32)
                return launch(pointwise_vec<kF32, OP, 1>, dim3((unsigned)grid), dim3(kThreads), 0, st, a, b, y, n);
            return launch(pointwise_vec<kBF16, OP, 1>, dim3((unsigned)grid), dim3(kThreads), 0, st, a, b, y, n);
        }
        if (dtype == kF32)
            return launch(pointwise_vec<kF32, OP, kU>, dim3((unsigned)grid), dim3(kThreads), 0, st, a, b, y, n);
        return launch(pointwise_vec<kBF16, OP, kU>, dim3((unsigned)grid), dim3(kThreads), 0, st, a, b, y, n);
    }
    const int64_t grid = (n + per_cta - 1) / per_cta;
    if (dtype == kF32) return launch(pointwise_scalar<kF32, OP>, dim3((unsigned)grid), dim3(kThreads), 0, st, a, b, y, n);
    return launch(pointwise_scalar<kBF16, OP>, dim3((unsigned)grid), dim3(kThreads), 0, st, a, b, y, n);
}

}  // namespace

cudaError_t launch_silu_mul(const void* gate, const void* up, void* y, int64_t n, int dtype, bool vec,
                            cudaStream_t st) {
    return launch_pw<kSiluMul>(gate, up, y, n, dtype, vec, st);
}

cudaError_t launch_add(const void* a, const void* b, void* y, int64_t n, int dtype, bool vec, cudaStream_t st) {
    return launch_pw<kAdd>(a, b, y, n, dtype, vec, st);
}

}  // namespace gbe
