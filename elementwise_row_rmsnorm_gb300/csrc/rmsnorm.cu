// rmsnorm.cu -- RMSNorm and fused residual add + RMSNorm on sm_103a.
//
// Definition ("Elementwise kernels in C", section 2.1; "Operations",
// section 2, RmsNorm): y_i = x_i / sqrt(mean_j(x_j^2) + eps) * w_i over each
// row of d entries, eps inside the root.  The fused form ("Operations",
// section 10, FusedSkipNorm) first forms h = x + residual, stores h in the
// storage type, and normalises the stored h, so it equals the unfused
// add-then-norm composition bit for bit.
//
// Layout in HBM: x, residual, y, h are [rows, d] row-major and contiguous;
// w is [d].  All are the same storage type (f32 or bf16); the math is f32.
//
// Work map.  A row is cut into chunks of one 16-byte vector (4 f32 or 8
// bf16).  Chunk c belongs to thread (c mod TPR) of the row's TPR threads, as
// that thread's (c div TPR)-th slot.  TPR and the slot count depend only on
// (d, storage type).  A thread sums the squares of its chunks in slot order
// and element order (fused multiply-add), the row's threads are combined by
// a butterfly within each warp and then warp by warp in warp order.  So the
// summation tree of a row is fixed by (d, type): the row's output bits do
// not depend on how many rows the call holds or where the row sits.  The
// aligned (vector) and unaligned (scalar) paths use the same map and the
// same operation order, so they agree bit for bit too.
//
// The whole row stays in registers between the sum and the write (one HBM
// read of x, one write of y), the 16-byte loads of all slots are issued
// before any is used, and the row's sum is complete before the first write,
// so y may be x (and h may be residual).
#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kMaxSlots = 4;  // more slots of 1024 threads would spill: such rows take the two-pass kernel

template <int DT, bool VEC>
__device__ __forceinline__ void load_chunk(const void* p, int64_t e0, int d_left, float (&f)[Store<DT>::V],
                                           Vec16& raw) {
    using S = Store<DT>;
    if (VEC) {
        raw = ld_stream(static_cast<const char*>(p) + e0 * (int64_t)sizeof(typename S::T));
    } else {
#pragma unroll
        for (int e = 0; e < S::V; ++e) f[e] = e < d_left ? S::load1(p, e0 + e) : 0.0f;
    }
}

template <int DT, int K, bool VEC, bool ADD, int MAXT>
__global__ void __launch_bounds__(MAXT)
rmsnorm_rows(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows, int d, float eps,
             int tpr) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    const int rpc = blockDim.x / tpr;
    const int sub = threadIdx.x / tpr;
    const int t = threadIdx.x - sub * tpr;
    const int64_t row = (int64_t)blockIdx.x * rpc + sub;
    if (row >= rows) return;  // only when several one-warp rows share a CTA: no CTA barrier follows
    const int nchunks = (d + V - 1) / V;
    const int64_t base = row * (int64_t)d;
    __shared__ float red[32];

    float v[K][V];
    Vec16 rx[K], rr[K];
    // 1) every load of the row's slots in flight before any use
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            load_chunk<DT, VEC>(x, base + (int64_t)c * V, d - c * V, v[k], rx[k]);
            if (ADD) {
                float vr[V];
                load_chunk<DT, VEC>(res, base + (int64_t)c * V, d - c * V, vr, rr[k]);
                if (!VEC) {
#pragma unroll
                    for (int e = 0; e < V; ++e) v[k][e] = S::round(__fadd_rn(v[k][e], vr[e]));
                }
            }
        }
    }
    // 2) widen (vector path), form h = x + residual in the storage type, square-sum
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            if (VEC) {
                S::unpack(rx[k], v[k]);
                if (ADD) {
                    float vr[V];
                    S::unpack(rr[k], vr);
#pragma unroll
                    for (int e = 0; e < V; ++e) v[k][e] = S::round(__fadd_rn(v[k][e], vr[e]));
                    st_stream(static_cast<char*>(h) + (base + (int64_t)c * V) * ES, S::pack(v[k]));
                }
            } else if (ADD) {
                for (int e = 0; e < V && c * V + e < d; ++e) S::store1(h, base + (int64_t)c * V + e, v[k][e]);
            }
#pragma unroll
            for (int e = 0; e < V; ++e) s = __fmaf_rn(v[k][e], v[k][e], s);
        }
    }
    // 3) the row's sum, fixed order
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float total = rpc > 1 ? warp_sum(s) : row_sum(s, red, warp, lane, tpr >> 5);
    const float ms = __fdiv_rn(total, (float)d);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    // 4) y = x * inv * w
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            float wv[V];
            if (VEC) {
                S::unpack(ld_reuse(static_cast<const char*>(w) + (int64_t)c * V * ES), wv);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) wv[e] = c * V + e < d ? S::load1(w, (int64_t)c * V + e) : 0.0f;
            }
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e) o[e] = __fmul_rn(__fmul_rn(v[k][e], inv), wv[e]);
            if (VEC) {
                st_stream(static_cast<char*>(y) + (base + (int64_t)c * V) * ES, S::pack(o));
            } else {
                for (int e = 0; e < V && c * V + e < d; ++e) S::store1(y, base + (int64_t)c * V + e, o[e]);
            }
        }
    }
}

// Rows wider than the register map holds (more than 4 slots of 1024
// threads: over 16384 f32 or 32768 bf16 entries): the same chunk map and sum order, with x (or h) read twice.
template <int DT, bool ADD>
__global__ void __launch_bounds__(1024)
rmsnorm_wide_rows(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows, int d,
                  float eps) {
    using S = Store<DT>;
    constexpr int V = S::V;
    const int tpr = blockDim.x;
    const int t = threadIdx.x;
    const int64_t row = blockIdx.x;
    const int nchunks = (d + V - 1) / V;
    const int64_t base = row * (int64_t)d;
    __shared__ float red[32];
    const void* src = ADD ? h : x;
    float s = 0.0f;
    for (int c = t; c < nchunks; c += tpr) {
        for (int e = 0; e < V; ++e) {
            const int64_t i = (int64_t)c * V + e;
            float a = e + c * V < d ? S::load1(x, base + i) : 0.0f;
            if (ADD && e + c * V < d) {
                a = S::round(__fadd_rn(a, S::load1(res, base + i)));
                S::store1(h, base + i, a);
            }
            s = __fmaf_rn(a, a, s);
        }
    }
    const float total = row_sum(s, red, t >> 5, t & 31, tpr >> 5);
    const float ms = __fdiv_rn(total, (float)d);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    for (int c = t; c < nchunks; c += tpr) {
        for (int e = 0; e < V && c * V + e < d; ++e) {
            const int64_t i = (int64_t)c * V + e;
            S::store1(y, base + i, __fmul_rn(__fmul_rn(S::load1(src, base + i), inv), S::load1(w, i)));
        }
    }
}

template <int DT, bool ADD>
cudaError_t launch_dt(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows, int64_t d,
                      float eps, bool vec, cudaStream_t st) {
    constexpr int V = Store<DT>::V;
    const int64_t nchunks = (d + V - 1) / V;
    int64_t tpr = ((nchunks + 3) / 4 + 31) / 32 * 32;
    if (tpr < 32) tpr = 32;
    if (tpr > 1024) tpr = 1024;
    const int64_t slots = (nchunks + tpr - 1) / tpr;
    if (slots > kMaxSlots) {
        rmsnorm_wide_rows<DT, ADD><<<(unsigned)rows, 1024, 0, st>>>(x, res, w, y, h, rows, (int)d, eps);
        return cudaGetLastError();
    }
    const int rpc = tpr == 32 ? 4 : 1;
    const int64_t grid = (rows + rpc - 1) / rpc;
    const dim3 block((unsigned)(tpr * rpc));
    const int di = (int)d, ti = (int)tpr;
#define GBE_RMS_CASE(KK, MT)                                                                          \
    if (slots <= KK) {                                                                                \
        if (vec)                                                                                      \
            rmsnorm_rows<DT, KK, true, ADD, MT><<<(unsigned)grid, block, 0, st>>>(x, res, w, y, h, rows, di, eps, ti);  \
        else                                                                                          \
            rmsnorm_rows<DT, KK, false, ADD, MT><<<(unsigned)grid, block, 0, st>>>(x, res, w, y, h, rows, di, eps, ti); \
        return cudaGetLastError();                                                                    \
    }
    if (tpr * rpc <= 256) {
        GBE_RMS_CASE(1, 256)
        GBE_RMS_CASE(2, 256)
        GBE_RMS_CASE(4, 256)
    } else {
        GBE_RMS_CASE(4, 1024)
    }
#undef GBE_RMS_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_rmsnorm(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows, int64_t d,
                           float eps, int dtype, bool vec, cudaStream_t st) {
    const bool add = res != nullptr;
    if (dtype == kF32)
        return add ? launch_dt<kF32, true>(x, res, w, y, h, rows, d, eps, vec, st)
                   : launch_dt<kF32, false>(x, res, w, y, h, rows, d, eps, vec, st);
    return add ? launch_dt<kBF16, true>(x, res, w, y, h, rows, d, eps, vec, st)
               : launch_dt<kBF16, false>(x, res, w, y, h, rows, d, eps, vec, st);
}

}  // namespace gbe
