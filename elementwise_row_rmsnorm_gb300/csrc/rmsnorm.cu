// rmsnorm.cu -- RMSNorm, fused residual add + RMSNorm, and LayerNorm on
// sm_103a.
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
// that thread's (c div TPR)-th slot; TPR is the smallest multiple of 32 that
// leaves each thread at most 4 slots (rows of more than 4096 chunks use 1024
// threads and more slots).  TPR and the slot count depend only on (d,
// storage type).  A thread sums the squares of its chunks in slot order and
// element order (fused multiply-add), the row's threads are combined by a
// butterfly within each warp and then warp by warp in warp order.  So the
// summation tree of a row is fixed by (d, type): the row's output bits do
// not depend on how many rows the call holds or where the row sits.  The
// aligned (vector) and unaligned (scalar) paths use the same map and the
// same operation order, so they agree bit for bit too.
//
// Aligned rows (every pointer 16-byte aligned, d a multiple of the vector)
// stay in registers as packed vectors between the sum and the write (one HBM
// read of x, one write of y), with the 16-byte loads of all slots issued
// before any is used.  Other rows, and rows wider than 4096 chunks, take a
// two-pass kernel with the same map.  The row's sum is complete before the
// first write, so y may be x (and h may be residual).  Launches overlap the
// previous kernel's tail (programmatic dependent launch, see common.cuh).
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kMaxSlots = 4;

// (x_lo + c_lo, x_hi + c_hi) for the two bf16 values of a packed word by the
// mixed-precision add (the bf16 operand widened exactly, then one rounding:
// the bits of __fadd_rn on the widened value), with no unpacking.
__device__ __forceinline__ float2 bf16x2_plus(uint32_t w, float c_lo, float c_hi) {
    float d0, d1;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %4;\n\t}"
        : "=f"(d0), "=f"(d1) : "r"(w), "f"(c_lo), "f"(c_hi));
    return make_float2(d0, d1);
}

// s + x_lo + x_hi, in that order, for the two bf16 values of a packed word
// (the same mixed-precision add: the bits of two __fadd_rn).
__device__ __forceinline__ float bf16x2_sum_acc(uint32_t w, float s) {
    float d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.bf16 %0, lo, %2;\n\tadd.rn.f32.bf16 %0, hi, %0;\n\t}"
        : "=f"(d) : "r"(w), "f"(s));
    return d;
}

// Threads per row for a row of `nchunks` 16-byte chunks: enough that each
// owns at most kMaxSlots chunks.  A function of (d, dtype) only.
inline int64_t threads_per_row(int64_t nchunks) {
    int64_t tpr = ((nchunks + kMaxSlots - 1) / kMaxSlots + 31) / 32 * 32;
    return tpr < 32 ? 32 : tpr;
}

// Aligned rows: the row's chunks stay in registers as packed 16-byte vectors
// (4 f32 or 8 bf16 each) from the load to the write.
// TPR > 0: threads per row fixed at compile time (one row per CTA, or four
// one-warp rows when TPR is 32); TPR == 0: taken from `tpr_rt` (any multiple
// of 32 up to 1024, one row per CTA).  Either way the map and tree are those
// of the header comment.
template <int TPR>
struct RowShape {
    static constexpr int kRpc = TPR == 32 ? 4 : 1;
    static constexpr int kMaxThreads = TPR == 0 ? 1024 : TPR * kRpc;
    // Wide rows (512 or 1024 threads each): at least two rows resident per
    // SM, so that one row's reduction overlaps another's loads (a single
    // 1024-thread CTA per SM left the SM's load and store phases in turn).
    // Not for the fused add, whose second input would then spill.
    template <bool ADD>
    static constexpr int min_blocks() { return (TPR >= 512 && !ADD) ? 2048 / TPR : 1; }
    // LayerNorm rows of 64 to 256 threads: 1536 threads resident per SM (40
    // registers, no spill), as many rows as RMSNorm keeps, where the
    // unbounded kernel took 47 registers and fit 1280.
    static constexpr int ln_min_blocks() {
        return (TPR >= 64 && TPR <= 256) ? 1536 / (TPR > 0 ? TPR : 1) : min_blocks<false>();
    }
};

template <int DT, int K, bool ADD, int TPR>
__global__ void __launch_bounds__(RowShape<TPR>::kMaxThreads, RowShape<TPR>::template min_blocks<ADD>())
rmsnorm_rows(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows, int d, float eps,
             int tpr_rt) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    constexpr int rpc = RowShape<TPR>::kRpc;
    const int tpr = TPR > 0 ? TPR : tpr_rt;
    pdl_begin();
    const int sub = threadIdx.x / tpr;
    const int t = threadIdx.x - sub * tpr;
    const int64_t row = (int64_t)blockIdx.x * rpc + sub;
    if (row >= rows) return;  // only when several one-warp rows share a CTA: no CTA barrier follows
    const int nchunks = d / V;
    const int64_t boff = row * (int64_t)d * ES;
    __shared__ float red[32];

    Vec16 rx[K];
    Vec16 rr[ADD ? K : 1];
    // 1) every load of the row's slots in flight before any use
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            rx[k] = ld_stream(static_cast<const char*>(x) + boff + (int64_t)c * 16);
            if (ADD) rr[k] = ld_stream(static_cast<const char*>(res) + boff + (int64_t)c * 16);
        }
    }
    // 2) h = x + residual rounded to the storage type (stored, and kept as the
    //    row), then the sum of squares in slot order and element order
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            if (ADD) {
                float f[V], g[V];
                S::unpack(rx[k], f);
                S::unpack(rr[k], g);
#pragma unroll
                for (int e = 0; e < V; ++e) f[e] = __fadd_rn(f[e], g[e]);
                rx[k] = S::pack(f);
                st_stream(static_cast<char*>(h) + boff + (int64_t)c * 16, rx[k]);
            }
            s = vec_sq_acc<DT>(rx[k], s);  // the stored values' squares, element order
        }
    }
    // 3) the row's sum, fixed order
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float total = (TPR == 32) ? warp_sum(s) : row_sum(s, red, warp, lane, tpr >> 5);
    const float ms = __fdiv_rn(total, (float)d);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    // 4) y = x * inv * w
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            float f[V], wv[V];
            S::unpack(rx[k], f);
            S::unpack(ld_reuse(static_cast<const char*>(w) + (int64_t)c * 16), wv);
#pragma unroll
            for (int e = 0; e < V; ++e) f[e] = __fmul_rn(__fmul_rn(f[e], inv), wv[e]);
            st_stream(static_cast<char*>(y) + boff + (int64_t)c * 16, S::pack(f));
        }
    }
}

// Aligned rows of 1024 threads (more than 3072 chunks: f32 d up to 16384,
// bf16 up to 32768), plain RMSNorm, when the call holds more rows than two
// per SM: rmsnorm_rows keeps two such rows resident per SM, so a batch of R
// rows takes ceil(R / 2 SMs) waves of one row each, the last partly empty.
// Here one CTA per SM walks the rows blockIdx.x, + gridDim.x, ... with the
// next two rows' chunks already in flight into a ring of shared memory
// (cp.async, 16 bytes per copy).  Each thread copies exactly the chunks it
// will read, so its own wait_group (a hardware wait, not a loop) is the only
// wait before it reads them, and it refills a ring slot only after it has
// read that slot itself.  The map, the per-thread order and the reduction
// tree are rmsnorm_rows<DT, 4, false, 1024>'s, so the bits are the same.
constexpr int kStreamSlots = 3;  // rows a CTA holds: the one it works on and two in flight

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}

template <int DT>
__global__ void __launch_bounds__(1024, 1)
rmsnorm_stream(const void* x, const void* w, void* y, int64_t rows, int d, float eps) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int K = kMaxSlots;
    constexpr int TPR = 1024;
    constexpr int NS = kStreamSlots;
    constexpr int64_t ES = sizeof(typename S::T);
    extern __shared__ Vec16 ring[];  // [NS][K][TPR]
    __shared__ float red[2][32];
    pdl_begin();
    const int t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31;
    const int nchunks = d / V;
    const int64_t rb = (int64_t)d * ES;
    const int64_t G = gridDim.x;
    auto issue = [&](int64_t r, int slot) {
        if (r < rows) {
            const char* src = static_cast<const char*>(x) + r * rb;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int c = k * TPR + t;
                if (c < nchunks) cp_async16(&ring[(slot * K + k) * TPR + t], src + (int64_t)c * 16);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");  // empty past the last row: the count stays even
    };
    int64_t r = blockIdx.x;
#pragma unroll
    for (int q = 0; q < NS - 1; ++q) issue(r + q * G, q);
    // this thread's gains, the same for every row
    Vec16 wv[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * TPR + t;
        if (c < nchunks) wv[k] = ld_reuse(static_cast<const char*>(w) + (int64_t)c * 16);
    }
    int slot = 0, fill = NS - 1;
    for (int it = 0; r < rows; ++it, r += G) {  // r depends on blockIdx only: the CTA stays together
        issue(r + (NS - 1) * G, fill);
        asm volatile("cp.async.wait_group %0;" ::"n"(NS - 1) : "memory");  // this thread's chunks of row r
        Vec16 rx[K];
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int c = k * TPR + t;
            if (c < nchunks) {
                rx[k] = ring[(slot * K + k) * TPR + t];
                s = vec_sq_acc<DT>(rx[k], s);
            }
        }
        // the reduction's words alternate between rows: a row's are rewritten
        // two rows later, after every thread has passed the barrier between
        const float total = row_sum(s, red[it & 1], warp, lane, TPR >> 5);
        const float ms = __fdiv_rn(total, (float)d);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
        char* yr = static_cast<char*>(y) + r * rb;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int c = k * TPR + t;
            if (c < nchunks) {
                float f[V], g[V];
                S::unpack(rx[k], f);
                S::unpack(wv[k], g);
#pragma unroll
                for (int e = 0; e < V; ++e) f[e] = __fmul_rn(__fmul_rn(f[e], inv), g[e]);
                st_stream(yr + (int64_t)c * 16, S::pack(f));
            }
        }
        slot = slot + 1 == NS ? 0 : slot + 1;
        fill = fill + 1 == NS ? 0 : fill + 1;
    }
}

// Unaligned rows (and rows wider than kMaxSlots chunks of 1024 threads): the
// same chunk map, the same per-thread order and the same reduction tree as
// rmsnorm_rows would use for this d, element by element, with x (or the
// stored h) read a second time for the write.  One row per CTA of `tpr`
// threads.
template <int DT, bool ADD>
__global__ void __launch_bounds__(1024)
rmsnorm_two_pass(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows, int d,
                 float eps) {
    using S = Store<DT>;
    constexpr int V = S::V;
    pdl_begin();
    const int tpr = blockDim.x;
    const int t = threadIdx.x;
    const int64_t row = blockIdx.x;
    const int nchunks = (d + V - 1) / V;
    const int64_t base = row * (int64_t)d;
    __shared__ float red[32];
    const void* src = ADD ? h : x;
    float s = 0.0f;
    for (int c = t; c < nchunks; c += tpr) {
        for (int e = 0; e < V && c * V + e < d; ++e) {
            const int64_t i = base + (int64_t)c * V + e;
            float a = S::load1(x, i);
            if (ADD) {
                a = S::round(__fadd_rn(a, S::load1(res, i)));
                S::store1(h, i, a);
            }
            s = __fmaf_rn(a, a, s);
        }
    }
    const float total = row_sum(s, red, t >> 5, t & 31, tpr >> 5);
    const float ms = __fdiv_rn(total, (float)d);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    for (int c = t; c < nchunks; c += tpr) {
        for (int e = 0; e < V && c * V + e < d; ++e) {
            const int64_t j = (int64_t)c * V + e;
            S::store1(y, base + j, __fmul_rn(__fmul_rn(S::load1(src, base + j), inv), S::load1(w, j)));
        }
    }
}

// LayerNorm ("Operations", section 2): mu = mean(x), var = mean((x - mu)^2),
// y = ((x - mu) * (1 / sqrt(var + eps))) * g (+ b).  The same chunk map as
// RMSNorm; the row's two sums (of x, then of (x - mu)^2) each take the same
// fixed tree, so a row's bits depend only on the row, d and the type.
template <int DT, int K, int TPR>
__global__ void __launch_bounds__(RowShape<TPR>::kMaxThreads, RowShape<TPR>::ln_min_blocks())
layernorm_rows(const void* x, const void* g, const void* b, void* y, int64_t rows, int d, float eps, int tpr_rt) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    constexpr int rpc = RowShape<TPR>::kRpc;
    const int tpr = TPR > 0 ? TPR : tpr_rt;
    pdl_begin();
    const int sub = threadIdx.x / tpr;
    const int t = threadIdx.x - sub * tpr;
    const int64_t row = (int64_t)blockIdx.x * rpc + sub;
    if (row >= rows) return;  // only when several one-warp rows share a CTA
    const int nchunks = d / V;
    const int64_t boff = row * (int64_t)d * ES;
    __shared__ float red[2][32];
    Vec16 rx[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) rx[k] = ld_stream(static_cast<const char*>(x) + boff + (int64_t)c * 16);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            if (DT == kBF16) {  // the packed words added as they are: the same sums
#pragma unroll
                for (int w = 0; w < 4; ++w) s = bf16x2_sum_acc(rx[k].w[w], s);
            } else {
                float f[V];
                S::unpack(rx[k], f);
#pragma unroll
                for (int e = 0; e < V; ++e) s = __fadd_rn(s, f[e]);
            }
        }
    }
    const float mu = __fdiv_rn((TPR == 32) ? warp_sum(s) : row_sum(s, red[0], warp, lane, tpr >> 5), (float)d);
    float s2 = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks) {
            if (DT == kBF16) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float2 cc = bf16x2_plus(rx[k].w[w], -mu, -mu);  // x - mu == x + (-mu)
                    s2 = __fmaf_rn(cc.x, cc.x, s2);
                    s2 = __fmaf_rn(cc.y, cc.y, s2);
                }
            } else {
                float f[V];
                S::unpack(rx[k], f);
                const float2 m2 = make_float2(mu, mu);
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                    const float2 cc = sub2_rn(make_float2(f[e], f[e + 1]), m2);
                    s2 = __fmaf_rn(cc.x, cc.x, s2);
                    s2 = __fmaf_rn(cc.y, cc.y, s2);
                }
            }
        }
    }
    const float var = __fdiv_rn((TPR == 32) ? warp_sum(s2) : row_sum(s2, red[1], warp, lane, tpr >> 5), (float)d);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int c = k * tpr + t;
        if (c < nchunks && DT == kBF16) {
            // x - mu and the bias added to the packed words as they are (the
            // bits of the unpacked form below; b + u == u + b)
            float f[V], gv[V];
            const Vec16 bw = b != nullptr ? ld_reuse(static_cast<const char*>(b) + (int64_t)c * 16) : Vec16{};
            S::unpack(ld_reuse(static_cast<const char*>(g) + (int64_t)c * 16), gv);
            const float2 i2 = make_float2(inv, inv);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float2 u = mul2_rn(mul2_rn(bf16x2_plus(rx[k].w[w], -mu, -mu), i2),
                                         make_float2(gv[2 * w], gv[2 * w + 1]));
                const float2 o = b != nullptr ? bf16x2_plus(bw.w[w], u.x, u.y) : u;
                f[2 * w] = o.x;
                f[2 * w + 1] = o.y;
            }
            st_stream(static_cast<char*>(y) + boff + (int64_t)c * 16, S::pack(f));
        } else if (c < nchunks) {
            float f[V], gv[V], bv[V];
            S::unpack(rx[k], f);
            S::unpack(ld_reuse(static_cast<const char*>(g) + (int64_t)c * 16), gv);
            if (b != nullptr) S::unpack(ld_reuse(static_cast<const char*>(b) + (int64_t)c * 16), bv);
            const float2 m2 = make_float2(mu, mu), i2 = make_float2(inv, inv);
#pragma unroll
            for (int e = 0; e < V; e += 2) {
                // (x - mu) * inv * g for two entries per instruction; the bias
                // added by scalar adds (a packed product feeding a packed add
                // may be fused into one rounding)
                const float2 u = mul2_rn(mul2_rn(sub2_rn(make_float2(f[e], f[e + 1]), m2), i2),
                                         make_float2(gv[e], gv[e + 1]));
                f[e] = b != nullptr ? __fadd_rn(u.x, bv[e]) : u.x;
                f[e + 1] = b != nullptr ? __fadd_rn(u.y, bv[e + 1]) : u.y;
            }
            st_stream(static_cast<char*>(y) + boff + (int64_t)c * 16, S::pack(f));
        }
    }
}

// LayerNorm for unaligned or very wide rows: the same map and trees, x read
// three times (sum, centred sum of squares, write).  One row per CTA.
template <int DT>
__global__ void __launch_bounds__(1024)
layernorm_three_pass(const void* x, const void* g, const void* b, void* y, int64_t rows, int d, float eps) {
    using S = Store<DT>;
    constexpr int V = S::V;
    pdl_begin();
    const int tpr = blockDim.x;
    const int t = threadIdx.x;
    const int64_t base = (int64_t)blockIdx.x * d;
    const int nchunks = (d + V - 1) / V;
    __shared__ float red[2][32];
    float s = 0.0f;
    for (int c = t; c < nchunks; c += tpr)
        for (int e = 0; e < V && c * V + e < d; ++e) s = __fadd_rn(s, S::load1(x, base + (int64_t)c * V + e));
    const float mu = __fdiv_rn(row_sum(s, red[0], t >> 5, t & 31, tpr >> 5), (float)d);
    float s2 = 0.0f;
    for (int c = t; c < nchunks; c += tpr)
        for (int e = 0; e < V && c * V + e < d; ++e) {
            const float cc = __fsub_rn(S::load1(x, base + (int64_t)c * V + e), mu);
            s2 = __fmaf_rn(cc, cc, s2);
        }
    const float var = __fdiv_rn(row_sum(s2, red[1], t >> 5, t & 31, tpr >> 5), (float)d);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
    for (int c = t; c < nchunks; c += tpr)
        for (int e = 0; e < V && c * V + e < d; ++e) {
            const int64_t j = (int64_t)c * V + e;
            const float u = __fmul_rn(__fmul_rn(__fsub_rn(S::load1(x, base + j), mu), inv), S::load1(g, j));
            S::store1(y, base + j, b != nullptr ? __fadd_rn(u, S::load1(b, j)) : u);
        }
}

template <int DT>
cudaError_t launch_ln(const void* x, const void* g, const void* b, void* y, int64_t rows, int64_t d, float eps,
                      bool vec, cudaStream_t st) {
    constexpr int V = Store<DT>::V;
    const int64_t nchunks = (d + V - 1) / V;
    int64_t tpr = threads_per_row(nchunks);
    const bool wide = tpr > 1024;
    if (wide) tpr = 1024;
    const int di = (int)d, ti = (int)tpr;
    if (wide || !vec)
        return launch(layernorm_three_pass<DT>, dim3((unsigned)rows), dim3((unsigned)tpr), 0, st, x, g, b, y, rows,
                      di, eps);
    const int64_t slots = (nchunks + tpr - 1) / tpr;
    const dim3 one((unsigned)rows), four((unsigned)((rows + 3) / 4));
#define GBE_LN(KK, TT, GRID, BLOCK) \
    return launch(layernorm_rows<DT, KK, TT>, GRID, dim3(BLOCK), 0, st, x, g, b, y, rows, di, eps, ti)
    switch (tpr) {
        case 32:
            if (slots <= 1) GBE_LN(1, 32, four, 128);
            if (slots <= 2) GBE_LN(2, 32, four, 128);
            GBE_LN(4, 32, four, 128);
        case 64: GBE_LN(4, 64, one, 64);
        case 128: GBE_LN(4, 128, one, 128);
        case 256: GBE_LN(4, 256, one, 256);
        case 512: GBE_LN(4, 512, one, 512);
        case 1024: GBE_LN(4, 1024, one, 1024);
        default: GBE_LN(4, 0, one, tpr);
    }
#undef GBE_LN
}

// rmsnorm_stream with one CTA per SM, after the shared-memory opt-in (once
// per device); cudaErrorNotReady when the opt-in is refused, and the caller
// takes rmsnorm_rows.
template <int DT>
cudaError_t launch_stream(const void* x, const void* w, void* y, int64_t rows, int d, float eps, cudaStream_t st) {
    const size_t smem = (size_t)kStreamSlots * kMaxSlots * 1024 * sizeof(Vec16);
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (!(opted.load(std::memory_order_acquire) & bit) || bit == 0) {
        if (cudaFuncSetAttribute(rmsnorm_stream<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return cudaErrorNotReady;
        }
        opted.fetch_or(bit, std::memory_order_release);
    }
    const int64_t grid = std::min<int64_t>(rows, sm_count());
    return launch(rmsnorm_stream<DT>, dim3((unsigned)grid), dim3(1024), smem, st, x, w, y, rows, d, eps);
}

template <int DT, bool ADD>
cudaError_t launch_dt(const void* x, const void* res, const void* w, void* y, void* h, int64_t rows, int64_t d,
                      float eps, bool vec, cudaStream_t st) {
    constexpr int V = Store<DT>::V;
    const int64_t nchunks = (d + V - 1) / V;
    int64_t tpr = threads_per_row(nchunks);
    const bool wide = tpr > 1024;
    if (wide) tpr = 1024;
    const int di = (int)d, ti = (int)tpr;
    if (wide || !vec) {
        return launch(rmsnorm_two_pass<DT, ADD>, dim3((unsigned)rows), dim3((unsigned)tpr), 0, st, x, res, w, y, h,
                      rows, di, eps);
    }
    if (!ADD && tpr == 1024 && rows > 2LL * sm_count()) {
        const cudaError_t e = launch_stream<DT>(x, w, y, rows, di, eps, st);
        if (e != cudaErrorNotReady) return e;
    }
    const int64_t slots = (nchunks + tpr - 1) / tpr;
    const dim3 one((unsigned)rows), four((unsigned)((rows + 3) / 4));
#define GBE_RMS(KK, TT, GRID, BLOCK) \
    return launch(rmsnorm_rows<DT, KK, ADD, TT>, GRID, dim3(BLOCK), 0, st, x, res, w, y, h, rows, di, eps, ti)
    switch (tpr) {
        case 32:
            if (slots <= 1) GBE_RMS(1, 32, four, 128);
            if (slots <= 2) GBE_RMS(2, 32, four, 128);
            GBE_RMS(4, 32, four, 128);
        case 64: GBE_RMS(4, 64, one, 64);
        case 128: GBE_RMS(4, 128, one, 128);
        case 256: GBE_RMS(4, 256, one, 256);
        case 512: GBE_RMS(4, 512, one, 512);
        case 1024: GBE_RMS(4, 1024, one, 1024);
        default: GBE_RMS(4, 0, one, tpr);
    }
#undef GBE_RMS
}

}  // namespace

cudaError_t launch_layernorm(const void* x, const void* g, const void* b, void* y, int64_t rows, int64_t d,
                             float eps, int dtype, bool vec, cudaStream_t st) {
    return dtype == kF32 ? launch_ln<kF32>(x, g, b, y, rows, d, eps, vec, st)
                         : launch_ln<kBF16>(x, g, b, y, rows, d, eps, vec, st);
}

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
