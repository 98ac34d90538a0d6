// argmax.cu -- greedy argmax over each row on sm_103a.
//
// Definition ("Elementwise kernels in C", section 2.4 and 4; "Operations",
// section 1, Argmax, and section 8, greedy sampling): the index of the
// largest value of the row, the lowest index among equal values, NaN entries
// skipped, and -1 when the row holds no number.  -0 and +0 are equal (so the
// lower index wins); +inf is a number; a row of -inf gives 0.
//
// The answer is unique, so any split of the row and any combining order give
// the same index: a candidate (value, index) beats another when it is a
// number and the other is not, or its value is greater, or the values are
// equal and its index is lower.  That rule is associative and commutative.
//
// Map: CL CTAs per row (CL in {1, 2, 4, 8}, a thread-block cluster when
// CL > 1).  The row is cut into CL contiguous segments of 16-byte vectors;
// within a segment thread t reads vectors t, t + 256, ... in increasing order
// (8 loads in flight before any compare), so a strict > keeps the first
// index within a thread.  Per vector, the largest number is found first
// (fmaxf, which skips NaN) and only a vector whose maximum beats the thread's
// best is searched for the first position of that maximum.  Threads combine
// by a warp butterfly and then warp by warp; the CTAs of a cluster combine
// through distributed shared memory on rank 0 after a cluster barrier (a
// hardware barrier over co-scheduled CTAs, no spin loop), and a second
// barrier keeps every CTA's shared memory alive until rank 0 has read it.
// CL grows only while rows * CL stays below eight CTAs per SM, so few long
// rows (decode) still fill the GPU.
#include <atomic>
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace gbe {

int sm_count() {
    static std::atomic<int> cached[64];  // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return 152;
    }
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = 152;
    }
    if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;

// (bv, bi) <- better of (bv, bi) and (v, i); bi < 0 means "no number yet".
__device__ __forceinline__ void take_better(float& bv, int& bi, float v, int i) {
    if (i >= 0 && (bi < 0 || v > bv || (v == bv && i < bi))) {
        bv = v;
        bi = i;
    }
}

// Forward scan step: entries arrive in increasing index order.
__device__ __forceinline__ void scan(float& bv, int& bi, float v, int i) {
    if (v == v && (bi < 0 || v > bv)) {
        bv = v;
        bi = i;
    }
}

template <int DT, bool VEC, int CL>
__device__ __forceinline__ void argmax_body(const void* x, int32_t* out, int64_t rows, int64_t n) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    pdl_begin();
    const int64_t row = blockIdx.x / CL;
    const int rank = (int)(blockIdx.x % CL);
    const char* base = static_cast<const char*>(x) + row * n * ES;
    float bv = 0.0f;
    int bi = -1;
    if (VEC) {
        const int64_t nvec = n / V;
        const int64_t per = (nvec + CL - 1) / CL;
        const int64_t s0 = rank * per;
        const int64_t s1 = min(nvec, s0 + per);
        for (int64_t j0 = s0 + threadIdx.x; j0 < s1; j0 += (int64_t)kBatch * kThreads) {
            Vec16 r[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t j = j0 + (int64_t)u * kThreads;
                if (j < s1) r[u] = ld_stream(base + j * 16);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t j = j0 + (int64_t)u * kThreads;
                if (j < s1) {
                    float f[V];
                    S::unpack(r[u], f);
                    // the vector's largest number (fmaxf skips NaN; NaN only if all are NaN) ...
                    float m = f[0];
#pragma unroll
                    for (int e = 1; e < V; ++e) m = fmaxf(m, f[e]);
                    // ... wins over the thread's best only if strictly greater (earlier
                    // vectors have lower indices), then its first position is taken
                    if (m > bv || (bi < 0 && m == m)) {
                        int e0 = V - 1;
#pragma unroll
                        for (int e = V - 1; e >= 0; --e)
                            if (f[e] == m) e0 = e;
                        bv = m;
                        bi = (int)(j * V + e0);
                    }
                }
            }
        }
    } else {
        const int64_t per = (n + CL - 1) / CL;
        const int64_t s0 = rank * per;
        const int64_t s1 = min(n, s0 + per);
        for (int64_t i = s0 + threadIdx.x; i < s1; i += kThreads) scan(bv, bi, S::load1(base, i), (int)i);
    }
    // warp butterfly, then the warps in order
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, m);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, m);
        take_better(bv, bi, ov, oi);
    }
    __shared__ float wv[kThreads / 32];
    __shared__ int wi[kThreads / 32];
    __shared__ float cv;
    __shared__ int ci;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        wv[warp] = bv;
        wi[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float v = wv[0];
        int i = wi[0];
        for (int w = 1; w < kThreads / 32; ++w) take_better(v, i, wv[w], wi[w]);
        cv = v;
        ci = i;
        if (CL == 1) out[row] = i;
    }
    if (CL > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (rank == 0 && threadIdx.x == 0) {
            float v = cv;
            int i = ci;
            for (int q = 1; q < CL; ++q) {
                const float* rv = cluster.map_shared_rank(&cv, q);
                const int* ri = cluster.map_shared_rank(&ci, q);
                take_better(v, i, *rv, *ri);
            }
            out[row] = i;
        }
        cluster.sync();
    }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) argmax_rows1(const void* x, int32_t* out, int64_t rows, int64_t n) {
    argmax_body<DT, VEC, 1>(x, out, rows, n);
}
template <int DT, bool VEC>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads)
argmax_rows2(const void* x, int32_t* out, int64_t rows, int64_t n) {
    argmax_body<DT, VEC, 2>(x, out, rows, n);
}
template <int DT, bool VEC>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kThreads)
argmax_rows4(const void* x, int32_t* out, int64_t rows, int64_t n) {
    argmax_body<DT, VEC, 4>(x, out, rows, n);
}
template <int DT, bool VEC>
__global__ void __cluster_dims__(8, 1, 1) __launch_bounds__(kThreads)
argmax_rows8(const void* x, int32_t* out, int64_t rows, int64_t n) {
    argmax_body<DT, VEC, 8>(x, out, rows, n);
}

template <int DT, bool VEC>
cudaError_t launch_cl(const void* x, int32_t* out, int64_t rows, int64_t n, cudaStream_t st) {
    const int64_t target = 8LL * sm_count();
    int cl = 1;
    while (cl < 8 && rows * cl < target && n / (cl * 2) >= 2048) cl *= 2;
    const dim3 grid((unsigned)(rows * cl));
    switch (cl) {
        case 1: return launch(argmax_rows1<DT, VEC>, grid, dim3(kThreads), 0, st, x, out, rows, n);
        case 2: return launch(argmax_rows2<DT, VEC>, grid, dim3(kThreads), 0, st, x, out, rows, n);
        case 4: return launch(argmax_rows4<DT, VEC>, grid, dim3(kThreads), 0, st, x, out, rows, n);
        default: return launch(argmax_rows8<DT, VEC>, grid, dim3(kThreads), 0, st, x, out, rows, n);
    }
}

}  // namespace

cudaError_t launch_argmax(const void* x, int32_t* out, int64_t rows, int64_t n, int dtype, bool vec,
                          cudaStream_t st) {
    if (dtype == kF32)
        return vec ? launch_cl<kF32, true>(x, out, rows, n, st) : launch_cl<kF32, false>(x, out, rows, n, st);
    return vec ? launch_cl<kBF16, true>(x, out, rows, n, st) : launch_cl<kBF16, false>(x, out, rows, n, st);
}

}  // namespace gbe
