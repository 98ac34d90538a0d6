// sample.cu -- sampling beyond greedy on sm_103a.
//
// Definition ("Operations", section 8, Sample): Temperature(t) draws from
// softmax(logits / t); TopK(k, t) from the softmax of the k largest logits,
// taken in descending order; TopP(p, t) from the descending softmax cut to
// the prefix whose running sum stays <= p (its first entry always kept) and
// renormalised; MinP(p, t) from the softmax cut to the entries >= p times its
// maximum and renormalised; Greedy is argmax.  The draw (sample_categorical)
// is the inverse CDF: with the caller's uniform u in [0, 1) for the row, the
// first entry, in the distribution's order, whose running sum exceeds u times
// the sum.  NaN logits take no part; equal logits order by ascending index;
// a row whose largest logit / t is not finite gives -1.
//
// Arithmetic.  For every logit e = expf(x / t - m), m the largest x / t, so
// 0 <= e <= 1; e is then held as the integer w = rn(e * 2^40), and every sum,
// histogram and threshold is an integer.  Integer sums do not depend on their
// order, so a draw is deterministic however the threads are scheduled, and
// the normalisation by the sum is never divided out: the target of a draw
// is floor(u * W) for the kept mass W.  (The min-p cut e / S >= p * max(e / S)
// is taken as the equivalent e >= p, since max(e) = 1.)  Rows are limited to
// 2^23 entries so that W < 2^63.
//
// Map: one CTA of 1024 threads per row; thread i owns a contiguous chunk of
// the row (index order within a thread, threads in order), read with 16-byte
// loads when the row allows, from L2 after the first pass.
//  * temperature, min-p (index order): one pass forms the chunk sums, a block
//    scan finds the chunk holding the target, its thread walks the chunk.
//  * top-k, top-p (descending order): the position where the descending
//    running count (top-k's cut) or mass (top-p's cut, and the draw) passes
//    its target is found digit by digit -- 8-bit digits of an order-keeping
//    32-bit key of the logit, a 256-bin histogram per digit (the first
//    digit's built once) -- then inside the group of logits equal to the
//    found key, in index order.  No sort of the vocabulary and no memory
//    beyond the inputs and the outputs.
#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kT = 1024;
constexpr int kWarps = kT / 32;
constexpr float kScale = 1099511627776.0f;  // 2^40
typedef unsigned long long u64;

enum { kGreedy = 0, kTemperature = 1, kTopK = 2, kTopP = 3, kMinP = 4 };

// Larger logit, larger key (the IEEE order of non-NaN floats, -0 below +0).
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct Smem {
    u64 mass0[256];  // first-digit histogram of every valid entry, kept for reuse
    unsigned cnt0[256];
    u64 mass[256];  // histogram of the current digit
    unsigned cnt[256];
    u64 wu[kWarps];
    float wf[kWarps];
    int wi[kWarps];
    u64 bu[2];
    int bi[2];
};

template <int DT, bool VEC>
struct Row {
    const void* x;
    int64_t base;  // element offset of the row
    float t, m;    // temperature; the largest x / t
    int c0, c1;    // this thread's chunk [c0, c1)

    __device__ __forceinline__ float e_of(float v) const { return expf(__fsub_rn(__fdiv_rn(v, t), m)); }
    __device__ __forceinline__ static u64 w_of(float e) { return __float2ull_rn(__fmul_rn(e, kScale)); }
    // fixed-point weight of a logit that is not NaN
    __device__ __forceinline__ u64 weight(float v) const { return w_of(e_of(v)); }

    // f(i, v) for every entry of the chunk in index order, NaN included
    template <typename F>
    __device__ __forceinline__ void each(F f) const {
        if (VEC) {
            constexpr int V = Store<DT>::V;
            const char* p = static_cast<const char*>(x) + (base + c0) * (int64_t)sizeof(typename Store<DT>::T);
            for (int i = c0; i < c1; i += V, p += 16) {
                float fv[V];
                Store<DT>::unpack(ld_reuse(p), fv);
#pragma unroll
                for (int e = 0; e < V; ++e) f(i + e, fv[e]);
            }
        } else {
            for (int i = c0; i < c1; ++i) f(i, Store<DT>::load1(x, base + i));
        }
    }
};

// ---- block primitives (1024 threads; each opens with a barrier so that the
//      shared slots of the previous call are free) -------------------------------

__device__ __forceinline__ float block_max(float v, Smem& sh) {
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.wf[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = sh.wf[0];
    for (int w = 1; w < kWarps; ++w) r = fmaxf(r, sh.wf[w]);
    return r;
}

__device__ __forceinline__ int block_sum_int(int v, Smem& sh) {
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.wi[threadIdx.x >> 5] = v;
    __syncthreads();
    int r = 0;
    for (int w = 0; w < kWarps; ++w) r += sh.wi[w];
    return r;
}

// exclusive prefix of v over the threads in order; *total gets the sum
__device__ __forceinline__ u64 block_exscan(u64 v, Smem& sh, u64* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    u64 inc = v;
    for (int o = 1; o < 32; o <<= 1) {
        const u64 y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();
    if (lane == 31) sh.wu[warp] = inc;
    __syncthreads();
    u64 before = 0, all = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before += sh.wu[w];
        all += sh.wu[w];
    }
    *total = all;
    return before + inc - v;
}

// ---- descending order ------------------------------------------------------------
//
// The entry at which the descending running count (BY_COUNT) or mass first
// exceeds `target` (target < the total of the valid entries).  Returns its
// index; *ahead gets the mass of the entries before it in descending order.
// The first digit's histogram must be in mass0 / cnt0.
template <int DT, bool VEC, bool BY_COUNT>
__device__ int find_descending(const Row<DT, VEC>& row, u64 target, Smem& sh, u64* ahead) {
    uint32_t prefix = 0;
    u64 base_m = 0, base_c = 0;  // mass and count of the entries above the current bin
    for (int level = 0; level < 4; ++level) {
        const int shift = 24 - 8 * level;
        if (level > 0) {
            __syncthreads();
            for (int b = threadIdx.x; b < 256; b += kT) {
                sh.mass[b] = 0;
                sh.cnt[b] = 0;
            }
            __syncthreads();
            row.each([&](int, float v) {
                if (v != v) return;
                const uint32_t key = order_key(v);
                if ((key >> (shift + 8)) != prefix) return;
                const int bin = (key >> shift) & 255;
                atomicAdd(&sh.cnt[bin], 1u);
                atomicAdd(&sh.mass[bin], row.weight(v));
            });
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            const u64* mm = level == 0 ? sh.mass0 : sh.mass;
            const unsigned* cc = level == 0 ? sh.cnt0 : sh.cnt;
            int chosen = 0;
            for (int b = 255; b >= 0; --b) {
                const u64 step = BY_COUNT ? (u64)cc[b] : mm[b];
                const u64 run = BY_COUNT ? base_c : base_m;
                if (step > 0 && run + step > target) {
                    chosen = b;
                    break;
                }
                base_m += mm[b];
                base_c += cc[b];
            }
            sh.bu[0] = base_m;
            sh.bu[1] = base_c;
            sh.bi[0] = chosen;
        }
        __syncthreads();
        base_m = sh.bu[0];
        base_c = sh.bu[1];
        prefix = (prefix << 8) | (uint32_t)sh.bi[0];
        __syncthreads();
    }
    // The group of entries equal to `prefix`, in index order.  All of them
    // carry the same weight w (the same logit), so within the group the
    // position follows from a count: the found entry is the group's j-th,
    // j = (target - base) / (1 or w), and `ahead` adds the j entries before it.
    const uint32_t key = prefix;
    u64 w_key = 0, mine = 0;
    row.each([&](int, float v) {
        if (v == v && order_key(v) == key) {
            ++mine;
            w_key = row.weight(v);
        }
    });
    u64 dummy;
    // every thread learns the group's weight (the largest of the per-thread copies)
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.wu[threadIdx.x >> 5] = 0;
    __syncthreads();
    if (mine > 0) atomicMax(&sh.wu[threadIdx.x >> 5], w_key);
    __syncthreads();
    u64 w = 0;
    for (int q = 0; q < kWarps; ++q) w = sh.wu[q] > w ? sh.wu[q] : w;
    const u64 ex = block_exscan(mine, sh, &dummy);  // entries of the group in earlier chunks
    const u64 j = BY_COUNT ? target - base_c : (target - base_m) / w;
    __syncthreads();
    if (threadIdx.x == 0) sh.bi[1] = -1;
    __syncthreads();
    if (mine > 0 && ex <= j && j < ex + mine) {
        u64 seen = ex;
        int found = -1;
        row.each([&](int i, float v) {
            if (found < 0 && v == v && order_key(v) == key) {
                if (seen == j) found = i;
                ++seen;
            }
        });
        sh.bi[1] = found;
    }
    __syncthreads();
    *ahead = base_m + j * w;
    return sh.bi[1];
}

__device__ __forceinline__ u64 scaled(float u, u64 total) {
    const u64 t = (u64)((double)u * (double)total);
    return t >= total ? total - 1 : t;
}

template <int DT, bool VEC>
__device__ __forceinline__ void sample_body(const void* x, int32_t* out, int n, int method, float t, int k, float p,
                                            const float* u, Smem& sh) {
    const int64_t r = blockIdx.x;
    Row<DT, VEC> row;
    row.x = x;
    row.base = r * (int64_t)n;
    row.t = t;
    row.m = 0.0f;
    // chunk length: a whole number of 16-byte vectors for either storage type
    const int chunk = ((n + kT - 1) / kT + 7) & ~7;
    row.c0 = min(n, (int)threadIdx.x * chunk);
    row.c1 = min(n, row.c0 + chunk);

    // pass 0: the largest logit and the count of valid entries
    float mx = -INFINITY;
    int nv = 0;
    row.each([&](int, float v) {
        if (v == v) {
            mx = fmaxf(mx, v);
            ++nv;
        }
    });
    mx = block_max(mx, sh);
    nv = block_sum_int(nv, sh);
    row.m = __fdiv_rn(mx, t);
    if (nv == 0 || !isfinite(row.m)) {
        if (threadIdx.x == 0) out[r] = -1;
        return;
    }
    const float ur = u[r];

    if (method == kTemperature || method == kMinP) {
        const bool minp = method == kMinP;
        u64 mine = 0;
        row.each([&](int, float v) {
            if (v != v) return;
            const float e = row.e_of(v);
            if (minp && !(e >= p)) return;
            mine += row.w_of(e);
        });
        u64 total;
        const u64 ex = block_exscan(mine, sh, &total);
        const u64 target = scaled(ur, total);
        if (mine > 0 && ex <= target && target < ex + mine) {
            u64 run = ex;
            int found = -1;
            row.each([&](int i, float v) {
                if (found >= 0 || v != v) return;
                const float e = row.e_of(v);
                if (minp && !(e >= p)) return;
                run += row.w_of(e);
                if (run > target) found = i;
            });
            out[r] = found;
        }
        return;
    }

    // top-k, top-p: the first digit's histogram of every valid entry
    for (int b = threadIdx.x; b < 256; b += kT) {
        sh.mass0[b] = 0;
        sh.cnt0[b] = 0;
    }
    __syncthreads();
    row.each([&](int, float v) {
        if (v != v) return;
        const int bin = order_key(v) >> 24;
        atomicAdd(&sh.cnt0[bin], 1u);
        atomicAdd(&sh.mass0[bin], row.weight(v));
    });
    __syncthreads();
    u64 all = 0;
    for (int b = 0; b < 256; ++b) all += sh.mass0[b];
    u64 kept = all;
    if (method == kTopK) {
        if (k < nv) find_descending<DT, VEC, true>(row, (u64)k, sh, &kept);  // first entry past the k-th
    } else {
        // keep the prefix whose running mass stays <= p * W; the first entry always
        const u64 cut = (u64)((double)p * (double)all);
        if (cut < all) {
            find_descending<DT, VEC, false>(row, cut, sh, &kept);
            if (kept == 0) kept = 1;  // a target of 0 lands on the first entry
        }
    }
    u64 unused;
    const int idx = find_descending<DT, VEC, false>(row, scaled(ur, kept), sh, &unused);
    if (threadIdx.x == 0) out[r] = idx;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kT)
sample_rows(const void* x, int32_t* out, int n, int method, float t, int k, float p, const float* u) {
    pdl_begin();
    __shared__ Smem sh;
    sample_body<DT, VEC>(x, out, n, method, t, k, p, u, sh);
}

template <int DT>
cudaError_t launch_dt(const void* x, int32_t* out, int64_t rows, int n, int method, float t, int k, float p,
                      const float* u, bool vec, cudaStream_t st) {
    if (vec) return launch(sample_rows<DT, true>, dim3((unsigned)rows), dim3(kT), 0, st, x, out, n, method, t, k, p, u);
    return launch(sample_rows<DT, false>, dim3((unsigned)rows), dim3(kT), 0, st, x, out, n, method, t, k, p, u);
}

}  // namespace

cudaError_t launch_sample(const void* x, int32_t* out, int64_t rows, int64_t n, int method, float t, int64_t k,
                          float p, const float* u, int dtype, bool vec, cudaStream_t st) {
    if (method == kGreedy) return launch_argmax(x, out, rows, n, dtype, vec, st);
    const int ki = (int)(k > n ? n : k), ni = (int)n;
    if (dtype == kF32) return launch_dt<kF32>(x, out, rows, ni, method, t, ki, p, u, vec, st);
    return launch_dt<kBF16>(x, out, rows, ni, method, t, ki, p, u, vec, st);
}

}  // namespace gbe
