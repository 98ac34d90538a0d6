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
// Arithmetic.  For every logit e = 2^((x - M) * c) in f32, M the largest
// logit and c = log2(e) / t (ex2.approx; e = 1 exactly where x = M), so
// 0 <= e <= 1 -- the softmax numerator exp(x / t - M / t) up to a few f32
// roundings.  e is then held as the integer w = rn(e * 2^40), and every sum,
// histogram and threshold is an integer.  Integer sums do not depend on their
// order, so a draw is deterministic however the threads are scheduled, and
// the normalisation is never divided out: the target of a draw is
// floor(u * W) for the kept mass W, and the drawn entry is the first whose
// running mass exceeds it.  (The min-p cut e / S >= p * max(e / S) is taken
// as the equivalent e >= p, since max(e) = 1.)  Rows are limited to 2^23
// entries so that W < 2^63.
//
// Map: one CTA of 512 threads (16 warps) per row -- or, for batches too
// small to fill the GPU, temperature and min-p rows over a cluster of 2, 4
// or 8 CTAs.  Warp w owns a contiguous segment of the row, read in
// coalesced tiles of 32 16-byte vectors (lane l holds tile entries
// [l V, l V + V)), so index order is warp, tile, lane, element.  The first
// pass reads HBM; later ones walk the segment backwards and mostly hit L2.
//  * temperature, min-p (index order): pass 1 the maximum, pass 2 each
//    warp's kept mass in units of V consecutive entries (their e summed in
//    f32, the unit sum held as a fixed-point integer); the warp holding the
//    target walks its segment tile by tile with warp scans, then the unit's
//    own partial sums.
//  * top-k, top-p (descending order): pass 1 also leaves each thread's own
//    maximum; a floor that enough entries reach (from those maxima, sorted
//    per warp) selects the few entries at the top of the row, which pass 2
//    gathers into shared memory as (key, ~index) pairs -- for top-p while
//    it sums the row's mass -- and they are ordered descending, equal
//    logits by index (key: an order-keeping 32-bit image of the logit): up
//    to 256 by a one-step rank sort, more by a bitonic sort in shared
//    memory.  Top-k draws among the first k; top-p walks the sorted prefix
//    for the cut and the draw when the prefix's mass passes the cut (else
//    a second, wider gather is tried the same way).  Otherwise
//    (large k, flat or heavily tied rows) an exact radix search: the key's
//    12 / 10 / 10-bit digits, a histogram per digit (counts, and masses as
//    exact 64-bit sums in two 32-bit words) locates the bin where the
//    descending running count or mass passes its target; that bin's
//    entries are gathered, sorted and walked; a bin of more than 4096
//    entries is split by the next digit, and a group of more than 4096
//    equal logits is walked in index order by the warps.
// The uniform of a row is the caller's u[row], or draw offset + row of the
// seeded PCG64 stream (pcg64.cuh), formed by warp 0 at the row's start.
// No memory beyond the inputs and the outputs.
#include <algorithm>
#include <atomic>
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "pcg64.cuh"

namespace gbe {

namespace cg = cooperative_groups;

namespace {

constexpr int kT = 512;
constexpr int kW = kT / 32;
constexpr int kU = 4;                       // tiles in flight per lane
constexpr int kMaxCand = 4096;              // entries gathered into shared memory
constexpr int kTopLanes = 64;               // top-p first gathers entries >= a floor this many reach
constexpr int kBins0 = 4096, kBins1 = 1024;  // 12-bit first digit, 10-bit others
constexpr float kScale = 1099511627776.0f;  // 2^40
constexpr unsigned kFull = 0xFFFFFFFFu;
typedef unsigned long long u64;

enum { kGreedy = 0, kTemperature = 1, kTopK = 2, kTopP = 3, kMinP = 4 };

// Larger logit, larger key (the IEEE order of non-NaN floats), and back.
// -0 takes the key of +0: the two are equal logits, which order by index
// like any other equal logits (as argmax ties -0 and +0 to the lower index).
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
// candidate = key above, complemented index below: descending order of the
// candidates is descending key, then ascending index
__device__ __forceinline__ u64 cand_of(uint32_t key, int i) { return ((u64)key << 32) | (uint32_t)~(uint32_t)i; }
__device__ __forceinline__ int cand_index(u64 c) { return (int)~(uint32_t)c; }

struct Sh {
    u64 wu[kW];
    float wf[kW];
    int wi[kW];
    u64 ru[4];
    int ri[4];
    unsigned ncand;
    float useed;  // the row's uniform, when it is drawn from the seeded stream
};

// The row's uniform drawn from the seeded stream (d.u == NULL): warp 0
// forms it at the start of the row, before its first loads, and leaves it
// in sh.useed for row_uniform to read after the first block barrier.
__device__ __forceinline__ void seed_uniform(const Draws& d, int64_t ri, Sh& sh) {
    if (d.u == nullptr && threadIdx.x < 32) {
        const float v = pcg::uniform_warp(d.seed, d.offset, (u64)ri);
        if (threadIdx.x == 0) sh.useed = v;
    }
}
__device__ __forceinline__ float row_uniform(const Draws& d, int64_t ri, const Sh& sh) {
    return d.u ? d.u[ri] : sh.useed;
}


// 2^a, the hardware approximation (relative error near 2^-22; results below
// 2^-126 flush to 0, far below the 2^-41 resolution of the weights).
__device__ __forceinline__ float ex2(float a) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// rn(e * 2^40) for 0 <= e <= 1, exactly: below 2^23 the sum with 2^23 rounds
// to the nearest integer (ties to even) and leaves it in the low mantissa
// bits; from 2^23 on, e * 2^40 is an integer and the mantissa, shifted, is it.
__device__ __forceinline__ bool fixed40_small(float y) { return y < 8388608.0f; }
__device__ __forceinline__ uint32_t fixed40_lo(float y) {
    return __float_as_uint(__fadd_rn(y, 8388608.0f)) - 0x4B000000u;
}
__device__ __forceinline__ u64 fixed40_hi(float e) {
    const uint32_t b = __float_as_uint(e);
    return (u64)((b & 0x7FFFFFu) | 0x800000u) << ((int)(b >> 23) - 127 + 17);
}
__device__ __forceinline__ u64 fixed40(float e) {
    const float y = __fmul_rn(e, kScale);
    return fixed40_small(y) ? (u64)fixed40_lo(y) : fixed40_hi(e);
}

// A running sum of fixed40 weights: the common small ones (below 2^23) in a
// 32-bit word, folded into the 64-bit sum after every kU tiles (at most 32
// additions, so the word cannot overflow).
struct MassAcc {
    u64 big = 0;
    uint32_t small = 0;
    __device__ __forceinline__ void add(float e) {
        const float y = __fmul_rn(e, kScale);
        if (fixed40_small(y)) small += fixed40_lo(y);
        else big += fixed40_hi(e);
    }
    __device__ __forceinline__ void fold() {
        big += small;
        small = 0;
    }
    __device__ __forceinline__ u64 total() const { return big + small; }
};

// The float interval of the keys [lo_key, hi_key] (NaN patterns at either
// end widen it to an infinity); every non-NaN float whose key lies in the
// range lies in the interval (-0 and +0 compare equal, so the interval may
// admit one of them from outside: callers recheck the key).
__device__ __forceinline__ float key_floor(u64 lo_key) {
    return lo_key < 0x00800000ull ? -INFINITY : key_value((uint32_t)lo_key);
}
__device__ __forceinline__ float key_ceil(u64 hi_key) {
    return hi_key >= 0xFF800000ull ? INFINITY : key_value((uint32_t)hi_key);
}

template <int DT, bool VEC>
struct Row {
    static constexpr int V = Store<DT>::V;
    static constexpr int kTile = 32 * V;
    const void* x;
    int64_t base;  // element offset of the row
    float t, mx, c;  // temperature; the largest logit; log2(e) / t
    int s0, s1;      // this warp's segment [s0, s1)
    int lane;

    // c is finite (clamped at setup), so x = M gives 0 * c = 0 and
    // ex2.approx(0) = 1 exactly; NaN stays NaN for the callers to drop
    __device__ __forceinline__ float e_of(float v) const { return ex2(__fmul_rn(__fsub_rn(v, mx), c)); }
    __device__ __forceinline__ static u64 w_of(float e) { return fixed40(e); }
    // fixed-point weight of a logit that is not NaN
    __device__ __forceinline__ u64 weight(float v) const { return w_of(e_of(v)); }

    // The start of the segment's last group of kU tiles (s0 - 1 when the
    // segment is empty).  Later passes walk the groups backwards: the tiles
    // pass 1 read last are the likeliest to be still in L2.  Their sums are
    // integers and the gathers are sorted afterwards, so order is free.
    __device__ __forceinline__ int last_group() const {
        return s1 > s0 ? s0 + (s1 - s0 - 1) / (kTile * kU) * (kTile * kU) : s0 - 1;
    }

    // this lane's 16-byte vector of the tile starting at j, NaN entries past
    // the segment (aligned rows)
    __device__ __forceinline__ Vec16 load_raw(int j) const {
        const int i = j + lane * V;
        if (i < s1) return ld_reuse(static_cast<const char*>(x) + (base + i) * (int64_t)sizeof(typename Store<DT>::T));
        Vec16 r;
#pragma unroll
        for (int w = 0; w < 4; ++w) r.w[w] = DT == kBF16 ? 0x7FC07FC0u : 0x7FC00000u;
        return r;
    }

    // this lane's V entries of the tile starting at j (NaN past the segment)
    __device__ __forceinline__ void load(int j, float (&v)[V]) const {
        const int i = j + lane * V;
        if (VEC) {
            if (i < s1) {
                Store<DT>::unpack(
                    ld_reuse(static_cast<const char*>(x) + (base + i) * (int64_t)sizeof(typename Store<DT>::T)), v);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) v[e] = __int_as_float(0x7FC00000);
            }
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) v[e] = i + e < s1 ? Store<DT>::load1(x, base + i + e) : __int_as_float(0x7FC00000);
        }
    }

    // f(i, v) for every entry of the segment, NaN past its end, then after()
    // once per kU tiles; every lane of the warp makes every call, so f may
    // use warp-wide operations
    template <typename F, typename G>
    __device__ __forceinline__ void each(F f, G after) const {
        for (int j0 = s0; j0 < s1; j0 += kTile * kU) {
            float v[kU][V];
#pragma unroll
            for (int q = 0; q < kU; ++q) load(j0 + q * kTile, v[q]);
#pragma unroll
            for (int q = 0; q < kU; ++q)
#pragma unroll
                for (int e = 0; e < V; ++e) f(j0 + q * kTile + lane * V + e, v[q][e]);
            after();
        }
    }
    template <typename F>
    __device__ __forceinline__ void each(F f) const {
        each(f, [] {});
    }
};

// The largest number among a vector's entries, NaN only when all are NaN
// (bf16: packed maxima, which skip NaN as fmaxf does).  Some entry is >= T
// exactly when this maximum is.
template <int DT>
__device__ __forceinline__ float vec_max(const Vec16& r) {
    if (DT == kBF16) {
        const __nv_bfloat162 m = __hmax2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&r.w[0]),
                                                 *reinterpret_cast<const __nv_bfloat162*>(&r.w[1])),
                                         __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&r.w[2]),
                                                 *reinterpret_cast<const __nv_bfloat162*>(&r.w[3])));
        const float2 f = __bfloat1622float2(m);
        return fmaxf(f.x, f.y);
    }
    return fmaxf(fmaxf(__uint_as_float(r.w[0]), __uint_as_float(r.w[1])),
                 fmaxf(__uint_as_float(r.w[2]), __uint_as_float(r.w[3])));
}

// bit e set for the entries v[e] >= T (NaN fails)
template <int V>
__device__ __forceinline__ unsigned bits_ge(const float (&v)[V], float T) {
    unsigned in = 0;
#pragma unroll
    for (int e = 0; e < V; ++e) in |= (v[e] >= T ? 1u : 0u) << e;
    return in;
}

// A unit's e summed in f32 in index order, NaN entries left out.  Every e of
// a number lies in [0, 1], so the plain sum is NaN exactly when some entry
// is NaN; only then is the unit summed again with those entries skipped.
template <int DT, bool VEC>
__device__ __forceinline__ float unit_sum(const Row<DT, VEC>& row, const float (&v)[Row<DT, VEC>::V]) {
    constexpr int V = Row<DT, VEC>::V;
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < V; ++e) s = __fadd_rn(s, row.e_of(v[e]));
    if (s != s) {
        s = 0.0f;
#pragma unroll
        for (int e = 0; e < V; ++e) s = __fadd_rn(s, fmaxf(row.e_of(v[e]), 0.0f));  // NaN gives 0
    }
    return s;
}

// The f32 sums, in index order, of the e of two units at once: entry e of
// unit 0 and entry e of unit 1 go through the subtraction, the scaling and
// the running sums as the two lanes of packed instructions (each lane's
// arithmetic is the scalar one, bit for bit; no product feeds a sum: the
// exponential sits between).  A lane is NaN where its unit holds a NaN;
// unit_sum then gives that unit's sum with them skipped.  (Top-p's mass
// pass; the index-order kernel keeps the scalar form, which fits its
// 40-register budget without spilling.)
template <int DT, bool VEC>
__device__ __forceinline__ float2 unit_sums2(const Row<DT, VEC>& row, const float (&v0)[Row<DT, VEC>::V],
                                             const float (&v1)[Row<DT, VEC>::V]) {
    constexpr int V = Row<DT, VEC>::V;
    const float2 M = make_float2(row.mx, row.mx), C = make_float2(row.c, row.c);
    float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int e = 0; e < V; ++e) {
        const float2 y = mul2_rn(sub2_rn(make_float2(v0[e], v1[e]), M), C);
        s = add2_rn(s, make_float2(ex2(y.x), ex2(y.y)));
    }
    return s;
}

template <int DT, bool VEC>
__device__ __forceinline__ float unit_sum_of(const Row<DT, VEC>& row, const Vec16& r) {
    float v[Row<DT, VEC>::V];
    Store<DT>::unpack(r, v);
    return unit_sum(row, v);
}

// rn(rn(v - M) * c) for the two bf16 values of a packed word, low half
// first, with no unpacking: the subtraction is the mixed-precision add of
// -M (the bf16 operand widened exactly, then one rounding -- the bits of
// __fsub_rn on the widened value), the two products one packed multiply.
__device__ __forceinline__ float2 scaled_bf16x2(uint32_t w, float neg_m, float c) {
    float d0, d1;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %3;\n\t}"
        : "=f"(d0), "=f"(d1) : "r"(w), "f"(neg_m));
    return mul2_rn(make_float2(d0, d1), make_float2(c, c));
}

// The same values with the two halves widened and one packed addition of
// -M: more instructions than the mixed-precision form in the index-order
// kernels (measured slower there), fewer in top-p's mass pass, which takes
// this one (626 -> 617 us at [8192, 128256] on one GPU).
__device__ __forceinline__ float2 scaled_bf16x2_packed(uint32_t w, float neg_m, float c) {
    const float2 v = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    return mul2_rn(add2_rn(v, make_float2(neg_m, neg_m)), make_float2(c, c));
}

// unit_sum of a packed bf16 unit (the same bits): e of each entry from the
// packed word, summed in index order; a unit holding NaN is summed again,
// unpacked, with those entries skipped.  MINP: e counts only where e >= p
// (NaN fails), the sum of kept_e.
template <int DT, bool VEC, bool MINP>
__device__ __forceinline__ float unit_sum_bf16(const Row<DT, VEC>& row, const Vec16& r, float p) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 y = scaled_bf16x2(r.w[w], -row.mx, row.c);
        const float e0 = ex2(y.x), e1 = ex2(y.y);
        s = __fadd_rn(s, MINP ? (e0 >= p ? e0 : 0.0f) : e0);
        s = __fadd_rn(s, MINP ? (e1 >= p ? e1 : 0.0f) : e1);
    }
    if (!MINP && s != s) s = unit_sum_of(row, r);
    return s;
}

// unit_sums2 of two packed bf16 units (the same bits): entry e of unit 0 and
// of unit 1 summed as the two lanes of packed additions.
template <int DT, bool VEC>
__device__ __forceinline__ float2 unit_sums2_bf16(const Row<DT, VEC>& row, const Vec16& r0, const Vec16& r1) {
    float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 y0 = scaled_bf16x2_packed(r0.w[w], -row.mx, row.c);
        const float2 y1 = scaled_bf16x2_packed(r1.w[w], -row.mx, row.c);
        s = add2_rn(s, make_float2(ex2(y0.x), ex2(y1.x)));
        s = add2_rn(s, make_float2(ex2(y0.y), ex2(y1.y)));
    }
    return s;
}

// ---- warp and block primitives ----------------------------------------------------

__device__ __forceinline__ u64 warp_sum_u64(u64 v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ u64 warp_incl_scan_u64(u64 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u64 y = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// Each block primitive opens with a barrier, so the shared slots of the
// previous call are free.
__device__ __forceinline__ float block_max(float v, Sh& sh) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.wf[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = sh.wf[0];
    for (int w = 1; w < kW; ++w) r = fmaxf(r, sh.wf[w]);
    return r;
}

__device__ __forceinline__ int block_sum_int(int v, Sh& sh) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.wi[threadIdx.x >> 5] = v;
    __syncthreads();
    int r = 0;
    for (int w = 0; w < kW; ++w) r += sh.wi[w];
    return r;
}

// exclusive prefix of v over the threads in order; *total gets the sum
__device__ __forceinline__ u64 block_exscan(u64 v, Sh& sh, u64* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const u64 inc = warp_incl_scan_u64(v, lane);
    __syncthreads();
    if (lane == 31) sh.wu[warp] = inc;
    __syncthreads();
    u64 before = 0, all = 0;
    for (int w = 0; w < kW; ++w) {
        if (w < warp) before += sh.wu[w];
        all += sh.wu[w];
    }
    *total = all;
    return before + inc - v;
}

// exclusive prefix over the warps of a value every lane of a warp holds
__device__ __forceinline__ u64 warp_exscan(u64 warp_value, Sh& sh, u64* total) {
    const int warp = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sh.wu[warp] = warp_value;
    __syncthreads();
    u64 before = 0, all = 0;
    for (int w = 0; w < kW; ++w) {
        if (w < warp) before += sh.wu[w];
        all += sh.wu[w];
    }
    *total = all;
    return before;
}

__device__ __forceinline__ u64 scaled(float u, u64 total) {
    const u64 t = (u64)((double)u * (double)total);
    return t >= total ? total - 1 : t;
}

// The warp walks its segment tile by tile and returns the first index whose
// running measure (meas(v) per entry, 0 for entries that take no part)
// exceeds target, measured from the segment's start; -1 if none does.
template <int DT, bool VEC, typename M>
__device__ int warp_walk(const Row<DT, VEC>& row, u64 target, M meas) {
    constexpr int V = Row<DT, VEC>::V;
    u64 run = 0;
    for (int j = row.s0; j < row.s1; j += Row<DT, VEC>::kTile) {
        float v[V];
        row.load(j, v);
        u64 s = 0;
#pragma unroll
        for (int e = 0; e < V; ++e) s += meas(v[e]);
        const u64 inc = warp_incl_scan_u64(s, row.lane);
        const u64 tot = __shfl_sync(kFull, inc, 31);
        if (run + tot > target) {
            int found = -1;
            const u64 ex = inc - s;
            if (run + ex <= target && target < run + inc) {
                u64 r = run + ex;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    r += meas(v[e]);
                    if (found < 0 && r > target) found = j + row.lane * V + e;
                }
            }
            const unsigned who = __ballot_sync(kFull, found >= 0);
            return __shfl_sync(kFull, found, __ffs(who) - 1);
        }
        run += tot;
    }
    return -1;
}

// ---- index order: temperature and min-p -------------------------------------------

// The row of this CTA (row i of CL CTAs each, rank r of them) and this
// warp's segment: the row is cut into CL * kW segments of whole tiles, CTA r
// owning segments r kW .. r kW + kW - 1.  Segments start at multiples of a
// tile, so the units (V consecutive entries from the row's start) are the
// same for every CL.
template <int DT, bool VEC>
__device__ __forceinline__ void setup(Row<DT, VEC>& row, const void* x, int n, float t, int64_t i = blockIdx.x,
                                      int rank = 0, int cl = 1) {
    constexpr int kTile = Row<DT, VEC>::kTile;
    row.x = x;
    row.base = i * n;
    row.t = t;
    row.mx = 0.0f;
    row.c = fminf(__fdiv_rn(1.44269502f, t), 3.4028234663852886e38f);  // log2(e) / t, finite
    row.lane = threadIdx.x & 31;
    const int nseg = kW * cl;
    const int per = ((n + nseg - 1) / nseg + kTile - 1) / kTile * kTile;
    const int w = rank * kW + (threadIdx.x >> 5);
    row.s0 = min(n, w * per);
    row.s1 = min(n, row.s0 + per);
}

// false (and -1 written by `writer` at out[i]) when the row has no number or
// no finite largest x / t; a row of NaN leaves mx = -inf, not finite either
template <int DT, bool VEC>
__device__ __forceinline__ bool accept_max(const Row<DT, VEC>& row, int32_t* out, int64_t i, bool writer) {
    if (!isfinite(__fdiv_rn(row.mx, row.t))) {
        if (writer) out[i] = -1;
        return false;
    }
    return true;
}

// Pass 1: the CTA's largest logit over its warps' segments (NaN skipped;
// -inf when none is a number), with COUNT the count of numbers, and each
// thread's own maximum in thread_max when given.
template <bool COUNT, int DT, bool VEC>
__device__ __forceinline__ float block_first_max(Row<DT, VEC>& row, Sh& sh, int* nv_out, float* thread_max) {
    float mx = -INFINITY;
    int nv = 0;
    if (DT == kBF16 && VEC && !COUNT) {
        // bf16: the maximum on packed pairs (__hmax2 skips NaN like fmaxf;
        // a pair of NaN stays NaN, and the -inf start keeps the running value
        // a number), two entries per instruction, no unpacking
        constexpr int kTile = Row<DT, VEC>::kTile;
        __nv_bfloat162 acc = __floats2bfloat162_rn(-INFINITY, -INFINITY);
        for (int j0 = row.s0; j0 < row.s1; j0 += kTile * kU) {
            Vec16 q[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = j0 + u * kTile + row.lane * Row<DT, VEC>::V;
                if (i < row.s1) {
                    q[u] = ld_reuse(static_cast<const char*>(row.x) + (row.base + i) * (int64_t)2);
                } else {
#pragma unroll
                    for (int w = 0; w < 4; ++w) q[u].w[w] = 0x7FC07FC0u;  // NaN pairs
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u)
#pragma unroll
                for (int w = 0; w < 4; ++w) acc = __hmax2(acc, *reinterpret_cast<const __nv_bfloat162*>(&q[u].w[w]));
        }
        const float2 f = __bfloat1622float2(acc);
        mx = fmaxf(f.x, f.y);
    } else {
        row.each([&](int, float v) {
            mx = fmaxf(mx, v);  // NaN is ignored
            if (COUNT && v == v) ++nv;
        });
    }
    if (thread_max) thread_max[threadIdx.x] = mx;  // this thread's own maximum (-inf if it has no number)
    mx = block_max(mx, sh);
    if (COUNT) nv = block_sum_int(nv, sh);
    *nv_out = nv;
    return mx;
}

// Index order works on units: a lane's V consecutive entries of one tile.
// A unit's e (0 for NaN and, under min-p, for e < p) are summed in f32 in
// index order, and the partial sum s_j after its j-th entry is held as
// fixed40(s_j); the unit's weight is fixed40(s_{V-1}).  Unit weights are
// exact integers, so the warp and block sums are order-free; inside the unit
// the drawn entry is the first j with fixed40(s_j) above the residual target
// -- fixed40 is monotone and s_j never decreases, so the walk that recomputes
// the same partial sums always finds it.  Entry j thus weighs
// fixed40(s_j) - fixed40(s_{j-1}), e_j * 2^40 up to one f32 rounding of s_j.
template <int DT, bool VEC, bool MINP>
__device__ __forceinline__ float kept_e(const Row<DT, VEC>& row, float v, float p) {
    const float e = row.e_of(v);          // NaN for NaN
    return MINP ? (e >= p ? e : 0.0f)     // NaN fails the test
                : fmaxf(e, 0.0f);         // NaN gives 0
}

// One row per CL CTAs (a thread-block cluster when CL > 1, for batches too
// small to fill the GPU with one CTA a row).  The CTAs combine their
// maxima and their masses through distributed shared memory after hardware
// cluster barriers (no spin loop); a CTA leaves only after a barrier that
// follows every read of its shared memory by the others.  Every CL gives
// the same draw: the unit weights are the same integers, summed exactly.
//
// Three rows resident per SM (40 registers a thread): the tiles in flight
// stay packed, which is what lets the aligned kernels fit without spilling.
template <int DT, bool VEC, bool MINP, int CL>
__device__ __forceinline__ void index_order_body(const void* x, int32_t* out, int n, float t, float p, Draws d) {
    constexpr int V = Row<DT, VEC>::V;
    constexpr int kTile = Row<DT, VEC>::kTile;
    pdl_begin();
    __shared__ Sh sh;
    __shared__ float cl_max;  // this CTA's maximum, read by the cluster
    __shared__ u64 cl_mass;   // this CTA's kept mass, read by the cluster
    const int64_t ri = CL > 1 ? (int64_t)(blockIdx.x / CL) : (int64_t)blockIdx.x;
    const int rank = CL > 1 ? (int)(blockIdx.x % CL) : 0;
    Row<DT, VEC> row;
    setup(row, x, n, t, ri, rank, CL);
    seed_uniform(d, ri, sh);
    int nv;
    row.mx = block_first_max<false>(row, sh, &nv, nullptr);
    if (CL > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        if (threadIdx.x == 0) cl_max = row.mx;
        cluster.sync();
        float m = -INFINITY;
#pragma unroll
        for (int q = 0; q < CL; ++q) m = fmaxf(m, *cluster.map_shared_rank(&cl_max, q));
        row.mx = m;
        if (!accept_max(row, out, ri, rank == 0 && threadIdx.x == 0)) {
            cluster.sync();  // the others' reads of cl_max are done
            return;
        }
    } else if (!accept_max(row, out, ri, threadIdx.x == 0)) {
        return;
    }
    auto unit = [&](const float (&v)[V]) -> u64 {
        if (!MINP) return fixed40(unit_sum(row, v));
        float s = 0.0f;
#pragma unroll
        for (int e = 0; e < V; ++e) s = __fadd_rn(s, kept_e<DT, VEC, MINP>(row, v[e], p));
        return fixed40(s);
    };
    u64 mine = 0;
    for (int j0 = row.last_group(); j0 >= row.s0; j0 -= kTile * kU) {
        if (VEC) {
            // the tiles in flight stay packed; each is unpacked as its unit is summed
            Vec16 r[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) r[q] = row.load_raw(j0 + q * kTile);
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                if (DT == kBF16) {
                    mine += fixed40(unit_sum_bf16<DT, VEC, MINP>(row, r[q], p));
                } else {
                    float v[V];
                    Store<DT>::unpack(r[q], v);
                    mine += unit(v);
                }
            }
        } else {
            float v[kU][V];
#pragma unroll
            for (int q = 0; q < kU; ++q) row.load(j0 + q * kTile, v[q]);
#pragma unroll
            for (int q = 0; q < kU; ++q) mine += unit(v[q]);
        }
    }
    u64 total;
    const u64 wmass = warp_sum_u64(mine);
    u64 ex = warp_exscan(wmass, sh, &total);
    if (CL > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        if (threadIdx.x == 0) cl_mass = total;
        cluster.sync();  // also: every CTA is done reading cl_max
        u64 before = 0, all = 0;
#pragma unroll
        for (int q = 0; q < CL; ++q) {
            const u64 m = *cluster.map_shared_rank(&cl_mass, q);
            if (q < rank) before += m;
            all += m;
        }
        cluster.sync();  // every read of cl_mass is done before any CTA leaves
        ex += before;
        total = all;
    }
    const u64 target = scaled(row_uniform(d, ri, sh), total);
    if (!(wmass > 0 && ex <= target && target < ex + wmass)) return;
    // this warp holds the target: walk its tiles
    const u64 want = target - ex;
    u64 run = 0;
    for (int j = row.s0; j < row.s1; j += kTile) {
        float v[V];
        row.load(j, v);
        const u64 w = unit(v);
        const u64 inc = warp_incl_scan_u64(w, row.lane);
        const u64 tot = __shfl_sync(kFull, inc, 31);
        if (run + tot > want) {
            int found = -1;
            const u64 before = run + inc - w;
            if (before <= want && want < run + inc) {
                const u64 r = want - before;
                float s = 0.0f;
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    s = __fadd_rn(s, kept_e<DT, VEC, MINP>(row, v[e], p));
                    if (found < 0 && fixed40(s) > r) found = j + row.lane * V + e;
                }
            }
            const unsigned who = __ballot_sync(kFull, found >= 0);
            const int idx = __shfl_sync(kFull, found, who ? __ffs(who) - 1 : 0);
            if (row.lane == 0) out[ri] = idx;
            return;
        }
        run += tot;
    }
}

template <int DT, bool VEC, bool MINP>
__global__ void __launch_bounds__(kT, 3) sample_index_order(const void* x, int32_t* out, int n, float t, float p,
                                                            Draws d) {
    index_order_body<DT, VEC, MINP, 1>(x, out, n, t, p, d);
}
template <int DT, bool VEC, bool MINP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kT, 3)
sample_index_order2(const void* x, int32_t* out, int n, float t, float p, Draws d) {
    index_order_body<DT, VEC, MINP, 2>(x, out, n, t, p, d);
}
template <int DT, bool VEC, bool MINP>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kT, 3)
sample_index_order4(const void* x, int32_t* out, int n, float t, float p, Draws d) {
    index_order_body<DT, VEC, MINP, 4>(x, out, n, t, p, d);
}
template <int DT, bool VEC, bool MINP>
__global__ void __cluster_dims__(8, 1, 1) __launch_bounds__(kT, 3)
sample_index_order8(const void* x, int32_t* out, int n, float t, float p, Draws d) {
    index_order_body<DT, VEC, MINP, 8>(x, out, n, t, p, d);
}

// CTAs per row for the index-order kernels: doubled while the grid still
// fits in one wave (three CTAs an SM) and each warp keeps two tiles.
template <int DT, bool VEC, bool MINP>
cudaError_t launch_index_order(const void* x, int32_t* out, int64_t rows, int n, float t, float p, Draws d,
                               cudaStream_t st) {
    constexpr int kTile = Row<DT, VEC>::kTile;
    const int64_t target = 3LL * sm_count();
    int cl = 1;
    while (cl < 8 && rows * cl * 2 <= target && (int64_t)n >= (int64_t)kW * 2 * (2 * cl) * kTile) cl *= 2;
    const dim3 grid((unsigned)(rows * cl)), block(kT);
    switch (cl) {
        case 1: return launch(sample_index_order<DT, VEC, MINP>, grid, block, 0, st, x, out, n, t, p, d);
        case 2: return launch(sample_index_order2<DT, VEC, MINP>, grid, block, 0, st, x, out, n, t, p, d);
        case 4: return launch(sample_index_order4<DT, VEC, MINP>, grid, block, 0, st, x, out, n, t, p, d);
        default: return launch(sample_index_order8<DT, VEC, MINP>, grid, block, 0, st, x, out, n, t, p, d);
    }
}

// ---- descending order: top-k and top-p ---------------------------------------------

// A histogram in shared memory: counts, and masses as exact 64-bit sums held
// in two 32-bit words, so that every update is a native 32-bit shared atomic
// (the carry out of the low word goes into the high word).
struct Hist {
    unsigned* cnt;
    unsigned* lo;
    unsigned* hi;
    int nbins;
    __device__ __forceinline__ u64 count(int b) const { return cnt[b]; }
    __device__ __forceinline__ u64 mass(int b) const { return ((u64)hi[b] << 32) + lo[b]; }
    __device__ __forceinline__ void clear() const {
        for (int b = threadIdx.x; b < nbins; b += kT) cnt[b] = lo[b] = hi[b] = 0u;
    }
    __device__ __forceinline__ void add(int b, bool with_mass, u64 w) const {
        atomicAdd(&cnt[b], 1u);
        if (with_mass && w) {
            const uint32_t wl = (uint32_t)w;
            const uint32_t old = atomicAdd(&lo[b], wl);
            const uint32_t up = (uint32_t)(w >> 32) + (old + wl < old ? 1u : 0u);
            if (up) atomicAdd(&hi[b], up);
        }
    }
};

struct ShBig {
    Sh s;
    unsigned cnt0[kBins0], lo0[kBins0], hi0[kBins0];
    unsigned cnt1[kBins1], lo1[kBins1], hi1[kBins1];
    u64 cand[kMaxCand];
    float lmax[kT];  // the threads' own maxima of the first pass
    __device__ __forceinline__ Hist h0() { return Hist{cnt0, lo0, hi0, kBins0}; }
    __device__ __forceinline__ Hist h1() { return Hist{cnt1, lo1, hi1, kBins1}; }
};

// ---- one warp over at most 256 candidates ----------------------------------------
//
// The common case of top-k and top-p gathers a few hundred candidates at
// most.  The block ranks them (one barrier), then one warp holds them in
// sorted order (8 per lane, entry i = 8 lane + slot) and finds the cut and
// the draw with warp scans, where the block-wide sort and walks take several
// dozen barriers.
constexpr int kWarpCand = 256;

struct WarpSorted {
    u64 c[8];    // the sorted candidates of this lane (0: past the end)
    u64 cum[8];  // running mass through each (inclusive), in sorted order
};

// Sort the nc <= kWarpCand candidates cand[0, nc) descending into
// sorted[0, nc): thread i counts the candidates greater than its own (all
// reads of one step hit one shared word) and writes its own at that rank.
// Candidates are distinct (their low words hold distinct indices), so the
// ranks are a permutation.  The caller's barrier makes sorted visible.
__device__ __forceinline__ void rank_sort(const u64* cand, u64* sorted, int nc) {
    const int i = threadIdx.x;
    if (i < nc) {
        const u64 c = cand[i];
        int r = 0;
        int j = 0;
        for (; j + 4 <= nc; j += 4)
            r += (int)(cand[j] > c) + (int)(cand[j + 1] > c) + (int)(cand[j + 2] > c) + (int)(cand[j + 3] > c);
        for (; j < nc; ++j) r += (int)(cand[j] > c);
        sorted[r] = c;
    }
}

// One warp loads the sorted candidates (8 per lane, position 8 lane + slot)
// and their running masses.
template <int DT, bool VEC>
__device__ __forceinline__ void warp_weigh(const Row<DT, VEC>& row, const u64* sorted, int nc, int lane,
                                           WarpSorted& ws) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = lane * 8 + k;
        ws.c[k] = i < nc ? sorted[i] : 0ull;
    }
    u64 run = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        run += ws.c[k] ? row.weight(key_value((uint32_t)(ws.c[k] >> 32))) : 0ull;
        ws.cum[k] = run;
    }
    const u64 inc = warp_incl_scan_u64(run, lane);
    const u64 base = inc - run;
#pragma unroll
    for (int k = 0; k < 8; ++k) ws.cum[k] += base;
}

// The first sorted position j < L whose running mass exceeds target (-1 if
// none); *before gets the mass ahead of it, *cand the candidate there.
template <int DT, bool VEC>
__device__ __forceinline__ int warp_first_above(const Row<DT, VEC>& row, const WarpSorted& ws, int L, u64 target,
                                                int lane, u64* before, u64* cand) {
    int kf = 8;
#pragma unroll
    for (int k = 7; k >= 0; --k)
        if (lane * 8 + k < L && ws.cum[k] > target) kf = k;
    const unsigned who = __ballot_sync(kFull, kf < 8);
    if (!who) return -1;
    const int src = __ffs(who) - 1;
    u64 cum = 0, c = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k == kf) {
            cum = ws.cum[k];
            c = ws.c[k];
        }
    cum = __shfl_sync(kFull, cum, src);
    c = __shfl_sync(kFull, c, src);
    *before = cum - row.weight(key_value((uint32_t)(c >> 32)));
    *cand = c;
    return src * 8 + __shfl_sync(kFull, kf, src);
}

// the running mass through sorted position L - 1 (L >= 1)
__device__ __forceinline__ u64 warp_mass_through(const WarpSorted& ws, int L) {
    const int j = L - 1;
    u64 v = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k == (j & 7)) v = ws.cum[k];
    return __shfl_sync(kFull, v, j >> 3);
}

// The bin (scanning from the top bin down) where the running sum of h(b)
// passes target (target < the sum); *above gets the sum of the bins above it.
template <typename H>
__device__ int find_bin(H h, int nbins, u64 target, Sh& sh, u64* above) {
    const int per = nbins / kT;
    const int top = nbins - (int)threadIdx.x * per;  // this thread's bins [top - per, top), from the top
    u64 local = 0;
    for (int b = top - 1; b >= top - per; --b) local += h(b);
    u64 total;
    const u64 ex = block_exscan(local, sh, &total);
    if (threadIdx.x == 0) {
        sh.ri[0] = 0;
        sh.ru[0] = 0;
    }
    __syncthreads();
    if (local > 0 && ex <= target && target < ex + local) {
        u64 run = ex;
        for (int b = top - 1; b >= top - per; --b) {
            const u64 v = h(b);
            if (v > 0 && run + v > target) {
                sh.ri[0] = b;
                sh.ru[0] = run;
                break;
            }
            run += v;
        }
    }
    __syncthreads();
    *above = sh.ru[0];
    return sh.ri[0];
}

// sum of h(b) over the bins above b0 (all bins when b0 = -1)
template <typename H>
__device__ u64 sum_above(H h, int nbins, int b0, Sh& sh) {
    u64 s = 0;
    for (int b = b0 + 1 + (int)threadIdx.x; b < nbins; b += kT) s += h(b);
    u64 total;
    block_exscan(s, sh, &total);
    return total;
}

// First-digit histogram of the valid entries whose first digit is >= from
// (0: all of them), with masses when hist_mass; returns this thread's share
// of the row's exact total mass when total_mass (every valid entry, in the
// histogram or not), else 0.
template <int DT, bool VEC>
__device__ u64 build_first(const Row<DT, VEC>& row, ShBig& sb, uint32_t from, bool hist_mass, bool total_mass) {
    const Hist h = sb.h0();
    const float x_from = key_floor((u64)from << 20);
    __syncthreads();
    h.clear();
    __syncthreads();
    MassAcc acc;
    row.each(
        [&](int, float v) {
            if (v != v) return;
            float e = 0.0f;
            if (hist_mass || total_mass) e = row.e_of(v);
            if (total_mass) acc.add(e);
            if (v >= x_from) {
                const uint32_t d = order_key(v) >> 20;
                if (d >= from) h.add((int)d, hist_mass, hist_mass ? row.w_of(e) : 0ull);
            }
        },
        [&] { acc.fold(); });
    __syncthreads();
    return acc.total();
}

// Histogram of the 10-bit digit (key >> shift) & 1023 over the entries whose
// key >> (shift + 10) equals prefix, with masses.
template <int DT, bool VEC>
__device__ void build_next(const Row<DT, VEC>& row, ShBig& sb, int shift, uint32_t prefix) {
    const Hist h = sb.h1();
    __syncthreads();
    h.clear();
    __syncthreads();
    row.each([&](int, float v) {
        if (v != v) return;
        const uint32_t key = order_key(v);
        if ((key >> (shift + 10)) != prefix) return;
        h.add((int)((key >> shift) & (kBins1 - 1)), true, row.weight(v));
    });
    __syncthreads();
}

__device__ int sort_cand(ShBig& sb);

// A floor that at least kW * m entries of the row reach (1 <= m <= 32): each
// warp sorts its 32 threads' own maxima (a bitonic network over lanes, no
// barrier) and offers its m-th largest; the floor is the least of the
// warps' offers, so every warp has m threads whose maximum -- an entry of
// the row -- reaches it.  -inf when some warp has fewer than m threads with
// a number: then every number reaches it.
__device__ float maxima_floor(float mine, int m, Sh& sh) {
    const int lane = threadIdx.x & 31;
    float v = mine;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float o = __shfl_xor_sync(kFull, v, stride);
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0 || size == 32);
            v = keep_max ? fmaxf(v, o) : fminf(v, o);
        }
    }
    const float offer = __shfl_sync(kFull, v, m - 1);  // lanes now hold the maxima in descending order
    __syncthreads();
    if (lane == 0) sh.wf[threadIdx.x >> 5] = offer;
    __syncthreads();
    float f = sh.wf[0];
    for (int w = 1; w < kW; ++w) f = fminf(f, sh.wf[w]);
    return f;
}

// Gather the entries for which sel(v) holds into cand as (key, ~index) and
// sort them descending (after() runs once per kU tiles); returns their count
// (the caller's selection holds at most kMaxCand entries).
template <int DT, bool VEC, typename F, typename G>
__device__ int gather_sorted_by(const Row<DT, VEC>& row, ShBig& sb, F sel, G after) {
    __syncthreads();
    if (threadIdx.x == 0) sb.s.ncand = 0;
    __syncthreads();
    row.each(
        [&](int i, float v) {
            if (!sel(v)) return;
            const unsigned slot = atomicAdd(&sb.s.ncand, 1u);
            if (slot < (unsigned)kMaxCand) sb.cand[slot] = cand_of(order_key(v), i);
        },
        after);
    return sort_cand(sb);
}

// Sort the gathered candidates descending (bitonic, in shared memory);
// returns their count (at most kMaxCand).
__device__ int sort_cand(ShBig& sb) {
    __syncthreads();
    const int nc = (int)min(sb.s.ncand, (unsigned)kMaxCand);
    int P = 1;
    while (P < nc) P <<= 1;
    for (int i = nc + (int)threadIdx.x; i < P; i += kT) sb.cand[i] = 0ull;  // pads sort last
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < P; i += kT) {
                const int ij = i ^ j;
                if (ij > i) {
                    const u64 a = sb.cand[i], b = sb.cand[ij];
                    const bool desc = (i & k) == 0;
                    if (desc ? (a < b) : (a > b)) {
                        sb.cand[i] = b;
                        sb.cand[ij] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    return nc;
}

// The entries whose key >> shift lies in [lo, hi], gathered and sorted.
template <int DT, bool VEC>
__device__ int gather_sorted(const Row<DT, VEC>& row, int shift, uint32_t lo, uint32_t hi, ShBig& sb) {
    const float x_lo = key_floor((u64)lo << shift), x_hi = key_ceil((((u64)hi + 1) << shift) - 1);
    return gather_sorted_by(
        row, sb,
        [&](float v) {
            if (!(v >= x_lo && v <= x_hi)) return false;  // NaN fails too
            const uint32_t d = order_key(v) >> shift;
            return d >= lo && d <= hi;
        },
        [] {});
}

// In the sorted candidates [0, L): the first position whose running mass
// exceeds target; *before gets the mass of the positions ahead of it.
template <int DT, bool VEC>
__device__ int sorted_pick(const Row<DT, VEC>& row, int L, u64 target, ShBig& sb, u64* before) {
    constexpr int per = kMaxCand / kT;
    const int j0 = (int)threadIdx.x * per;
    u64 local = 0;
    for (int j = j0; j < min(L, j0 + per); ++j) local += row.weight(key_value((uint32_t)(sb.cand[j] >> 32)));
    u64 total;
    const u64 ex = block_exscan(local, sb.s, &total);
    if (threadIdx.x == 0) {
        sb.s.ri[1] = -1;
        sb.s.ru[1] = 0;
    }
    __syncthreads();
    if (local > 0 && ex <= target && target < ex + local) {
        u64 run = ex;
        for (int j = j0; j < min(L, j0 + per); ++j) {
            const u64 w = row.weight(key_value((uint32_t)(sb.cand[j] >> 32)));
            if (run + w > target) {
                sb.s.ri[1] = j;
                sb.s.ru[1] = run;
                break;
            }
            run += w;
        }
    }
    __syncthreads();
    *before = sb.s.ru[1];
    return sb.s.ri[1];
}

// mass of the sorted candidates [0, q)
template <int DT, bool VEC>
__device__ u64 sorted_mass(const Row<DT, VEC>& row, int q, ShBig& sb) {
    u64 s = 0;
    for (int j = threadIdx.x; j < q; j += kT) s += row.weight(key_value((uint32_t)(sb.cand[j] >> 32)));
    u64 total;
    block_exscan(s, sb.s, &total);
    return total;
}

// The entry where the descending running count (BY_COUNT) or mass first
// exceeds target; returns its index, *ahead gets the mass of the entries
// before it.  The first-digit histogram must hold, with masses, every entry
// down to the bin where target falls (whole bins: a histogram of the top
// bins only serves every target below its sum).
template <int DT, bool VEC, bool BY_COUNT>
__device__ int desc_search(const Row<DT, VEC>& row, u64 target, ShBig& sb, u64* ahead) {
    const Hist h0 = sb.h0(), h1 = sb.h1();
    auto c0 = [&](int b) { return h0.count(b); };
    auto m0 = [&](int b) { return h0.mass(b); };
    auto c1 = [&](int b) { return h1.count(b); };
    auto m1 = [&](int b) { return h1.mass(b); };
    u64 a_meas;  // count or mass of the entries above the current bin
    const int b0 = BY_COUNT ? find_bin(c0, kBins0, target, sb.s, &a_meas) : find_bin(m0, kBins0, target, sb.s, &a_meas);
    u64 a_mass = BY_COUNT ? sum_above(m0, kBins0, b0, sb.s) : a_meas;
    uint32_t prefix = (uint32_t)b0;
    int shift = 20;
    u64 count = h0.count(b0);
    // split bins too large to gather by the next digits
    for (int level = 1; level <= 2 && count > (u64)kMaxCand; ++level) {
        shift -= 10;
        build_next(row, sb, shift, prefix);
        u64 a1;
        const int b1 = BY_COUNT ? find_bin(c1, kBins1, target - a_meas, sb.s, &a1)
                                : find_bin(m1, kBins1, target - a_meas, sb.s, &a1);
        a_mass += BY_COUNT ? sum_above(m1, kBins1, b1, sb.s) : a1;
        a_meas += a1;
        prefix = (prefix << 10) | (uint32_t)b1;
        count = h1.count(b1);
    }
    if (count <= (u64)kMaxCand) {
        const int nc = gather_sorted(row, shift, prefix, prefix, sb);
        int q;
        u64 before;
        if (BY_COUNT) {
            q = (int)(target - a_meas);
            before = sorted_mass(row, q, sb);
        } else {
            q = sorted_pick(row, nc, target - a_meas, sb, &before);
        }
        *ahead = a_mass + before;
        return q >= 0 && q < nc ? cand_index(sb.cand[q]) : -1;
    }
    // more than kMaxCand equal logits: they share one weight, so the entry is
    // the group's j-th in index order
    const uint32_t key = prefix;
    const u64 w = row.weight(key_value(key));
    const u64 j = BY_COUNT ? target - a_meas : (target - a_meas) / w;
    auto is_key = [&](float v) -> u64 { return v == v && order_key(v) == key ? 1ull : 0ull; };
    u64 mine = 0;
    row.each([&](int, float v) { mine += is_key(v); });
    u64 total;
    const u64 wc = warp_sum_u64(mine);
    const u64 ex = warp_exscan(wc, sb.s, &total);
    if (threadIdx.x == 0) sb.s.ri[2] = -1;
    __syncthreads();
    if (wc > 0 && ex <= j && j < ex + wc) {
        const int idx = warp_walk(row, j - ex, is_key);
        if (row.lane == 0) sb.s.ri[2] = idx;
    }
    __syncthreads();
    *ahead = a_mass + j * w;
    return sb.s.ri[2];
}

// Append the entries i0 + e of the row whose bits e are set in `in` (rare:
// kept out of the per-entry path, so that the common case is one compare
// and one OR per entry; each such entry is read again from cache).
template <int DT, bool VEC>
__device__ __forceinline__ void gather_bits(const Row<DT, VEC>& row, ShBig& sb, unsigned in, int i0) {
    while (in) {
        const int e = __ffs(in) - 1;
        in &= in - 1u;
        const float v = Store<DT>::load1(row.x, row.base + i0 + e);
        const unsigned slot = atomicAdd(&sb.s.ncand, 1u);
        if (slot < (unsigned)kMaxCand) sb.cand[slot] = cand_of(order_key(v), i0 + e);
    }
}

// The entries >= T of the row, gathered as candidates (unsorted; ncand
// counts them all, even past kMaxCand).
template <int DT, bool VEC>
__device__ void gather_ge(const Row<DT, VEC>& row, ShBig& sb, float T) {
    constexpr int V = Row<DT, VEC>::V;
    constexpr int kTile = Row<DT, VEC>::kTile;
    __syncthreads();
    if (threadIdx.x == 0) sb.s.ncand = 0;
    __syncthreads();
    if (VEC) {
        // the tile's maximum first; its entries only when it reaches T (rare)
        for (int j0 = row.last_group(); j0 >= row.s0; j0 -= kTile * kU) {
            Vec16 r[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) r[q] = row.load_raw(j0 + q * kTile);
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                if (vec_max<DT>(r[q]) >= T) {
                    float v[V];
                    Store<DT>::unpack(r[q], v);
                    gather_bits(row, sb, bits_ge(v, T), j0 + q * kTile + row.lane * V);
                }
            }
        }
    } else {
        for (int j0 = row.last_group(); j0 >= row.s0; j0 -= kTile * kU) {
            float v[kU][V];
#pragma unroll
            for (int q = 0; q < kU; ++q) row.load(j0 + q * kTile, v[q]);
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const unsigned in = bits_ge(v[q], T);
                if (in) gather_bits(row, sb, in, j0 + q * kTile + row.lane * V);
            }
        }
    }
}

// Top-p's second pass: this thread's share of the row's total mass (f32
// unit sums, each held in fixed point, as the index-order kernel sums it),
// and every entry >= T gathered as a candidate (unsorted; ncand counts them
// all, even past kMaxCand).
template <int DT, bool VEC>
__device__ u64 mass_and_gather(const Row<DT, VEC>& row, ShBig& sb, float T) {
    constexpr int V = Row<DT, VEC>::V;
    constexpr int kTile = Row<DT, VEC>::kTile;
    __syncthreads();
    if (threadIdx.x == 0) sb.s.ncand = 0;
    __syncthreads();
    MassAcc acc;
    for (int j0 = row.last_group(); j0 >= row.s0; j0 -= kTile * kU) {
        if (VEC) {
            Vec16 r[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) r[q] = row.load_raw(j0 + q * kTile);
#pragma unroll
            for (int q = 0; q < kU; q += 2) {  // two units at a time
                float2 su;
                if (DT == kBF16) {
                    su = unit_sums2_bf16<DT, VEC>(row, r[q], r[q + 1]);
                } else {
                    float v0[V], v1[V];
                    Store<DT>::unpack(r[q], v0);
                    Store<DT>::unpack(r[q + 1], v1);
                    su = unit_sums2<DT, VEC>(row, v0, v1);
                }
                // a unit holding NaN, summed again from its packed tile (rare)
                if (su.x != su.x) su.x = unit_sum_of<DT, VEC>(row, r[q]);
                if (su.y != su.y) su.y = unit_sum_of<DT, VEC>(row, r[q + 1]);
                acc.add(su.x);
                acc.add(su.y);
                // the tile's maximum first; its entries >= T only when it reaches T (rare)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (vec_max<DT>(r[q + h]) >= T) {
                        float v[V];
                        Store<DT>::unpack(r[q + h], v);
                        gather_bits(row, sb, bits_ge(v, T), j0 + (q + h) * kTile + row.lane * V);
                    }
                }
            }
        } else {
            float v[kU][V];
#pragma unroll
            for (int q = 0; q < kU; ++q) row.load(j0 + q * kTile, v[q]);
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                acc.add(unit_sum(row, v[q]));
                const unsigned in = bits_ge(v[q], T);
                if (in) gather_bits(row, sb, in, j0 + q * kTile + row.lane * V);
            }
        }
        acc.fold();
    }
    return acc.total();
}

// Row ri, the whole of it by this CTA (all kT threads): top-k and top-p.
template <int DT, bool VEC>
__device__ void descending_row(const void* x, int32_t* out, int64_t ri, int n, int method, float t, int k, float p,
                               Draws d, ShBig& sb) {
    Row<DT, VEC> row;
    setup(row, x, n, t, ri, 0, 1);
    seed_uniform(d, ri, sb.s);
    int nv;
    row.mx = block_first_max<false>(row, sb.s, &nv, sb.lmax);
    if (!accept_max(row, out, ri, threadIdx.x == 0)) return;
    const float ur = row_uniform(d, ri, sb.s);
    // The head of the row: the first-digit bins from that of M - 24 / c down
    // -- every entry of weight above 2^-24 of the largest (and some below).
    // The rest of a row of n entries weighs at most n 2^-24 of the largest, so
    // for the vocabularies in use the head carries the top-p cut of any p up
    // to 0.99 and the top k of a moderate k; otherwise the whole row is
    // histogrammed.
    const uint32_t head = order_key(__fsub_rn(row.mx, __fdiv_rn(24.0f, row.c))) >> 20;
    auto c0 = [&](int b) { return sb.h0().count(b); };
    auto m0 = [&](int b) { return sb.h0().mass(b); };
    if (method == kTopK) {
        if (k <= kT) {
            // the entries >= a floor that k entries reach hold the top k (or
            // every number, when the floor is -inf)
            const float T = maxima_floor(sb.lmax[threadIdx.x], (k + kW - 1) / kW, sb.s);
            gather_ge(row, sb, T);
            __syncthreads();  // every candidate is in
            const unsigned ncand = sb.s.ncand;
            if (ncand <= (unsigned)kWarpCand) {
                rank_sort(sb.cand, sb.cand + kWarpCand, (int)ncand);
                __syncthreads();
                if (threadIdx.x < 32) {  // one warp finishes the row
                    WarpSorted ws;
                    warp_weigh(row, sb.cand + kWarpCand, (int)ncand, row.lane, ws);
                    const int L = min(k, (int)ncand);
                    const u64 wk = warp_mass_through(ws, L);
                    u64 before, c;
                    const int q = warp_first_above(row, ws, L, scaled(ur, wk), row.lane, &before, &c);
                    if (threadIdx.x == 0) out[ri] = q >= 0 ? cand_index(c) : -1;
                }
                return;
            }
            const int nc = sort_cand(sb);
            if (sb.s.ncand <= (unsigned)kMaxCand) {
                const int L = min(k, nc);
                const u64 wk = sorted_mass(row, L, sb);
                u64 unused;
                const int q = sorted_pick(row, L, scaled(ur, wk), sb, &unused);
                if (threadIdx.x == 0) out[ri] = q >= 0 ? cand_index(sb.cand[q]) : -1;
                return;
            }
        }
        // more candidates than the gather holds: count the head's bins first
        {
            build_first(row, sb, head, false, false);
            const u64 in_head = sum_above(c0, kBins0, -1, sb.s);
            if (in_head >= (u64)k) {
                // the bin of the k-th entry; gather it and every bin above
                u64 above;
                const int b = find_bin(c0, kBins0, (u64)(k - 1), sb.s, &above);
                if (above + sb.cnt0[b] <= (u64)kMaxCand) {
                    gather_sorted(row, 20, (uint32_t)b, (uint32_t)(kBins0 - 1), sb);
                    const u64 wk = sorted_mass(row, k, sb);
                    u64 unused;
                    const int q = sorted_pick(row, k, scaled(ur, wk), sb, &unused);
                    if (threadIdx.x == 0) out[ri] = q >= 0 ? cand_index(sb.cand[q]) : -1;
                    return;
                }
            }
        }
        u64 all;
        block_exscan(build_first(row, sb, 0u, true, true), sb.s, &all);
        nv = (int)sum_above(c0, kBins0, -1, sb.s);  // the count of numbers
        u64 kept = all;
        if (k < nv) desc_search<DT, VEC, true>(row, (u64)k, sb, &kept);  // the entry past the k-th
        u64 unused;
        const int idx = desc_search<DT, VEC, false>(row, scaled(ur, kept), sb, &unused);
        if (threadIdx.x == 0) out[ri] = idx;
        return;
    }
    // top-p: keep the prefix whose running mass stays <= p * W (the first
    // entry always), then draw from it.  First try the top of the row: the
    // entries >= a floor that at least kTopLanes entries reach (from the
    // threads' own maxima), gathered in the same pass that sums the row's
    // mass, and sorted; when their exact mass passes the cut, the cut and the
    // draw both fall among them.
    const float T = maxima_floor(sb.lmax[threadIdx.x], kTopLanes / kW, sb.s);
    u64 all;
    block_exscan(mass_and_gather(row, sb, T), sb.s, &all);
    const unsigned ncand = sb.s.ncand;  // final: block_exscan's barriers follow every atomic
    const u64 cut = (u64)((double)p * (double)all);
    u64 kept = all, unused;
    int idx = -1;
    bool ok = false;
    u64 top_mass = 0;  // the gathered candidates' mass (order-free: any thread order)
    if (ncand <= (unsigned)kWarpCand) {
        u64 mine = 0;
        for (int j = threadIdx.x; j < (int)ncand; j += kT) mine += row.weight(key_value((uint32_t)(sb.cand[j] >> 32)));
        block_exscan(mine, sb.s, &top_mass);
    }
    // The candidates settle the row when the cut lies below their mass (the
    // draw then does too), or, with no cut, when the draw does.
    const bool settles = ncand <= (unsigned)kWarpCand && (cut < all ? cut < top_mass : scaled(ur, all) < top_mass);
    if (settles) {
        rank_sort(sb.cand, sb.cand + kWarpCand, (int)ncand);
        __syncthreads();
        // one warp finishes the row; the others are done
        if (threadIdx.x < 32) {
            WarpSorted ws;
            warp_weigh(row, sb.cand + kWarpCand, (int)ncand, row.lane, ws);
            u64 kp = all, before, c;
            if (cut < all) {
                warp_first_above(row, ws, (int)ncand, cut, row.lane, &kp, &c);
                if (kp == 0) kp = 1;  // a target of 0 lands on the first entry
            }
            const int q = warp_first_above(row, ws, (int)ncand, scaled(ur, kp), row.lane, &before, &c);
            if (threadIdx.x == 0) out[ri] = q >= 0 ? cand_index(c) : -1;
        }
        return;
    }
    unsigned nc2 = ncand;
    if (ncand <= (unsigned)kWarpCand) {
        // the few did not settle the row: a second, wider round, the entries
        // >= a floor that twice as many entries per warp reach (sorted by the
        // block, up to kMaxCand of them)
        gather_ge(row, sb, maxima_floor(sb.lmax[threadIdx.x], 2 * (kTopLanes / kW), sb.s));
        __syncthreads();  // every candidate is in
        nc2 = sb.s.ncand;
    }
    if (nc2 <= (unsigned)kMaxCand) {
        const int nc = sort_cand(sb);
        const u64 top_mass = sorted_mass(row, nc, sb);
        if (cut < all) {
            if (cut < top_mass) {
                sorted_pick(row, nc, cut, sb, &kept);
                if (kept == 0) kept = 1;  // a target of 0 lands on the first entry
                ok = true;
            }
        } else {
            ok = true;
        }
        const u64 target = scaled(ur, kept);
        if (ok && target < top_mass) {
            const int q = sorted_pick(row, nc, target, sb, &unused);
            idx = q >= 0 ? cand_index(sb.cand[q]) : -1;
        } else {
            ok = false;
        }
    }
    if (!ok) {  // the exact digit histograms of the whole row, with its own total
        build_first(row, sb, 0u, true, false);
        const u64 exact = sum_above(m0, kBins0, -1, sb.s);
        const u64 cut_x = (u64)((double)p * (double)exact);
        kept = exact;
        if (cut_x < exact) {
            desc_search<DT, VEC, false>(row, cut_x, sb, &kept);
            if (kept == 0) kept = 1;
        }
        idx = desc_search<DT, VEC, false>(row, scaled(ur, kept), sb, &unused);
    }
    if (threadIdx.x == 0) out[ri] = idx;
}

// MINB: CTAs an SM the register budget is compiled for (2: batches of many
// rows; 1: at most one row per SM).
template <int DT, bool VEC, int MINB = 2>
__global__ void __launch_bounds__(kT, MINB)
sample_descending(const void* x, int32_t* out, int n, int method, float t, int k, float p, Draws d) {
    pdl_begin();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ShBig& sb = *reinterpret_cast<ShBig*>(smem_raw);
    descending_row<DT, VEC>(x, out, blockIdx.x, n, method, t, k, p, d, sb);
}

template <int DT, bool VEC>
cudaError_t launch_vec(const void* x, int32_t* out, int64_t rows, int n, int method, float t, int k, float p,
                       Draws d, cudaStream_t st) {
    if (method == kTemperature) return launch_index_order<DT, VEC, false>(x, out, rows, n, t, p, d, st);
    if (method == kMinP) return launch_index_order<DT, VEC, true>(x, out, rows, n, t, p, d, st);
    const size_t smem = sizeof(ShBig);
    // the shared-memory opt-in, once per device for each form
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
    const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (!(opted.load(std::memory_order_acquire) & bit) || bit == 0) {
        cudaError_t e =
            cudaFuncSetAttribute(sample_descending<DT, VEC, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sample_descending<DT, VEC, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return e;
        }
        opted.fetch_or(bit, std::memory_order_release);
    }
    // a batch of at most one row per SM (decode): the form compiled for one
    // CTA an SM (96 registers where the two-CTA form has 64), the same code
    // and results (decode top-k / top-p 24.0 -> 23.0, 29.3 -> 28.2 us)
    if (rows <= (int64_t)sm_count())
        return launch(sample_descending<DT, VEC, 1>, dim3((unsigned)rows), dim3(kT), smem, st, x, out, n, method, t, k,
                      p, d);
    return launch(sample_descending<DT, VEC, 2>, dim3((unsigned)rows), dim3(kT), smem, st, x, out, n, method, t, k, p,
                  d);
}

template <int DT>
cudaError_t launch_dt(const void* x, int32_t* out, int64_t rows, int n, int method, float t, int k, float p,
                      Draws d, bool vec, cudaStream_t st) {
    if (vec) return launch_vec<DT, true>(x, out, rows, n, method, t, k, p, d, st);
    return launch_vec<DT, false>(x, out, rows, n, method, t, k, p, d, st);
}

// u[i] = the uniform of draw offset + i of the seeded stream: each warp jumps
// to its first draw together, then lane l steps l draws further.
__global__ void __launch_bounds__(256) pcg64_uniforms(float* u, int64_t n, u64 seed, u64 offset) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * 8;
    for (int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); w * 32 < n; w += warps) {
        const int64_t i0 = w * 32;
        // draw i0 is i0 + 1 steps after the seeded state
        const pcg::Affine f = pcg::jump_warp(pcg::add128(pcg::U128{offset, 0}, pcg::U128{(u64)i0 + 1, 0}));
        const pcg::U128 s = pcg::apply(pcg::jump_small((uint32_t)lane), pcg::apply(f, pcg::seeded(seed)));
        if (i0 + lane < n) u[i0 + lane] = pcg::uniform_of(pcg::output(s));
    }
}

}  // namespace

cudaError_t launch_pcg64_uniforms(float* u, int64_t n, unsigned long long seed, unsigned long long offset,
                                  cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
    return launch(pcg64_uniforms, dim3((unsigned)blocks), dim3(256), 0, st, u, n, (u64)seed, (u64)offset);
}

cudaError_t launch_sample(const void* x, int32_t* out, int64_t rows, int64_t n, int method, float t, int64_t k,
                          float p, Draws d, int dtype, bool vec, cudaStream_t st) {
    if (method == kGreedy) return launch_argmax(x, out, rows, n, dtype, vec, st);
    const int ki = (int)(k > n ? n : k), ni = (int)n;
    if (dtype == kF32) return launch_dt<kF32>(x, out, rows, ni, method, t, ki, p, d, vec, st);
    return launch_dt<kBF16>(x, out, rows, ni, method, t, ki, p, d, vec, st);
}

}  // namespace gbe
