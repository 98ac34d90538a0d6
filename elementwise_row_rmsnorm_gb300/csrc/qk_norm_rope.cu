// qk_norm_rope.cu -- QK-norm followed by RoPE, in one pass, on sm_103a.
//
// Definition ("Operations", section 5, QK-norm): before RoPE, every head of
// q and of k is RMS-normalised on its own -- the mean of squares runs over
// head_dim, not over heads x head_dim -- with a gain of [head_dim] (g_q for
// q, g_k for k); then q and k are rotated as gbe_rope defines
// ("Elementwise kernels in C", section 2.2; "Operations", section 3).
//
// The fused pass equals the unfused composition bit for bit: gbe_rmsnorm
// over the T*H head rows (d = head_dim), the result stored in the storage
// type, then gbe_rope / gbe_rope_qk on the stored values.  To get there:
//  * a head row is reduced with the very tree gbe_rmsnorm uses for d =
//    head_dim: lane c of a row sums chunk c (one 16-byte vector, in element
//    order, fused multiply-add) and the lanes are combined by a butterfly.
//    gbe_rmsnorm puts such rows on one warp whose lanes past the last chunk
//    hold zero; a butterfly over the W = next power of two >= chunks lanes
//    adds exactly the same values (the wider steps only add +0), so several
//    rows can share a warp;
//  * the normalised value is rounded to the storage type before the
//    rotation reads it, as a stored intermediate would be;
//  * the angles are float(p) * omega_i and rope_sincos (or the same values
//    from the cos/sin table), as in rope.cu.
//
// Map: one CTA per token (qk_norm_rope_pair and qk_norm_rope_tok, aligned
// rows), a warp per chunk of the token's head rows of q or k; the token's
// angles are formed once into shared memory.  Unaligned rows take
// qk_norm_rope_kernel: a warp per chunk of head rows that stages the
// normalised rows in shared memory (so a lane can read the partner of each
// of its entries).  Head rows of 33 to 64 chunks (f32 head_dim up to 256,
// bf16 up to 512) take qk_norm_rope_wide: a warp per row, two chunks a lane.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kWarps = 4;   // warps (tokens) per CTA
constexpr int kPasses = 4;      // head-row passes whose loads are in flight together
constexpr int kPassesShfl = 4;  // the same for the shuffle path (eight measured slower: fewer warps per SM)
constexpr int kMaxRow = 256;  // floats of one warp's staging: 32 chunks of <= 8 entries

struct QkSide {
    const char* x;
    char* y;
    const char* g;
    int64_t xs, ys;  // token strides in elements
    int H;
};

template <int DT, bool VEC>
__device__ __forceinline__ void load_chunk(const char* row, int c, int D, float (&f)[Store<DT>::V]) {
    using S = Store<DT>;
    constexpr int V = S::V;
    if (VEC) {
        S::unpack(ld_stream(row + (int64_t)c * 16), f);
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e) f[e] = c * V + e < D ? S::load1(row, (int64_t)c * V + e) : 0.0f;
    }
}

// A load kept in L1 for a second read by the same warp (ld.global.ca: a
// coherent load, so rows written in place by this kernel are never read
// stale -- each address is read twice and then written once, by one warp).
__device__ __forceinline__ Vec16 ld_twice(const void* p) {
    Vec16 v;
    asm volatile("ld.global.ca.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}

// Aligned rows whose pair partners lie a whole number of chunks apart (the
// half layout with r/2 a multiple of the vector, or the interleaved layout
// with r a multiple of it).  One CTA per token, one warp per chunk of R * 4
// head rows of q or k (a warp loops when the token has more chunks than
// warps).  The token's r/2 angles are formed once, one pair per thread,
// while the head rows' loads are in flight, and read back from shared memory
// after one CTA barrier, which a warp reaches once its first rows are reduced
// (so no warp idles there while the angles are formed).  A lane's partner
// chunk is fetched from the partner
// lane with four register shuffles (half layout), or sits in the lane's own
// chunk (interleaved).
//
// The four rows' sums of squares are reduced by a transposed butterfly: at
// the step of distance W/2 a lane keeps two of its four rows and hands the
// other two to its partner, at distance W/4 it keeps one, and the remaining
// steps reduce that one.  Each addition is the one the per-row butterfly
// does (own partial + partner partial, the same pairs, the same order), so
// every total is bit-identical to gbe_rmsnorm's; each lane then takes the
// reciprocal root of its one row and shuffles the other three in.
constexpr int kTokWarps = 16;  // most warps of one token's CTA
constexpr int kMaxHalf = 128;  // r/2 <= 128: head_dim <= 256

// Where angle i sits in the token's cos (or sin) table.  QPL = 2 (a lane
// reads two quads, bf16 half layout): quad s of the lane whose angles start
// at 8a sits at s * half/2 + 4a, so the eight lanes of one shared-memory
// phase read 128 contiguous bytes.  Otherwise angle i sits at i.
template <int QPL>
__device__ __forceinline__ int angle_slot(int i, int half) {
    if (QPL == 2) return ((i & 7) >> 2) * (half >> 1) + (i >> 3) * 4 + (i & 3);
    return i;
}

// A shared-memory load the compiler keeps where it stands (volatile): the
// angles are re-read in every pass instead of held in sixteen registers.
__device__ __forceinline__ float4 lds4(const float* p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"((unsigned)__cvta_generic_to_shared(p)));
    return v;
}
__device__ __forceinline__ float2 lds2(const float* p) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"((unsigned)__cvta_generic_to_shared(p)));
    return v;
}

template <int DT, int LAYOUT, bool CACHE>
__global__ void __launch_bounds__(kTokWarps * 32, 2)
qk_norm_rope_tok(QkSide A, QkSide B, int nca, int ncb, float eps, const int32_t* pos, int D, int r,
                 const float* inv_freq, const float2* cache, int64_t cache_len, float mu, int W) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    constexpr int NP = kPassesShfl;
    constexpr int NA = LAYOUT == 0 ? V : V / 2;  // angles of one lane's chunk
    constexpr int QPL = NA >= 8 ? 2 : 1;          // 16-byte quads of them (NA = 2: one 8-byte pair)
    __shared__ __align__(16) float cs_cos[kMaxHalf];
    __shared__ __align__(16) float cs_sin[kMaxHalf];
    __shared__ __align__(16) float cs_nsin[LAYOUT == 0 ? kMaxHalf : 1];  // -sin, for first members
    pdl_begin();
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int64_t t = blockIdx.x;
    const int per_tok = nca + ncb;
    const int nchunks = D / V;
    const int R = 32 / W;
    const int sub = lane / W;
    const int c = lane - sub * W;
    const bool has = c < nchunks;
    const int half = r >> 1;
    const int G = half / V;  // chunks between pair members (half layout)
    const int32_t p = pos[t];

    // the first item's loads go out before anything else
    int ci = wib;
    Vec16 raw[NP];
    auto load_item = [&](int item) {
        const bool second = item >= nca;
        const QkSide& Q = second ? B : A;
        const int h0 = (second ? item - nca : item) * R * NP;
        const char* xt = Q.x + t * Q.xs * ES;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const int h = h0 + k * R + sub;
            raw[k] = Vec16{{0u, 0u, 0u, 0u}};
            if (has && h < Q.H) raw[k] = ld_stream(xt + ((int64_t)h * D + (int64_t)c * V) * ES);
        }
    };
    if (ci < per_tok) load_item(ci);

    // the token's angles, one pair per thread
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        float cv, sv;
        if (CACHE && p >= 0 && p < cache_len) {
            const float2 v = __ldg(cache + (int64_t)p * half + i);
            cv = v.x;
            sv = v.y;
        } else {
            rope_sincos(__fmul_rn((float)p, __ldg(inv_freq + i)), &sv, &cv);
        }
        const int slot = angle_slot<QPL>(i, half);
        cs_cos[slot] = cv;
        cs_sin[slot] = sv;
        if (LAYOUT == 0) cs_nsin[slot] = -sv;
    }

    const bool rot = has && c * V < r;  // this chunk is rotated
    const bool first_half = LAYOUT == 0 && c < G;
    const int src = LAYOUT == 0 ? (c < G ? lane + G : (c < 2 * G ? lane - G : lane)) : lane;
    // the starting angle of this lane's chunk, and its quads in the table
    const int ib = LAYOUT == 0 ? (first_half ? c : c - G) * V : c * (V / 2);
    int slot0 = 0;
    if (rot) slot0 = angle_slot<QPL>(ib, half);
    const float* tc = cs_cos + slot0;
    const float* tsn = (LAYOUT == 0 && first_half ? cs_nsin : cs_sin) + slot0;

    for (; ci < per_tok; ci += nw) {
        if (ci != wib) load_item(ci);
        const bool second = ci >= nca;
        const QkSide& Q = second ? B : A;
        const int h0 = (second ? ci - nca : ci) * R * NP;
        char* yt = Q.y + t * Q.ys * ES;
        float gv[V];
        if (has) S::unpack(ld_reuse(Q.g + (int64_t)c * 16), gv);

        // sums of squares of the four rows this lane holds a chunk of
        float s[NP];
#pragma unroll
        for (int k = 0; k < NP; ++k) s[k] = vec_sq_acc<DT>(raw[k], 0.0f);  // zero for absent rows and chunks
        float inv[NP];
        if (W >= 4) {
            const int m1 = W >> 1, m2 = W >> 2;
            const bool b1 = (lane & m1) != 0, b2 = (lane & m2) != 0;
            float k0 = b1 ? s[2] : s[0], k1 = b1 ? s[3] : s[1];
            const float g0 = b1 ? s[0] : s[2], g1 = b1 ? s[1] : s[3];
            k0 = __fadd_rn(k0, __shfl_xor_sync(0xFFFFFFFFu, g0, m1));
            k1 = __fadd_rn(k1, __shfl_xor_sync(0xFFFFFFFFu, g1, m1));
            float kk = b2 ? k1 : k0;
            const float gg = b2 ? k0 : k1;
            kk = __fadd_rn(kk, __shfl_xor_sync(0xFFFFFFFFu, gg, m2));
            for (int m = W >> 3; m >= 1; m >>= 1) kk = __fadd_rn(kk, __shfl_xor_sync(0xFFFFFFFFu, kk, m));
            // this lane's row is pass 2*b1 + b2
            const float own = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(kk, (float)D), eps)));
            const int base = sub * W;
#pragma unroll
            for (int k = 0; k < NP; ++k)
                inv[k] = __shfl_sync(0xFFFFFFFFu, own, base + ((k >> 1) ? m1 : 0) + ((k & 1) ? m2 : 0));
        } else {
            for (int m = W >> 1; m >= 1; m >>= 1) {
#pragma unroll
                for (int k = 0; k < NP; ++k) s[k] = __fadd_rn(s[k], __shfl_xor_sync(0xFFFFFFFFu, s[k], m));
            }
#pragma unroll
            for (int k = 0; k < NP; ++k)
                inv[k] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s[k], (float)D), eps)));
        }
        // the angles are in once every thread has passed here; each warp's
        // first item comes through (there are no more warps than items), so
        // every thread of the CTA arrives exactly once
        if (ci == wib) __syncthreads();

#pragma unroll
        for (int k = 0; k < NP; ++k) {
            if (h0 + k * R >= Q.H) break;  // uniform across the warp
            const int h = h0 + k * R + sub;
            const bool live = has && h < Q.H;
            float n[V];
            S::unpack(raw[k], n);
#pragma unroll
            for (int e = 0; e < V; ++e) n[e] = __fmul_rn(__fmul_rn(n[e], inv[k]), gv[e]);
            const Vec16 nv = S::pack(n);  // the stored (rounded) normalised chunk
            S::unpack(nv, n);
            float o[V], m2[V];
            if (LAYOUT == 0) {
                Vec16 pv;
#pragma unroll
                for (int q = 0; q < 4; ++q) pv.w[q] = __shfl_sync(0xFFFFFFFFu, nv.w[q], src);
                S::unpack(pv, m2);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) m2[e] = n[e ^ 1];
            }
            // The angles of this lane's entries.  Both members of a pair take
            // one formula, out = mu * (own * cos + partner * sg), sg = -sin for
            // the first member and +sin for the second: IEEE gives a - b ==
            // a + (-b) and a + b == b + a exactly, so this is the same
            // arithmetic as mu * (a cos - b sin) and mu * (a sin + b cos).  A
            // first-half lane (half layout) reads the negated sines; in the
            // interleaved layout the even entries are the first members.
            float ac[NA], as[NA];
#pragma unroll
            for (int q = 0; q < QPL; ++q) {
                if (NA >= 4) {
                    const float4 vc = lds4(tc + q * (half >> 1));
                    const float4 vs = lds4(tsn + q * (half >> 1));
                    ac[4 * q] = vc.x; ac[4 * q + 1] = vc.y; ac[4 * q + 2] = vc.z; ac[4 * q + 3] = vc.w;
                    as[4 * q] = vs.x; as[4 * q + 1] = vs.y; as[4 * q + 2] = vs.z; as[4 * q + 3] = vs.w;
                } else {
                    const float2 vc = lds2(tc);
                    const float2 vs = lds2(tsn);
                    ac[0] = vc.x; ac[1] = vc.y;
                    as[0] = vs.x; as[1] = vs.y;
                }
            }
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const float ce = LAYOUT == 0 ? ac[e] : ac[e >> 1];
                const float se = LAYOUT == 0 ? as[e] : ((e & 1) ? as[e >> 1] : -as[e >> 1]);
                o[e] = rot ? __fmul_rn(mu, __fadd_rn(__fmul_rn(n[e], ce), __fmul_rn(m2[e], se))) : n[e];
            }
            if (live) st_stream(yt + ((int64_t)h * D + (int64_t)c * V) * ES, S::pack(o));
        }
    }
}

// Both members of one lane's pairs rotated and stored: lo = mu (a cos - b
// sin), hi = mu (a sin + b cos), each product, sum and the scale rounded on
// its own as gbe_rope does, one quad of pairs at a time (its cos and sin read
// from shared memory then).  MU false: mu is 1, and 1 * x == x for every
// value the sum can take (-0, infinities and NaN included), so the scale is
// left out.
template <int DT, bool MU>
__device__ __forceinline__ void rotate_store(const float (&a)[Store<DT>::V], const float (&b)[Store<DT>::V],
                                             const float* tc, const float* ts, int qstride, float mu, char* lo_at,
                                             char* hi_at) {
    using S = Store<DT>;
    constexpr int V = S::V;
    float lo[V], hi[V];
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
        const float4 vc = lds4(tc + q * qstride);
        const float4 vs = lds4(ts + q * qstride);
        const float c4[4] = {vc.x, vc.y, vc.z, vc.w};
        const float s4[4] = {vs.x, vs.y, vs.z, vs.w};
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            // the products two lanes at a time; the sums scalar (a packed
            // multiply feeding a packed add may be fused into one rounding)
            const int e = 4 * q + j;
            const float2 A = make_float2(a[e], a[e + 1]), B = make_float2(b[e], b[e + 1]);
            const float2 C = make_float2(c4[j], c4[j + 1]), Sn = make_float2(s4[j], s4[j + 1]);
            const float2 ac = mul2_rn(A, C), bs = mul2_rn(B, Sn), as = mul2_rn(A, Sn), bc = mul2_rn(B, C);
            float2 l = make_float2(__fsub_rn(ac.x, bs.x), __fsub_rn(ac.y, bs.y));
            float2 h = make_float2(__fadd_rn(as.x, bc.x), __fadd_rn(as.y, bc.y));
            if (MU) {
                l = mul2_rn(make_float2(mu, mu), l);
                h = mul2_rn(make_float2(mu, mu), h);
            }
            lo[e] = l.x;
            lo[e + 1] = l.y;
            hi[e] = h.x;
            hi[e + 1] = h.y;
        }
    }
    st_stream(lo_at, S::pack(lo));
    st_stream(hi_at, S::pack(hi));
}

// Half layout, the whole head rotated (r = head_dim), a power-of-two number
// of chunks (2 to 32): a lane holds chunk c of the first half of a head row
// and chunk c + L of the second half (L = chunks / 2), so both members of
// every pair it rotates sit in its own registers -- no exchange between
// lanes.  gbe_rmsnorm's tree for such a row first adds the sums of chunks c
// and c + L (its butterfly step of distance L, chunk c's sum first): here
// that step is an addition inside the lane, and the remaining steps run
// over the L lanes of the row.  Rows: 32 / L per pass, NP passes per warp
// item, whose sums share the butterfly transposed (NP = 2: at distance L/2
// a lane keeps one pass and hands the other to its partner; NP = 4, L >= 4:
// at L/2 it keeps two of four, at L/4 one, as in qk_norm_rope_tok), so one
// reciprocal root per lane serves NP rows.  One CTA per token, the token's
// angles formed once into shared memory, as in qk_norm_rope_tok.
//
// NP = 4 (the compile-time row sizes) halves the per-item work of the two-pass
// form (addresses, the root, the butterfly): 1987 warp instructions per
// token against 2325 at [8192, 32+8, 128] bf16.  Four passes of rows do not
// fit beside the angle code in the 64 registers a thread has here (bounds
// of two 512-thread CTAs an SM: more registers cost more in occupancy than
// they save), so these loads go out after the angles are formed, kept in L1
// (ld_twice), and each pass reads its rows again from L1 for the
// normalisation instead of holding them from the sums.  So that the loads
// do not start only after the position's load and the angles, every lane
// first asks for one 128-byte line of the item's rows to be fetched into
// L2 (a prefetch holds no register): 29.3 -> 27.6 us at that shape.
//
// D = 2 L V is a power of two here, so the mean of squares s / D is taken as
// s * 2^-log2(D): both are the correctly rounded value of the same real
// number, so the bits are those of gbe_rmsnorm's division.  LGL >= 0 fixes
// log2(L) at compile time (the common head sizes); -1 reads it from lgL_arg.
template <int DT, bool CACHE, int LGL, int NP>
__global__ void __launch_bounds__(kTokWarps * 32, 2)
qk_norm_rope_pair(QkSide A, QkSide B, int nca, int ncb, float eps, const int32_t* pos, int lgL_arg,
                  const float* inv_freq, const float2* cache, int64_t cache_len, float mu) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int LGV = V == 8 ? 3 : 2;
    constexpr int64_t ES = sizeof(typename S::T);
    constexpr int QPL = V >= 8 ? 2 : 1;  // 16-byte quads of one lane's angles
    __shared__ __align__(16) float cs_cos[kMaxHalf];
    __shared__ __align__(16) float cs_sin[kMaxHalf];
    pdl_begin();
    const int lgL = LGL >= 0 ? LGL : lgL_arg;
    const int D = V << (lgL + 1);
    const float rD = __int_as_float((127 - (LGV + 1 + lgL)) << 23);  // 1 / D, exact
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int64_t t = blockIdx.x;
    const int per_tok = nca + ncb;
    const int L = 1 << lgL;    // lanes of one head row
    const int RP = 32 >> lgL;  // head rows per pass
    const int sub = lane >> lgL;
    const int c = lane & (L - 1);
    const int half = D >> 1;  // L * V
    const int32_t p = pos[t];

    constexpr int64_t kPassBytes = 64 * V * ES;  // RP * D entries: the rows of one pass
    static_assert(NP == 2 || (NP == 4 && LGL >= 2), "four passes need four or more lanes per row");
    int ci = wib;
    Vec16 raw[NP][2];
    auto load_item = [&](int item) {
        const bool second = item >= nca;
        const int H = second ? B.H : A.H;
        const int h = (second ? item - nca : item) * RP * NP + sub;
        const char* row = (second ? B.x : A.x) + (t * (second ? B.xs : A.xs) + (int64_t)h * D) * ES + c * 16;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            raw[k][0] = raw[k][1] = Vec16{{0u, 0u, 0u, 0u}};
            if (h + k * RP < H) {
                if (NP == 4) {
                    raw[k][0] = ld_twice(row + k * kPassBytes);
                    raw[k][1] = ld_twice(row + k * kPassBytes + half * ES);
                } else {
                    raw[k][0] = ld_stream(row + k * kPassBytes);
                    raw[k][1] = ld_stream(row + k * kPassBytes + half * ES);
                }
            }
        }
    };
    if (NP == 2 && ci < per_tok) load_item(ci);  // four passes: after the angles
    if (NP == 4 && ci < per_tok) {
        // the first item's rows (RP NP whole rows, contiguous: 256 V ES =
        // 4 KB, one 128-byte line a lane; those past H left out) start coming
        // into L2 while the angles form, so the loads after them wait for L2
        // rather than for DRAM
        const bool second = ci >= nca;
        const int h0 = (second ? ci - nca : ci) * RP * NP;
        const int64_t off = (int64_t)lane * 128;
        if (off < (int64_t)((second ? B.H : A.H) - h0) * D * ES)
            prefetch_l2((second ? B.x : A.x) + (t * (second ? B.xs : A.xs) + (int64_t)h0 * D) * ES + off);
    }

    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        float cv, sv;
        if (CACHE && p >= 0 && p < cache_len) {
            const float2 v = __ldg(cache + (int64_t)p * half + i);
            cv = v.x;
            sv = v.y;
        } else {
            rope_sincos(__fmul_rn((float)p, __ldg(inv_freq + i)), &sv, &cv);
        }
        const int slot = angle_slot<QPL>(i, half);
        cs_cos[slot] = cv;
        cs_sin[slot] = sv;
    }
    const int slot0 = angle_slot<QPL>(c * V, half);
    const bool mu_one = mu == 1.0f;

    for (; ci < per_tok; ci += nw) {
        if (NP == 4 || ci != wib) load_item(ci);
        const bool second = ci >= nca;
        const int H = second ? B.H : A.H;
        const int h0 = (second ? ci - nca : ci) * RP * NP;
        const char* gp = (second ? B.g : A.g) + c * 16;
        char* const yrow = (second ? B.y : A.y) + (t * (second ? B.ys : A.ys) + (int64_t)(h0 + sub) * D) * ES + c * 16;
        const char* const xrow = (second ? B.x : A.x) + (t * (second ? B.xs : A.xs) + (int64_t)(h0 + sub) * D) * ES + c * 16;

        // the sum of squares of each chunk in element order, then the
        // butterfly step of distance L inside the lane
        float s[NP];
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const float s0 = vec_sq_acc<DT>(raw[k][0], 0.0f), s1 = vec_sq_acc<DT>(raw[k][1], 0.0f);
            s[k] = __fadd_rn(s0, s1);
        }
        float inv[NP];
        if (NP == 4) {  // L >= 4
            const int m1 = L >> 1, m2 = L >> 2;
            const bool b1 = (lane & m1) != 0, b2 = (lane & m2) != 0;
            float k0 = b1 ? s[2 % NP] : s[0], k1 = b1 ? s[3 % NP] : s[1];
            const float g0 = b1 ? s[0] : s[2 % NP], g1 = b1 ? s[1] : s[3 % NP];
            k0 = __fadd_rn(k0, __shfl_xor_sync(0xFFFFFFFFu, g0, m1));
            k1 = __fadd_rn(k1, __shfl_xor_sync(0xFFFFFFFFu, g1, m1));
            float kk = b2 ? k1 : k0;
            const float gg = b2 ? k0 : k1;
            kk = __fadd_rn(kk, __shfl_xor_sync(0xFFFFFFFFu, gg, m2));
#pragma unroll
            for (int m = L >> 3; m >= 1; m >>= 1) kk = __fadd_rn(kk, __shfl_xor_sync(0xFFFFFFFFu, kk, m));
            // this lane's row is pass 2 * b1 + b2
            const float own = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(kk, rD), eps)));
            const int base = sub << lgL;
#pragma unroll
            for (int k = 0; k < NP; ++k)
                inv[k] = __shfl_sync(0xFFFFFFFFu, own, base + ((k >> 1) ? m1 : 0) + ((k & 1) ? m2 : 0));
        } else if (L >= 2) {
            const int m1 = L >> 1;
            const bool b1 = (lane & m1) != 0;
            float kk = b1 ? s[1 % NP] : s[0];
            const float gg = b1 ? s[0] : s[1 % NP];
            kk = __fadd_rn(kk, __shfl_xor_sync(0xFFFFFFFFu, gg, m1));
#pragma unroll
            for (int m = L >> 2; m >= 1; m >>= 1) kk = __fadd_rn(kk, __shfl_xor_sync(0xFFFFFFFFu, kk, m));
            const float own = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(kk, rD), eps)));
            const int base = sub << lgL;
            inv[0] = __shfl_sync(0xFFFFFFFFu, own, base);
            inv[1 % NP] = __shfl_sync(0xFFFFFFFFu, own, base + m1);
        } else {
#pragma unroll
            for (int k = 0; k < NP; ++k)
                inv[k] = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(s[k], rD), eps)));
        }
        // the angles are in once every thread has passed here; each warp's
        // first item comes through (there are no more warps than items), so
        // every thread of the CTA arrives exactly once
        if (ci == wib) __syncthreads();

#pragma unroll
        for (int k = 0; k < NP; ++k) {
            if (h0 + k * RP >= H) break;  // uniform across the warp
            float a[V], b[V], g[V];
            // normalised and rounded to storage, as a stored intermediate would be
            const float2 iv = make_float2(inv[k], inv[k]);
            // four passes: the rows are read again (from L1) rather than held;
            // a row past H contributes nothing and is not stored
            const bool here = h0 + k * RP + sub < H;
            Vec16 r0 = raw[k][0], r1 = raw[k][1];
            if (NP == 4) r0 = r1 = Vec16{{0u, 0u, 0u, 0u}};
            if (NP == 4 && here) {
                r0 = ld_twice(xrow + k * kPassBytes);
                r1 = ld_twice(xrow + k * kPassBytes + half * ES);
            }
            S::unpack(r0, a);
            S::unpack(ld_reuse(gp), g);
#pragma unroll
            for (int e = 0; e < V; e += 2) {
                const float2 u = mul2_rn(mul2_rn(make_float2(a[e], a[e + 1]), iv), make_float2(g[e], g[e + 1]));
                a[e] = S::round(u.x);
                a[e + 1] = S::round(u.y);
            }
            S::unpack(r1, b);
            S::unpack(ld_reuse(gp + half * ES), g);
#pragma unroll
            for (int e = 0; e < V; e += 2) {
                const float2 u = mul2_rn(mul2_rn(make_float2(b[e], b[e + 1]), iv), make_float2(g[e], g[e + 1]));
                b[e] = S::round(u.x);
                b[e + 1] = S::round(u.y);
            }
            if (h0 + k * RP + sub < H) {
                char* row = yrow + k * kPassBytes;
                if (mu_one)
                    rotate_store<DT, false>(a, b, cs_cos + slot0, cs_sin + slot0, half >> 1, mu, row, row + half * ES);
                else
                    rotate_store<DT, true>(a, b, cs_cos + slot0, cs_sin + slot0, half >> 1, mu, row, row + half * ES);
            }
        }
    }
}

template <int DT, int LAYOUT, bool VEC, bool CACHE>
__global__ void __launch_bounds__(kWarps * 32)
qk_norm_rope_kernel(QkSide A, QkSide B, int nca, int ncb, float eps, const int32_t* pos, int64_t T, int D, int r,
                    const float* inv_freq, const float2* cache, int64_t cache_len, float mu, int W) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    __shared__ float stage[kWarps][kPasses][kMaxRow];
    pdl_begin();
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // work item of this warp: (token, operand, chunk of R * kPasses heads)
    const int64_t item = (int64_t)blockIdx.x * kWarps + wib;
    const int per_tok = nca + ncb;
    const int64_t t = item / per_tok;
    if (t >= T) return;  // whole warps leave together: no CTA barrier follows
    const int ci = (int)(item - t * per_tok);
    const bool second = ci >= nca;
    const QkSide Q = second ? B : A;
    const int nchunks = (D + V - 1) / V;
    const int R = 32 / W;          // head rows per pass
    const int sub = lane / W;      // row of this lane within a pass
    const int c = lane - sub * W;  // chunk of this lane
    const bool has = c < nchunks;
    const int half = r >> 1;
    const int h0 = (second ? ci - nca : ci) * R * kPasses;

    // loads of every head row of the chunk, before anything else
    const char* xt = Q.x + t * Q.xs * ES;
    char* yt = Q.y + t * Q.ys * ES;
    float f[kPasses][V];
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
        const int h = h0 + k * R + sub;
        if (has && h < Q.H) load_chunk<DT, VEC>(xt + (int64_t)h * D * ES, c, D, f[k]);
    }
    // this lane's gain chunk
    float gv[V];
    if (has) {
        if (VEC)
            S::unpack(ld_reuse(Q.g + (int64_t)c * 16), gv);
        else
#pragma unroll
            for (int e = 0; e < V; ++e) gv[e] = c * V + e < D ? S::load1(Q.g, (int64_t)c * V + e) : 0.0f;
    }
    // the angle of every entry this lane writes (pair of entry j)
    float ca[V], sa[V];
    const int32_t p = pos[t];
#pragma unroll
    for (int e = 0; e < V; ++e) {
        const int j = c * V + e;
        ca[e] = 1.0f;
        sa[e] = 0.0f;
        if (has && j < r) {
            const int i = LAYOUT == 0 ? (j < half ? j : j - half) : (j >> 1);
            if (CACHE && p >= 0 && p < cache_len) {
                const float2 v = __ldg(cache + (int64_t)p * half + i);
                ca[e] = v.x;
                sa[e] = v.y;
            } else {
                rope_sincos(__fmul_rn((float)p, __ldg(inv_freq + i)), &sa[e], &ca[e]);
            }
        }
    }
    // 1) every row's mean of squares: lane sums, then width-W butterflies
    float s[kPasses];
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
        s[k] = 0.0f;
        if (has && h0 + k * R + sub < Q.H) {
#pragma unroll
            for (int e = 0; e < V; ++e) s[k] = __fmaf_rn(f[k][e], f[k][e], s[k]);
        }
    }
    for (int m = W >> 1; m >= 1; m >>= 1) {
#pragma unroll
        for (int k = 0; k < kPasses; ++k) s[k] = __fadd_rn(s[k], __shfl_xor_sync(0xFFFFFFFFu, s[k], m));
    }
    // 2) normalised, stored in the storage type, staged for the partners
    float* rows = &stage[wib][0][sub * (nchunks * V)];
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s[k], (float)D), eps)));
        if (has && h0 + k * R + sub < Q.H) {
#pragma unroll
            for (int e = 0; e < V; ++e) {
                f[k][e] = S::round(__fmul_rn(__fmul_rn(f[k][e], inv), gv[e]));
                if (c * V + e < D) rows[k * kMaxRow + c * V + e] = f[k][e];
            }
        }
    }
    __syncwarp();
    // 3) rotate every entry from itself and its partner, store
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
        const int h = h0 + k * R + sub;
        if (!(has && h < Q.H)) continue;
        const float* row = rows + k * kMaxRow;
        float o[V];
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const int j = c * V + e;
            const float n = f[k][e];
            o[e] = n;
            if (j < r) {
                float a, b;
                bool first;
                if (LAYOUT == 0) {
                    first = j < half;
                    a = first ? n : row[j - half];
                    b = first ? row[j + half] : n;
                } else {
                    first = (j & 1) == 0;
                    a = first ? n : row[j - 1];
                    b = first ? row[j + 1] : n;
                }
                o[e] = first ? __fmul_rn(mu, __fsub_rn(__fmul_rn(a, ca[e]), __fmul_rn(b, sa[e])))
                             : __fmul_rn(mu, __fadd_rn(__fmul_rn(a, sa[e]), __fmul_rn(b, ca[e])));
            }
        }
        char* yr = yt + (int64_t)h * D * ES;
        if (VEC) {
            st_stream(yr + (int64_t)c * 16, S::pack(o));
        } else {
            for (int e = 0; e < V && c * V + e < D; ++e) S::store1(yr, (int64_t)c * V + e, o[e]);
        }
    }
}

// Head rows of 33 to 64 chunks (f32 head_dim up to 256, bf16 up to 512):
// one warp per head row, a lane holding chunks c and c + 32 -- the map and
// the tree gbe_rmsnorm takes for such a row (32 threads, two slots each,
// summed slot by slot in element order, then the warp butterfly), so the
// result equals gbe_rmsnorm then gbe_rope_qk bit for bit as on the other
// paths.  The normalised row is staged in shared memory for the pair
// partners; each entry's angle is formed (or read from the table) by the
// lane that writes it.
constexpr int kWideSlots = 2;
constexpr int kMaxWideRow = 32 * kWideSlots * 8;  // floats: 64 chunks of <= 8 entries

template <int DT, int LAYOUT, bool VEC, bool CACHE>
__global__ void __launch_bounds__(kWarps * 32)
qk_norm_rope_wide(QkSide A, QkSide B, int nha, int nhb, float eps, const int32_t* pos, int64_t T, int D, int r,
                  const float* inv_freq, const float2* cache, int64_t cache_len, float mu) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    __shared__ float stage[kWarps][kMaxWideRow];
    pdl_begin();
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * kWarps + wib;  // (token, head row of q or k)
    const int per_tok = nha + nhb;
    const int64_t t = item / per_tok;
    if (t >= T) return;  // whole warps leave together: no CTA barrier follows
    const int hi = (int)(item - t * per_tok);
    const bool second = hi >= nha;
    const QkSide Q = second ? B : A;
    const int h = second ? hi - nha : hi;
    const int nchunks = (D + V - 1) / V;
    const int half = r >> 1;
    const char* xr = Q.x + (t * Q.xs + (int64_t)h * D) * ES;
    char* yr = Q.y + (t * Q.ys + (int64_t)h * D) * ES;
    float f[kWideSlots][V], gv[kWideSlots][V];
#pragma unroll
    for (int q = 0; q < kWideSlots; ++q) {
        const int c = lane + 32 * q;
#pragma unroll
        for (int e = 0; e < V; ++e) f[q][e] = gv[q][e] = 0.0f;
        if (c < nchunks) {
            load_chunk<DT, VEC>(xr, c, D, f[q]);
            if (VEC)
                S::unpack(ld_reuse(Q.g + (int64_t)c * 16), gv[q]);
            else
#pragma unroll
                for (int e = 0; e < V; ++e) gv[q][e] = c * V + e < D ? S::load1(Q.g, (int64_t)c * V + e) : 0.0f;
        }
    }
    // the row's sum of squares: slot by slot, element order, then the butterfly
    float s = 0.0f;
#pragma unroll
    for (int q = 0; q < kWideSlots; ++q)
        if (lane + 32 * q < nchunks)
#pragma unroll
            for (int e = 0; e < V; ++e) s = __fmaf_rn(f[q][e], f[q][e], s);
    s = warp_sum(s);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)D), eps)));
    // normalised, rounded to the storage type, staged for the partners
    float* row = stage[wib];
#pragma unroll
    for (int q = 0; q < kWideSlots; ++q) {
        const int c = lane + 32 * q;
        if (c < nchunks)
#pragma unroll
            for (int e = 0; e < V; ++e) {
                f[q][e] = S::round(__fmul_rn(__fmul_rn(f[q][e], inv), gv[q][e]));
                if (c * V + e < D) row[c * V + e] = f[q][e];
            }
    }
    __syncwarp();
    const int32_t p = pos[t];
#pragma unroll
    for (int q = 0; q < kWideSlots; ++q) {
        const int c = lane + 32 * q;
        if (c >= nchunks) continue;
        float o[V];
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const int j = c * V + e;
            const float n = f[q][e];
            o[e] = n;
            if (j < r) {
                const int i = LAYOUT == 0 ? (j < half ? j : j - half) : (j >> 1);
                float ca, sa;
                if (CACHE && p >= 0 && p < cache_len) {
                    const float2 v = __ldg(cache + (int64_t)p * half + i);
                    ca = v.x;
                    sa = v.y;
                } else {
                    rope_sincos(__fmul_rn((float)p, __ldg(inv_freq + i)), &sa, &ca);
                }
                float a, b;
                bool first;
                if (LAYOUT == 0) {
                    first = j < half;
                    a = first ? n : row[j - half];
                    b = first ? row[j + half] : n;
                } else {
                    first = (j & 1) == 0;
                    a = first ? n : row[j - 1];
                    b = first ? row[j + 1] : n;
                }
                o[e] = first ? __fmul_rn(mu, __fsub_rn(__fmul_rn(a, ca), __fmul_rn(b, sa)))
                             : __fmul_rn(mu, __fadd_rn(__fmul_rn(a, sa), __fmul_rn(b, ca)));
            }
        }
        if (VEC) {
            st_stream(yr + (int64_t)c * 16, S::pack(o));
        } else {
            for (int e = 0; e < V && c * V + e < D; ++e) S::store1(yr, (int64_t)c * V + e, o[e]);
        }
    }
}

template <int DT>
cudaError_t launch_dt(const QkNormRopeArgs& a, bool vec, cudaStream_t st) {
    constexpr int V = Store<DT>::V;
    const int64_t nchunks = (a.D + V - 1) / V;
    int W = 1;
    while (W < nchunks) W <<= 1;
    vec = vec && a.D % V == 0;
    QkSide sd[2];
    for (int k = 0; k < 2; ++k) {
        sd[k].x = static_cast<const char*>(a.side[k].x);
        sd[k].y = static_cast<char*>(a.side[k].y);
        sd[k].g = static_cast<const char*>(a.side[k].g);
        sd[k].xs = a.side[k].stride;
        sd[k].ys = a.side[k].stride;
        sd[k].H = (int)a.side[k].H;
    }
    if (nchunks > 32) {  // head rows of 33 to 64 chunks: a warp per row, two chunks a lane
        const int64_t rows_all = a.T * (a.side[0].H + a.side[1].H);
        const unsigned grid = (unsigned)((rows_all + kWarps - 1) / kWarps);
        const float2* cache = reinterpret_cast<const float2*>(a.cos_sin);
        const int nha = (int)a.side[0].H, nhb = (int)a.side[1].H, Di = (int)a.D, ri = (int)a.r;
#define GBE_QKW(L, VV, C)                                                                                      \
    return launch(qk_norm_rope_wide<DT, L, VV, C>, dim3(grid), dim3(kWarps * 32), 0, st, sd[0], sd[1], nha, nhb, \
                  a.eps, a.pos, a.T, Di, ri, a.inv_freq, cache, a.cache_len, a.mu)
        if (a.layout == 0) {
            if (vec) { if (cache) GBE_QKW(0, true, true); else GBE_QKW(0, true, false); }
            if (cache) GBE_QKW(0, false, true); else GBE_QKW(0, false, false);
        }
        if (vec) { if (cache) GBE_QKW(1, true, true); else GBE_QKW(1, true, false); }
        if (cache) GBE_QKW(1, false, true); else GBE_QKW(1, false, false);
#undef GBE_QKW
    }
    int lgL = 0;
    while ((2 << lgL) < nchunks) ++lgL;
    const bool pair = vec && a.layout == 0 && a.r == a.D && nchunks >= 2 && (2 << lgL) == nchunks;
    if (pair) {
        const int np = lgL >= 2 && lgL <= 4 ? 4 : 2;  // passes per warp item
        const int rows_item = (32 >> lgL) * np;
        const int pa = (int)((a.side[0].H + rows_item - 1) / rows_item);
        const int pb = (int)((a.side[1].H + rows_item - 1) / rows_item);
        const int warps = (int)std::min<int64_t>(pa + pb, kTokWarps);
        const float2* cs = reinterpret_cast<const float2*>(a.cos_sin);
#define GBE_QKP(C, G, N)                                                                                              \
    return launch(qk_norm_rope_pair<DT, C, G, N>, dim3((unsigned)a.T), dim3(warps * 32), 0, st, sd[0], sd[1], pa, pb, \
                  a.eps, a.pos, lgL, a.inv_freq, cs, a.cache_len, a.mu)
#define GBE_QKP_L(C)                      \
    switch (lgL) {                        \
        case 2: GBE_QKP(C, 2, 4);         \
        case 3: GBE_QKP(C, 3, 4);         \
        case 4: GBE_QKP(C, 4, 4);         \
        default: GBE_QKP(C, -1, 2);       \
    }
        if (cs != nullptr) GBE_QKP_L(true)
        GBE_QKP_L(false)
#undef GBE_QKP_L
#undef GBE_QKP
    }
    const bool shfl = vec && a.r > 0 && (a.layout == 0 ? (a.r / 2) % V == 0 : a.r % V == 0);
    const int rows_per_item = (32 / W) * (shfl ? kPassesShfl : kPasses);  // head rows one warp handles
    const int nca = (int)((a.side[0].H + rows_per_item - 1) / rows_per_item);
    const int ncb = (int)((a.side[1].H + rows_per_item - 1) / rows_per_item);
    const int64_t items = a.T * (nca + ncb);
    const unsigned grid = (unsigned)((items + kWarps - 1) / kWarps);
    const float2* cache = reinterpret_cast<const float2*>(a.cos_sin);
    const bool cached = cache != nullptr;
    const int Di = (int)a.D, ri = (int)a.r;
#define GBE_QKN(L, VV, C)                                                                                 \
    return launch(qk_norm_rope_kernel<DT, L, VV, C>, dim3(grid), dim3(kWarps * 32), 0, st, sd[0], sd[1], nca, ncb, \
                  a.eps, a.pos, a.T, Di, ri, a.inv_freq, cache, a.cache_len, a.mu, W)
    const int tok_warps = (int)std::min<int64_t>(nca + ncb, kTokWarps);
#define GBE_QKN_S(L, C)                                                                                  \
    return launch(qk_norm_rope_tok<DT, L, C>, dim3((unsigned)a.T), dim3(tok_warps * 32), 0, st, sd[0], sd[1], nca, \
                  ncb, a.eps, a.pos, Di, ri, a.inv_freq, cache, a.cache_len, a.mu, W)
    if (shfl) {
        if (a.layout == 0) {
            if (cached) GBE_QKN_S(0, true); else GBE_QKN_S(0, false);
        } else {
            if (cached) GBE_QKN_S(1, true); else GBE_QKN_S(1, false);
        }
    }
#undef GBE_QKN_S
#define GBE_QKN_L(L)                                                  \
    if (vec) {                                                        \
        if (cached) GBE_QKN(L, true, true); else GBE_QKN(L, true, false);   \
    } else {                                                          \
        if (cached) GBE_QKN(L, false, true); else GBE_QKN(L, false, false); \
    }
    if (a.layout == 0) {
        GBE_QKN_L(0)
    } else {
        GBE_QKN_L(1)
    }
#undef GBE_QKN_L
#undef GBE_QKN
}

}  // namespace

cudaError_t launch_qk_norm_rope(const QkNormRopeArgs& a, int dtype, bool vec, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    return dtype == kF32 ? launch_dt<kF32>(a, vec, st) : launch_dt<kBF16>(a, vec, st);
}

}  // namespace gbe
