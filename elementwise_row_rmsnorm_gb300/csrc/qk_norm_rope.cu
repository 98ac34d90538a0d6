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
//  * the angles are float(p) * omega_i and CUDA's sincosf (or the same values
//    from the cos/sin table), as in rope.cu.
//
// Map: a warp owns one chunk of head rows of one token (4 passes of 32 / W
// rows: 8 rows for bf16 head_dim 128), so the heads of a token spread over
// several warps.  It issues the loads of all its rows first, forms its
// lanes' angles while they are in flight, reduces the rows side by side,
// stages the normalised rows in shared memory (so a lane can read the
// partner of each of its entries), rotates and stores them.  Head width is
// limited to 32 chunks (head_dim <= 128 f32 / 256 bf16).
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

// Aligned rows whose pair partners lie a whole number of chunks apart (the
// half layout with r/2 a multiple of the vector, or the interleaved layout
// with r a multiple of it): no shared memory.  A lane's partner chunk is
// fetched from the partner lane with four register shuffles (half layout),
// or sits in the lane's own chunk (interleaved).  Same arithmetic as below.
template <int DT, int LAYOUT, bool CACHE>
__global__ void __launch_bounds__(kWarps * 32)
qk_norm_rope_shfl(QkSide A, QkSide B, int nca, int ncb, float eps, const int32_t* pos, int64_t T, int D, int r,
                  const float* inv_freq, const float2* cache, int64_t cache_len, float mu, int W) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    constexpr int NP = kPassesShfl;
    pdl_begin();
    const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * kWarps + wib;
    const int per_tok = nca + ncb;
    const int64_t t = item / per_tok;
    if (t >= T) return;  // whole warps leave together
    const int ci = (int)(item - t * per_tok);
    const bool second = ci >= nca;
    const QkSide Q = second ? B : A;
    const int nchunks = D / V;
    const int R = 32 / W;
    const int sub = lane / W;
    const int c = lane - sub * W;
    const bool has = c < nchunks;
    const int half = r >> 1;
    const int G = half / V;  // chunks between pair members (half layout)
    const int h0 = (second ? ci - nca : ci) * R * NP;
    const char* xt = Q.x + t * Q.xs * ES;
    char* yt = Q.y + t * Q.ys * ES;

    Vec16 raw[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        const int h = h0 + k * R + sub;
        raw[k] = Vec16{{0u, 0u, 0u, 0u}};
        if (has && h < Q.H) raw[k] = ld_stream(xt + ((int64_t)h * D + (int64_t)c * V) * ES);
    }
    float gv[V];
    if (has) S::unpack(ld_reuse(Q.g + (int64_t)c * 16), gv);
    // The angles of the pairs this lane's entries belong to, each formed once
    // per lane pair, with the same instructions in every lane (no divergent
    // branch): interleaved, the two members of a pair sit in one lane (even
    // entries form the angle, odd ones copy it); half layout, a first-member
    // lane and its partner lane hold the same pairs, so each forms half of
    // them and they swap the other half by shuffle.
    const int src = LAYOUT == 0 ? (c < G ? lane + G : (c < 2 * G ? lane - G : lane)) : lane;
    constexpr int HV = V / 2;
    const int32_t p = pos[t];
    float tc[HV], ts[HV];
    const bool low = LAYOUT == 0 ? c < G : true;
#pragma unroll
    for (int k = 0; k < HV; ++k) {
        const int e = LAYOUT == 0 ? k + (low ? 0 : HV) : 2 * k;  // the entry whose angle this lane forms
        const int j = c * V + e;
        tc[k] = 1.0f;
        ts[k] = 0.0f;
        if (has && j < r) {
            const int i = LAYOUT == 0 ? (j < half ? j : j - half) : (j >> 1);
            if (CACHE && p >= 0 && p < cache_len) {
                const float2 v = __ldg(cache + (int64_t)p * half + i);
                tc[k] = v.x;
                ts[k] = v.y;
            } else {
                sincosf(__fmul_rn((float)p, __ldg(inv_freq + i)), &ts[k], &tc[k]);
            }
        }
    }
    float ca[V], sa[V];
    if (LAYOUT == 1) {
#pragma unroll
        for (int k = 0; k < HV; ++k) {
            ca[2 * k] = ca[2 * k + 1] = tc[k];
            sa[2 * k] = sa[2 * k + 1] = ts[k];
        }
    } else {
#pragma unroll
        for (int k = 0; k < HV; ++k) {
            const float pc = __shfl_sync(0xFFFFFFFFu, tc[k], src);  // the partner's entry k (low) or k + HV
            const float ps = __shfl_sync(0xFFFFFFFFu, ts[k], src);
            ca[k] = low ? tc[k] : pc;
            sa[k] = low ? ts[k] : ps;
            ca[k + HV] = low ? pc : tc[k];
            sa[k + HV] = low ? ps : ts[k];
        }
    }
    float s[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        s[k] = 0.0f;
        if (has && h0 + k * R + sub < Q.H) {
            float f[V];
            S::unpack(raw[k], f);
#pragma unroll
            for (int e = 0; e < V; ++e) s[k] = __fmaf_rn(f[e], f[e], s[k]);
        }
    }
    for (int m = W >> 1; m >= 1; m >>= 1) {
#pragma unroll
        for (int k = 0; k < NP; ++k) s[k] = __fadd_rn(s[k], __shfl_xor_sync(0xFFFFFFFFu, s[k], m));
    }
    const bool rot = has && c * V < r;        // this chunk is rotated
    // Both members of a pair take one formula, out = mu * (own * cos + partner * sg)
    // with sg = -sin for the first member and +sin for the second: IEEE gives
    // a - b == a + (-b) and a + b == b + a exactly, so this is the same
    // arithmetic as mu * (a cos - b sin) and mu * (a sin + b cos).
#pragma unroll
    for (int e = 0; e < V; ++e) {
        const bool first_e = LAYOUT == 0 ? c < G : (e & 1) == 0;
        sa[e] = first_e ? -sa[e] : sa[e];
    }
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        if (h0 + k * R >= Q.H) break;  // uniform across the warp
        const int h = h0 + k * R + sub;
        const bool live = has && h < Q.H;
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s[k], (float)D), eps)));
        float n[V];
        S::unpack(raw[k], n);
#pragma unroll
        for (int e = 0; e < V; ++e) n[e] = __fmul_rn(__fmul_rn(n[e], inv), gv[e]);
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
#pragma unroll
        for (int e = 0; e < V; ++e)
            o[e] = rot ? __fmul_rn(mu, __fadd_rn(__fmul_rn(n[e], ca[e]), __fmul_rn(m2[e], sa[e]))) : n[e];
        if (live) st_stream(yt + ((int64_t)h * D + (int64_t)c * V) * ES, S::pack(o));
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
                sincosf(__fmul_rn((float)p, __ldg(inv_freq + i)), &sa[e], &ca[e]);
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
#define GBE_QKN_S(L, C)                                                                                        \
    return launch(qk_norm_rope_shfl<DT, L, C>, dim3(grid), dim3(kWarps * 32), 0, st, sd[0], sd[1], nca, ncb, a.eps, \
                  a.pos, a.T, Di, ri, a.inv_freq, cache, a.cache_len, a.mu, W)
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
