// rope.cu -- rotary position embedding on sm_103a.
//
// Definition ("Elementwise kernels in C", section 2.2 and 4; "Operations",
// section 3, Rope): x is [T, H, D]; pair i (0 <= i < r/2) of token t turns
// by theta = p_t * omega_i, and a' = mu (a cos - b sin),
// b' = mu (a sin + b cos).  Layout 0 ("half") pairs (i, i + r/2), layout 1
// ("interleaved") pairs (2i, 2i + 1).  Entries r .. D-1 pass through.
//
// The angle is the f32 product float(p_t) * omega_i (the correctly rounded
// product, equal to the double product rounded to f32 for p_t < 2^24), and
// its cosine and sine come from CUDA's accurate sincosf (never the __sinf
// approximation: at positions near 2^20 the angles reach 10^6 rad).  Each
// CTA owns a tile of tokens: it first forms the angles and their cos/sin for
// every (token, pair) of the tile into shared memory, once, then every head
// of those tokens reuses them -- the loop order the pages give (token, pair,
// head) with the angle hoisted out of the head loop.
//
// Both members of a pair are loaded (all loads of a thread's batch, in fact)
// before either is stored, and no two threads touch the same entry, so the
// call may run in place (y == x).  Out of place, entries r .. D-1 are
// copied; in place they are not touched at all.  The first batch's loads are
// issued before the tile's angles are formed, so the sincos work overlaps the
// memory latency.
//
// The rotation is written with explicit rounding intrinsics, in the order of
// the definition: mu * ((a * c) - (b * s)) and mu * ((a * s) + (b * c)).
#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 4;  // items a thread loads before it stores any

__device__ __forceinline__ void rotate(float a, float b, float2 cs, float mu, float& a2, float& b2) {
    a2 = __fmul_rn(mu, __fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, cs.y)));
    b2 = __fmul_rn(mu, __fadd_rn(__fmul_rn(a, cs.y), __fmul_rn(b, cs.x)));
}

template <int DT, int LAYOUT, bool VEC>
__global__ void __launch_bounds__(kThreads, 4)
rope_tokens(const void* x, void* y, const int32_t* pos, int64_t T, int H, int D, int r, const float* inv_freq,
            float mu, int tt, int copy_tail) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int64_t ES = sizeof(typename S::T);
    extern __shared__ float2 cs[];  // [tt][r/2] of (cos, sin)
    const int half = r >> 1;
    const int64_t t0 = (int64_t)blockIdx.x * tt;
    const int ntok = (int)min((int64_t)tt, T - t0);
    const char* px = static_cast<const char*>(x);
    char* py = static_cast<char*>(y);

    // cos / sin of every (token, pair) of the tile, once
    auto angles = [&]() {
        for (int j = threadIdx.x; j < ntok * half; j += blockDim.x) {
            const int tk = j / half, i = j - tk * half;
            const float th = __fmul_rn((float)pos[t0 + tk], inv_freq[i]);
            float s, c;
            sincosf(th, &s, &c);
            cs[j] = make_float2(c, s);
        }
    };

    if (VEC) {
        // an item is one 16-byte vector (layout 1) or one pair of vectors r/2
        // apart (layout 0) of one head of one token
        const int G = LAYOUT == 0 ? half / V : r / V;
        const int items = ntok * H * G;
        Vec16 va[kBatch], vb[kBatch];
        int64_t off[kBatch];
        int ci[kBatch];
        auto load_batch = [&](int b0) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int it = b0 + u * kThreads;
                if (it < items) {
                    const int g = it % G;
                    const int th_ = it / G;  // token-in-tile * H + head
                    const int tk = th_ / H;
                    off[u] = ((t0 * H + th_) * (int64_t)D + (int64_t)g * V) * ES;
                    ci[u] = tk * half + (LAYOUT == 0 ? g * V : g * (V / 2));
                    va[u] = ld_stream(px + off[u]);
                    if (LAYOUT == 0) vb[u] = ld_stream(px + off[u] + (int64_t)half * ES);
                }
            }
        };
        auto rotate_batch = [&](int b0) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int it = b0 + u * kThreads;
                if (it < items) {
                    float fa[V], fb[V];
                    S::unpack(va[u], fa);
                    if (LAYOUT == 0) {
                        S::unpack(vb[u], fb);
#pragma unroll
                        for (int e = 0; e < V; ++e) {
                            float a2, b2;
                            rotate(fa[e], fb[e], cs[ci[u] + e], mu, a2, b2);
                            fa[e] = a2;
                            fb[e] = b2;
                        }
                        st_stream(py + off[u], S::pack(fa));
                        st_stream(py + off[u] + (int64_t)half * ES, S::pack(fb));
                    } else {
#pragma unroll
                        for (int e = 0; e < V / 2; ++e) {
                            float a2, b2;
                            rotate(fa[2 * e], fa[2 * e + 1], cs[ci[u] + e], mu, a2, b2);
                            fa[2 * e] = a2;
                            fa[2 * e + 1] = b2;
                        }
                        st_stream(py + off[u], S::pack(fa));
                    }
                }
            }
        };
        // the first batch's loads go out before the angles are formed, so
        // the sincos work overlaps the memory latency
        int b0 = threadIdx.x;
        load_batch(b0);
        angles();
        __syncthreads();
        for (;;) {
            rotate_batch(b0);
            b0 += kBatch * kThreads;
            if (b0 - (int)threadIdx.x >= items) break;
            load_batch(b0);
        }
        // pass-through tail, out of place only
        if (copy_tail) {
            const int GT = (D - r) / V;
            const int titems = ntok * H * GT;
            for (int it = threadIdx.x; it < titems; it += kThreads) {
                const int g = it % GT;
                const int th_ = it / GT;
                const int64_t o = ((t0 * H + th_) * (int64_t)D + r + (int64_t)g * V) * ES;
                st_stream(py + o, ld_stream(px + o));
            }
        }
    } else {
        angles();
        __syncthreads();
        const int items = ntok * H * half;
        for (int it = threadIdx.x; it < items; it += kThreads) {
            const int i = it % half;
            const int th_ = it / half;
            const int tk = th_ / H;
            const int64_t row = (t0 * H + th_) * (int64_t)D;
            const int64_t ia = row + (LAYOUT == 0 ? i : 2 * i);
            const int64_t ib = row + (LAYOUT == 0 ? i + half : 2 * i + 1);
            const float a = S::load1(x, ia), b = S::load1(x, ib);
            float a2, b2;
            rotate(a, b, cs[tk * half + i], mu, a2, b2);
            S::store1(y, ia, a2);
            S::store1(y, ib, b2);
        }
        if (copy_tail) {
            const int w = D - r;
            const int titems = ntok * H * w;
            for (int it = threadIdx.x; it < titems; it += kThreads) {
                const int j = it % w;
                const int th_ = it / w;
                const int64_t o = (t0 * H + th_) * (int64_t)D + r + j;
                if (ES == 4)
                    static_cast<uint32_t*>(y)[o] = static_cast<const uint32_t*>(x)[o];
                else
                    static_cast<uint16_t*>(y)[o] = static_cast<const uint16_t*>(x)[o];
            }
        }
    }
}

template <int DT>
cudaError_t launch_dt(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D, int64_t r,
                      const float* inv_freq, float mu, int layout, bool vec, cudaStream_t st) {
    constexpr int V = Store<DT>::V;
    const int64_t half = r / 2;
    const bool copy_tail = x != y && r < D;
    vec = vec && D % V == 0 && (layout == 0 ? half % V == 0 : r % V == 0);
    // items per token: vector items of the rotation (or scalar pairs), plus the tail copy
    int64_t per_tok = vec ? H * (layout == 0 ? half / V : r / V) : H * half;
    if (copy_tail) per_tok += vec ? H * ((D - r) / V) : H * (D - r);
    if (per_tok < 1) per_tok = 1;
    int64_t tt = (kBatch * kThreads) / per_tok;
    if (tt < 1) tt = 1;
    if (tt > 64) tt = 64;
    if (half > 0 && tt > 4096 / half) tt = 4096 / half > 0 ? 4096 / half : 1;  // cos/sin tile <= 32 KB
    const int64_t grid = (T + tt - 1) / tt;
    const size_t smem = (size_t)tt * (size_t)half * sizeof(float2);
    const int Hi = (int)H, Di = (int)D, ri = (int)r, tti = (int)tt, ct = copy_tail ? 1 : 0;
#define GBE_ROPE(L, VV)                                                                                        \
    rope_tokens<DT, L, VV><<<(unsigned)grid, kThreads, smem, st>>>(x, y, pos, T, Hi, Di, ri, inv_freq, mu, tti, ct)
    if (layout == 0) {
        if (vec) GBE_ROPE(0, true); else GBE_ROPE(0, false);
    } else {
        if (vec) GBE_ROPE(1, true); else GBE_ROPE(1, false);
    }
#undef GBE_ROPE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D, int64_t r,
                        const float* inv_freq, float mu, int layout, int dtype, bool vec, cudaStream_t st) {
    if (dtype == kF32) return launch_dt<kF32>(x, y, pos, T, H, D, r, inv_freq, mu, layout, vec, st);
    return launch_dt<kBF16>(x, y, pos, T, H, D, r, inv_freq, mu, layout, vec, st);
}

}  // namespace gbe
