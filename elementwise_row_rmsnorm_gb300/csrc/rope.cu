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
// its cosine and sine come from rope_sincos (common.cuh: a quarter-turn
// reduction and Taylor series; never the __sinf approximation: at positions
// near 2^20 the angles reach 10^6 rad).  The pages' loop order is token,
// pair, head with one angle per (token, pair); here a thread owns a group of
// pairs of one token and has their angles in registers for a chunk of up to
// four heads, with no shared memory and no barrier -- formed by itself, or,
// where K chunks of a token sit in one warp, one K-th of them formed by each
// of K lanes and exchanged by shuffles (an angle formed once per token for
// every 4 K heads).
//
// Both members of a pair are loaded (all loads of a thread, in fact) before
// either is stored, and no two threads touch the same entry, so the call may
// run in place (y == x).  Out of place, entries r .. D-1 are copied; in
// place they are not touched at all.
//
// One launch may serve two operands that share positions and frequencies
// (q and k), each with its own token stride, so q and k can be slices of a
// fused QKV buffer.  Optionally the cos / sin come from a table indexed by
// position ("Operations", section 3, Cos/sin cache; "Elementwise kernels in
// C", Going further), built by rope_cos_sin_table with the very same
// arithmetic, so the cached and the formed results agree bit for bit; a
// position outside the table is formed instead of read.
//
// The rotation is written with explicit rounding intrinsics, in the order of
// the definition: mu * ((a * c) - (b * s)) and mu * ((a * s) + (b * c)).
#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kThreads = 256;
constexpr int kHeadsPerThread = 4;  // heads a thread rotates with one set of angles

// One [T, H, D] operand of a launch: input and output bases, their token
// strides (in elements), its own rotated width, frequencies and scale (the
// layout is a template parameter of the kernel), and the number of threads
// this operand takes.
struct Operand {
    const char* x;
    char* y;
    int64_t xs, ys;
    int H;
    int r;                  // rotated width (even)
    const float* inv_freq;  // f32[r / 2]
    float mu;
    int NC;           // head chunks of kHeadsPerThread (vector path)
    int copy_tail;    // out of place with r < D: entries r .. D-1 are copied
    int64_t threads;  // threads of the launch that serve this operand
};

__device__ __forceinline__ void rotate(float a, float b, float c, float s, float mu, float& a2, float& b2) {
    a2 = __fmul_rn(mu, __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)));
    b2 = __fmul_rn(mu, __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c)));
}

// rotate() for two pairs at once, (a.x, b.x) by (c.x, s.x) and (a.y, b.y)
// by (c.y, s.y): the products and the scale two lanes at a time (packed
// f32x2 multiplies, each lane rounded as the scalar product), the sums
// scalar -- a packed multiply feeding a packed add may be fused into one
// rounding -- so the bits are rotate()'s.
__device__ __forceinline__ void rotate2(float2 a, float2 b, float2 c, float2 s, float mu, float2& a2, float2& b2) {
    const float2 ac = mul2_rn(a, c), bs = mul2_rn(b, s), as = mul2_rn(a, s), bc = mul2_rn(b, c);
    const float2 m = make_float2(mu, mu);
    a2 = mul2_rn(m, make_float2(__fsub_rn(ac.x, bs.x), __fsub_rn(ac.y, bs.y)));
    b2 = mul2_rn(m, make_float2(__fadd_rn(as.x, bc.x), __fadd_rn(as.y, bc.y)));
}

// cos / sin of the angle of pair i at position p: from the table when one is
// given and p lies inside it (it holds exactly these values), else formed.
template <bool CACHE>
__device__ __forceinline__ void angle(int32_t p, int i, const float* inv_freq, const float2* cache,
                                      int64_t cache_len, int half, float& c, float& s) {
    if (CACHE && p >= 0 && p < cache_len) {
        const float2 v = __ldg(cache + (int64_t)p * half + i);
        c = v.x;
        s = v.y;
    } else {
        rope_sincos(__fmul_rn((float)p, __ldg(inv_freq + i)), &s, &c);
    }
}

// Aligned path, one thread's work.  A thread owns one group of P consecutive
// pairs (one 16-byte vector of each pair member) of one token of operand R,
// for a chunk of up to HC heads
// (4, or 1 when the launch would otherwise hold too few threads to fill the
// GPU, as at decode sizes):
// it issues the loads of all its heads first, gets the P angles' cos / sin
// into registers while those loads are in flight, then rotates and stores
// every head.  Threads of one token and head chunk cover consecutive 16-byte
// vectors, so each warp-wide access is contiguous.
//
// K > 1 (angles formed, not read from a table): the launch guarantees that
// the G K consecutive lanes holding items 0..G-1 of K head chunks of one
// token lie in one warp (K divides the operand's chunks, G K divides 32, the
// operand starts on a warp).  Those lanes share the token's angles: lane
// (item g, chunk kq = hc mod K) forms the P / K angles of item g with
// e = kq (mod K), and takes each of its item's P from the lane that formed
// it -- lane g + G (e mod K) of the group, its value e / K -- by register
// shuffles: K times fewer sin/cos evaluations, the same values.
template <int DT, int LAYOUT, bool CACHE, int HC, int K>
__device__ __forceinline__ void rope_vec_item(const Operand& R, int64_t gt, const int32_t* pos, int D,
                                              const float2* cache, int64_t cache_len) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int P = LAYOUT == 0 ? V : V / 2;  // pairs per 16-byte item
    constexpr int64_t ES = sizeof(typename S::T);
    const int r = R.r;
    const float* inv_freq = R.inv_freq;
    const float mu = R.mu;
    const int half = r >> 1;
    const int G = LAYOUT == 0 ? half / V : r / V;  // items per head
    const int g = (int)(gt % G);
    const int64_t rest = gt / G;
    const int hc = (int)(rest % R.NC);
    const int64_t t = rest / R.NC;
    const int h0 = hc * HC;
    const int nh = min(HC, R.H - h0);
    const char* xr = R.x + (t * R.xs + (int64_t)h0 * D) * ES;  // (t, h0, 0)
    char* yr = R.y + (t * R.ys + (int64_t)h0 * D) * ES;
    const int64_t ia = (int64_t)g * V * ES;       // byte offset of the item in a head
    const int64_t hb = (int64_t)half * ES;        // byte distance to the b member (layout 0)
    const int64_t hd = (int64_t)D * ES;           // byte distance between heads

    // the position first: the angles wait for it while the data loads fly
    const int32_t p = pos[t];
    Vec16 va[HC], vb[HC];
#pragma unroll
    for (int j = 0; j < HC; ++j) {
        if (j < nh) {
            va[j] = ld_stream(xr + j * hd + ia);
            if (LAYOUT == 0) vb[j] = ld_stream(xr + j * hd + ia + hb);
        }
    }
    // this thread's pairs, once for all its heads
    float c[P], sn[P];
    const int i0 = g * P;
    if (K > 1) {
        constexpr int PK = P / K > 0 ? P / K : 1;
        const int kq = hc % K;
        float mc[PK], ms[PK];
#pragma unroll
        for (int m = 0; m < PK; ++m) rope_sincos(__fmul_rn((float)p, __ldg(inv_freq + i0 + kq + m * K)), &ms[m], &mc[m]);
        // the lanes of this warp that serve the operand (whole groups)
        const int lane = (int)(gt & 31);
        const int64_t live = R.threads - (gt - lane);
        const unsigned mask = live >= 32 ? 0xFFFFFFFFu : (1u << live) - 1u;
#pragma unroll
        for (int e = 0; e < P; ++e) {
            const int src = g + G * (e % K);
            c[e] = __shfl_sync(mask, mc[e / K], src, G * K);
            sn[e] = __shfl_sync(mask, ms[e / K], src, G * K);
        }
    } else {
#pragma unroll
        for (int e = 0; e < P; ++e) angle<CACHE>(p, i0 + e, inv_freq, cache, cache_len, half, c[e], sn[e]);
    }

#pragma unroll
    for (int j = 0; j < HC; ++j) {
        if (j < nh) {
            char* q = yr + j * hd + ia;
            float fa[V];
            S::unpack(va[j], fa);
            if (LAYOUT == 0) {
                float fb[V];
                S::unpack(vb[j], fb);
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                    float2 a2, b2;
                    rotate2(make_float2(fa[e], fa[e + 1]), make_float2(fb[e], fb[e + 1]),
                            make_float2(c[e], c[e + 1]), make_float2(sn[e], sn[e + 1]), mu, a2, b2);
                    fa[e] = a2.x;
                    fa[e + 1] = a2.y;
                    fb[e] = b2.x;
                    fb[e + 1] = b2.y;
                }
                st_stream(q, S::pack(fa));
                st_stream(q + hb, S::pack(fb));
            } else {
#pragma unroll
                for (int e = 0; e < P; e += 2) {
                    float2 a2, b2;
                    rotate2(make_float2(fa[2 * e], fa[2 * e + 2]), make_float2(fa[2 * e + 1], fa[2 * e + 3]),
                            make_float2(c[e], c[e + 1]), make_float2(sn[e], sn[e + 1]), mu, a2, b2);
                    fa[2 * e] = a2.x;
                    fa[2 * e + 2] = a2.y;
                    fa[2 * e + 1] = b2.x;
                    fa[2 * e + 3] = b2.y;
                }
                st_stream(q, S::pack(fa));
            }
        }
    }
    // pass-through entries, out of place only: the G threads of this token and
    // head chunk share the (D - r) / V tail vectors of each head
    if (R.copy_tail) {
        const int GT = (D - r) / V;
        for (int j = 0; j < nh; ++j)
            for (int k = g; k < GT; k += G) {
                const int64_t o = j * hd + ((int64_t)r + (int64_t)k * V) * ES;
                st_stream(yr + o, ld_stream(xr + o));
            }
    }
}

// The launch's threads serve operand A first, then operand B, each with its
// own layout (LA, LB), width, frequencies and scale.
template <int DT, int LA, int LB, bool CACHE, int HC, int K = 1>
__global__ void __launch_bounds__(kThreads)
rope_vec(Operand A, Operand B, const int32_t* pos, int D, const float2* cache, int64_t cache_len) {
    pdl_begin();
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (gt < A.threads)
        rope_vec_item<DT, LA, CACHE, HC, K>(A, gt, pos, D, cache, cache_len);
    else if (gt - A.threads < B.threads)
        rope_vec_item<DT, LB, CACHE, HC, K>(B, gt - A.threads, pos, D, cache, cache_len);
}

// Unaligned path (or widths that do not split into 16-byte vectors): a
// thread owns one pair of one token, gets its angle once and rotates that
// pair in every head; tail threads copy one entry per head.
template <int DT, int LAYOUT, bool CACHE>
__device__ __forceinline__ void rope_scalar_item(const Operand& R, int64_t gt, const int32_t* pos, int D,
                                                 const float2* cache, int64_t cache_len) {
    using S = Store<DT>;
    constexpr int64_t ES = sizeof(typename S::T);
    const int r = R.r;
    const float* inv_freq = R.inv_freq;
    const float mu = R.mu;
    const int half = r >> 1;
    const int per_tok = half + (R.copy_tail ? D - r : 0);
    const int64_t t = gt / per_tok;
    const int k = (int)(gt - t * per_tok);
    if (k < half) {
        float c, sn;
        angle<CACHE>(pos[t], k, inv_freq, cache, cache_len, half, c, sn);
        const int ia = LAYOUT == 0 ? k : 2 * k;
        const int ib = LAYOUT == 0 ? k + half : 2 * k + 1;
        for (int h = 0; h < R.H; ++h) {
            const int64_t xo = t * R.xs + (int64_t)h * D, yo = t * R.ys + (int64_t)h * D;
            const float a = S::load1(R.x, xo + ia), b = S::load1(R.x, xo + ib);
            float a2, b2;
            rotate(a, b, c, sn, mu, a2, b2);
            S::store1(R.y, yo + ia, a2);
            S::store1(R.y, yo + ib, b2);
        }
    } else {
        const int j = r + (k - half);
        for (int h = 0; h < R.H; ++h) {
            const int64_t xo = t * R.xs + (int64_t)h * D + j, yo = t * R.ys + (int64_t)h * D + j;
            if (ES == 4)
                reinterpret_cast<uint32_t*>(R.y)[yo] = reinterpret_cast<const uint32_t*>(R.x)[xo];
            else
                reinterpret_cast<uint16_t*>(R.y)[yo] = reinterpret_cast<const uint16_t*>(R.x)[xo];
        }
    }
}

template <int DT, int LA, int LB, bool CACHE>
__global__ void __launch_bounds__(kThreads)
rope_scalar(Operand A, Operand B, const int32_t* pos, int D, const float2* cache, int64_t cache_len) {
    pdl_begin();
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (gt < A.threads)
        rope_scalar_item<DT, LA, CACHE>(A, gt, pos, D, cache, cache_len);
    else if (gt - A.threads < B.threads)
        rope_scalar_item<DT, LB, CACHE>(B, gt - A.threads, pos, D, cache, cache_len);
}

// Multi-axis RoPE ("Operations", section 3): head_dim is cut into per-axis
// slices; slice a (entries off[a] .. off[a] + 2 half[a] - 1) turns at the
// token's position for axis a, pos[t * A + a], with its own frequencies
// (inv_freq[poff[a] + j] for its pair j).  A thread owns one pair of one
// token: it forms that pair's angle once and rotates the pair in every head.
// Out of place, tail threads copy the entries past the last slice.
template <int DT, int LAYOUT>
__global__ void __launch_bounds__(kThreads)
rope_multi_kernel(const void* x, void* y, const int32_t* pos, int64_t T, int H, int D,
                  const __grid_constant__ MultiAxis ax,
                  const float* inv_freq, float mu, int copy_tail) {
    using S = Store<DT>;
    constexpr int64_t ES = sizeof(typename S::T);
    pdl_begin();
    const int npairs = ax.poff[ax.A];
    const int rot = 2 * npairs;  // rotated entries, all slices
    const int per_tok = npairs + (copy_tail ? D - rot : 0);
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t t = gt / per_tok;
    if (t >= T) return;
    const int k = (int)(gt - t * per_tok);
    if (k < npairs) {
        int a = 0;
        while (a + 1 < ax.A && k >= ax.poff[a + 1]) ++a;
        const int j = k - ax.poff[a];
        const int half = ax.poff[a + 1] - ax.poff[a];
        float c, sn;
        rope_sincos(__fmul_rn((float)pos[t * ax.A + a], __ldg(inv_freq + k)), &sn, &c);
        const int ia = ax.off[a] + (LAYOUT == 0 ? j : 2 * j);
        const int ib = ax.off[a] + (LAYOUT == 0 ? j + half : 2 * j + 1);
        for (int h = 0; h < H; ++h) {
            const int64_t row = (t * H + h) * (int64_t)D;
            const float av = S::load1(x, row + ia), bv = S::load1(x, row + ib);
            float a2, b2;
            rotate(av, bv, c, sn, mu, a2, b2);
            S::store1(y, row + ia, a2);
            S::store1(y, row + ib, b2);
        }
    } else {
        const int jj = rot + (k - npairs);
        for (int h = 0; h < H; ++h) {
            const int64_t o = (t * H + h) * (int64_t)D + jj;
            if (ES == 4)
                static_cast<uint32_t*>(y)[o] = static_cast<const uint32_t*>(x)[o];
            else
                static_cast<uint16_t*>(y)[o] = static_cast<const uint16_t*>(x)[o];
        }
    }
}

// Multi-axis, aligned path (every slice offset and width, and D, split into
// 16-byte vectors).  rope_vec's map with items drawn from all slices: a
// thread owns one item (P pairs of one slice) of one token for a chunk of up
// to four heads, loads all of them first, forms the P angles from its
// slice's position and frequencies while they are in flight, then rotates
// and stores.  Item g belongs to the slice whose item range holds it.
//
// HC heads a thread; K > 1: the G K lanes of K head chunks of one token (one
// warp: the launch checks that K divides NC and G K divides 32) share the
// angles as in rope_vec_item, lane (g, kq) forming the P / K of item g with
// e = kq (mod K) from its item's slice.
template <int DT, int LAYOUT, int HC, int K>
__global__ void __launch_bounds__(kThreads)
rope_multi_vec(const char* x, char* y, const int32_t* pos, int64_t T, int H, int D,
               const __grid_constant__ MultiAxis ax,
               const float* inv_freq, float mu, int copy_tail, int G, int NC) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int P = LAYOUT == 0 ? V : V / 2;  // pairs per 16-byte item
    constexpr int64_t ES = sizeof(typename S::T);
    pdl_begin();
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int g = (int)(gt % G);
    const int64_t rest = gt / G;
    const int hc = (int)(rest % NC);
    const int64_t t = rest / NC;
    if (t >= T) return;
    // the slice of item g and the item's first pair within it
    int a = 0, first = 0;
    for (;;) {
        const int items = (ax.poff[a + 1] - ax.poff[a]) / P;
        if (g < first + items || a + 1 == ax.A) break;
        first += items;
        ++a;
    }
    const int half = ax.poff[a + 1] - ax.poff[a];
    const int i0 = (g - first) * P;  // first pair of the item within its slice
    const int h0 = hc * HC;
    const int nh = min(HC, H - h0);
    const int64_t hd = (int64_t)D * ES;
    const char* xr = x + (t * H + h0) * hd;
    char* yr = y + (t * H + h0) * hd;
    const int64_t ia = ((int64_t)ax.off[a] + (LAYOUT == 0 ? i0 : 2 * i0)) * ES;
    const int64_t hb = (int64_t)half * ES;

    Vec16 va[HC], vb[HC];
#pragma unroll
    for (int j = 0; j < HC; ++j) {
        if (j < nh) {
            va[j] = ld_stream(xr + j * hd + ia);
            if (LAYOUT == 0) vb[j] = ld_stream(xr + j * hd + ia + hb);
        }
    }
    float c[P], sn[P];
    const float p = (float)pos[t * ax.A + a];
    const int k0 = ax.poff[a] + i0;
    if (K > 1) {
        constexpr int PK = P / K > 0 ? P / K : 1;
        const int kq = hc % K;
        float mc[PK], ms[PK];
#pragma unroll
        for (int m = 0; m < PK; ++m) rope_sincos(__fmul_rn(p, __ldg(inv_freq + k0 + kq + m * K)), &ms[m], &mc[m]);
        const int lane = (int)(gt & 31);
        const int64_t live = T * NC * G - (gt - lane);
        const unsigned mask = live >= 32 ? 0xFFFFFFFFu : (1u << live) - 1u;
#pragma unroll
        for (int e = 0; e < P; ++e) {
            const int src = g + G * (e % K);
            c[e] = __shfl_sync(mask, mc[e / K], src, G * K);
            sn[e] = __shfl_sync(mask, ms[e / K], src, G * K);
        }
    } else {
#pragma unroll
        for (int e = 0; e < P; ++e) rope_sincos(__fmul_rn(p, __ldg(inv_freq + k0 + e)), &sn[e], &c[e]);
    }

#pragma unroll
    for (int j = 0; j < HC; ++j) {
        if (j < nh) {
            char* q = yr + j * hd + ia;
            float fa[V];
            S::unpack(va[j], fa);
            if (LAYOUT == 0) {
                float fb[V];
                S::unpack(vb[j], fb);
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                    float2 a2, b2;
                    rotate2(make_float2(fa[e], fa[e + 1]), make_float2(fb[e], fb[e + 1]),
                            make_float2(c[e], c[e + 1]), make_float2(sn[e], sn[e + 1]), mu, a2, b2);
                    fa[e] = a2.x;
                    fa[e + 1] = a2.y;
                    fb[e] = b2.x;
                    fb[e + 1] = b2.y;
                }
                st_stream(q, S::pack(fa));
                st_stream(q + hb, S::pack(fb));
            } else {
#pragma unroll
                for (int e = 0; e < P; e += 2) {
                    float2 a2, b2;
                    rotate2(make_float2(fa[2 * e], fa[2 * e + 2]), make_float2(fa[2 * e + 1], fa[2 * e + 3]),
                            make_float2(c[e], c[e + 1]), make_float2(sn[e], sn[e + 1]), mu, a2, b2);
                    fa[2 * e] = a2.x;
                    fa[2 * e + 2] = a2.y;
                    fa[2 * e + 1] = b2.x;
                    fa[2 * e + 3] = b2.y;
                }
                st_stream(q, S::pack(fa));
            }
        }
    }
    // entries past the last slice, out of place only: the G threads of this
    // token and head chunk share the tail vectors of each head
    if (copy_tail) {
        const int rot = 2 * ax.poff[ax.A];
        const int GT = (D - rot) / V;
        for (int j = 0; j < nh; ++j)
            for (int k = g; k < GT; k += G) {
                const int64_t o = j * hd + ((int64_t)rot + (int64_t)k * V) * ES;
                st_stream(yr + o, ld_stream(xr + o));
            }
    }
}

// The cos / sin table: entry (p, i) = (cos, sin) of float(p) * omega_i, formed
// exactly as the RoPE kernels form it.
__global__ void __launch_bounds__(kThreads)
rope_cos_sin_table(float2* cache, int64_t len, int half, const float* inv_freq) {
    pdl_begin();
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t p = gt / half;
    if (p >= len) return;
    const int i = (int)(gt - p * half);
    float c, s;
    rope_sincos(__fmul_rn((float)p, __ldg(inv_freq + i)), &s, &c);
    cache[gt] = make_float2(c, s);
}

template <int DT, int LA, int LB, bool CACHE>
cudaError_t launch_shape(bool vec, bool one_head, int K, unsigned grid, const Operand (&op)[2], const RopeArgs& a,
                         const float2* cache, cudaStream_t st) {
    const int Di = (int)a.D;
    if (vec && one_head)
        return launch(rope_vec<DT, LA, LB, CACHE, 1>, dim3(grid), dim3(kThreads), 0, st, op[0], op[1], a.pos, Di,
                      cache, a.cache_len);
    if (vec && !CACHE && K == 4)
        return launch(rope_vec<DT, LA, LB, false, kHeadsPerThread, 4>, dim3(grid), dim3(kThreads), 0, st, op[0],
                      op[1], a.pos, Di, cache, a.cache_len);
    if (vec && !CACHE && K == 2)
        return launch(rope_vec<DT, LA, LB, false, kHeadsPerThread, 2>, dim3(grid), dim3(kThreads), 0, st, op[0],
                      op[1], a.pos, Di, cache, a.cache_len);
    if (vec)
        return launch(rope_vec<DT, LA, LB, CACHE, kHeadsPerThread>, dim3(grid), dim3(kThreads), 0, st, op[0], op[1],
                      a.pos, Di, cache, a.cache_len);
    return launch(rope_scalar<DT, LA, LB, CACHE>, dim3(grid), dim3(kThreads), 0, st, op[0], op[1], a.pos, Di, cache,
                  a.cache_len);
}

template <int DT>
cudaError_t launch_dt(const RopeArgs& a, bool vec, cudaStream_t st) {
    constexpr int V = Store<DT>::V;
    const float2* cache = reinterpret_cast<const float2*>(a.cos_sin);
    bool used[2];
    int64_t G[2];
    vec = vec && a.D % V == 0;
    for (int k = 0; k < 2; ++k) {
        const RopeArgs::Side& sd = a.side[k];
        // in place with nothing to rotate: nothing to do for this operand
        used[k] = sd.H > 0 && a.T > 0 && !(sd.x == sd.y && sd.r == 0);
        G[k] = sd.layout == 0 ? sd.r / 2 / V : sd.r / V;  // 16-byte items per head (vector path)
        if (used[k]) vec = vec && sd.r > 0 && (sd.layout == 0 ? (sd.r / 2) % V == 0 : sd.r % V == 0);
    }
    Operand op[2];
    for (int k = 0; k < 2; ++k) {
        const RopeArgs::Side& sd = a.side[k];
        op[k].x = static_cast<const char*>(sd.x);
        op[k].y = static_cast<char*>(sd.y);
        op[k].xs = sd.stride;
        op[k].ys = sd.stride;
        op[k].H = (int)sd.H;
        op[k].r = (int)sd.r;
        op[k].inv_freq = sd.inv_freq;
        op[k].mu = sd.mu;
        op[k].copy_tail = (sd.x != sd.y && sd.r < a.D) ? 1 : 0;
        op[k].NC = (int)((sd.H + kHeadsPerThread - 1) / kHeadsPerThread);
        if (!used[k])
            op[k].threads = 0;
        else if (vec)
            op[k].threads = a.T * op[k].NC * G[k];
        else
            op[k].threads = a.T * (sd.r / 2 + (op[k].copy_tail ? a.D - sd.r : 0));
    }
    // few threads (decode sizes): one head per thread instead of four
    const bool one_head = vec && op[0].threads + op[1].threads < (int64_t)sm_count() * 256;
    if (one_head)
        for (int k = 0; k < 2; ++k) {
            op[k].NC = op[k].H;
            op[k].threads = op[k].threads ? a.T * op[k].NC * G[k] : 0;
        }
    const int64_t threads = op[0].threads + op[1].threads;
    if (threads == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((threads + kThreads - 1) / kThreads);
    // K chunks of a token share its angles (rope_vec_item) where the lane
    // groups fit whole in warps, for every operand of the launch
    int K = 1;
    if (vec && !one_head && cache == nullptr) {
        for (int kk = 4; kk >= 2 && K == 1; kk >>= 1) {
            bool ok = !(used[0] && used[1]) || op[0].threads % 32 == 0;
            for (int k = 0; k < 2; ++k) {
                if (!used[k]) continue;
                const int P = a.side[k].layout == 0 ? V : V / 2;
                ok = ok && op[k].NC % kk == 0 && P % kk == 0 && 32 % (G[k] * kk) == 0;
            }
            if (ok) K = kk;
        }
    }
    // an operand with no threads takes the other's layout (one kernel fewer)
    const int la = used[0] ? a.side[0].layout : a.side[1].layout;
    const int lb = used[1] ? a.side[1].layout : la;
    if (cache != nullptr) {  // one table: both operands share r, frequencies and layout
        if (la == 0) return launch_shape<DT, 0, 0, true>(vec, one_head, K, grid, op, a, cache, st);
        return launch_shape<DT, 1, 1, true>(vec, one_head, K, grid, op, a, cache, st);
    }
    if (la == 0) {
        if (lb == 0) return launch_shape<DT, 0, 0, false>(vec, one_head, K, grid, op, a, cache, st);
        return launch_shape<DT, 0, 1, false>(vec, one_head, K, grid, op, a, cache, st);
    }
    if (lb == 0) return launch_shape<DT, 1, 0, false>(vec, one_head, K, grid, op, a, cache, st);
    return launch_shape<DT, 1, 1, false>(vec, one_head, K, grid, op, a, cache, st);
}

}  // namespace

cudaError_t launch_rope(const RopeArgs& a, int dtype, bool vec, cudaStream_t st) {
    return dtype == kF32 ? launch_dt<kF32>(a, vec, st) : launch_dt<kBF16>(a, vec, st);
}

cudaError_t launch_rope_multi(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D,
                              const MultiAxis& ax, const float* inv_freq, float mu, int layout, int dtype,
                              cudaStream_t st) {
    const int npairs = ax.poff[ax.A];
    const int copy_tail = (x != y && 2 * npairs < D) ? 1 : 0;
    const int64_t per_tok = npairs + (copy_tail ? D - 2 * npairs : 0);
    if (per_tok == 0 || T == 0 || H == 0) return cudaSuccess;
    const int Hi = (int)H, Di = (int)D;
    // the aligned path: both pointers 16-byte aligned, D and every slice's
    // offset and item width in whole 16-byte vectors
    const int V = dtype == kF32 ? 4 : 8;
    bool vec = npairs > 0 && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0 &&
               D % V == 0;
    int G = 0;
    for (int a = 0; a < ax.A && vec; ++a) {
        const int half = ax.poff[a + 1] - ax.poff[a];
        const int P = layout == 0 ? V : V / 2;
        vec = ax.off[a] % V == 0 && half % P == 0;
        G += half / P;
    }
    if (vec) {
        // heads a thread and the chunks that share a token's angles: three
        // heads and four chunks where the lane groups fit (the angles formed
        // once per token for every 12 heads), else four heads and two, else
        // four heads alone
        const int P = layout == 0 ? V : V / 2;
        auto fits = [&](int hc, int k) {
            const int nc = (Hi + hc - 1) / hc;
            return nc % k == 0 && P % k == 0 && 32 % (G * k) == 0;
        };
        const int hc = fits(3, 4) ? 3 : 4;
        const int K = hc == 3 ? 4 : (fits(4, 2) ? 2 : 1);
        const int NC = (Hi + hc - 1) / hc;
        const dim3 grid((unsigned)((T * NC * G + kThreads - 1) / kThreads));
        const char* xc = static_cast<const char*>(x);
        char* yc = static_cast<char*>(y);
#define GBE_MULTI(D_, L_, H_, K_)                                                                              \
    return launch(rope_multi_vec<D_, L_, H_, K_>, grid, dim3(kThreads), 0, st, xc, yc, pos, T, Hi, Di, ax,     \
                  inv_freq, mu, copy_tail, G, NC)
#define GBE_MULTI_K(D_, L_)                            \
    if (K == 4) GBE_MULTI(D_, L_, 3, 4);               \
    if (K == 2) GBE_MULTI(D_, L_, kHeadsPerThread, 2); \
    GBE_MULTI(D_, L_, kHeadsPerThread, 1)
        if (dtype == kF32) {
            if (layout == 0) { GBE_MULTI_K(kF32, 0); } else { GBE_MULTI_K(kF32, 1); }
        }
        if (layout == 0) { GBE_MULTI_K(kBF16, 0); } else { GBE_MULTI_K(kBF16, 1); }
#undef GBE_MULTI_K
#undef GBE_MULTI
    }
    const dim3 grid((unsigned)((T * per_tok + kThreads - 1) / kThreads));
    if (dtype == kF32) {
        if (layout == 0)
            return launch(rope_multi_kernel<kF32, 0>, grid, dim3(kThreads), 0, st, x, y, pos, T, Hi, Di, ax, inv_freq,
                          mu, copy_tail);
        return launch(rope_multi_kernel<kF32, 1>, grid, dim3(kThreads), 0, st, x, y, pos, T, Hi, Di, ax, inv_freq, mu,
                      copy_tail);
    }
    if (layout == 0)
        return launch(rope_multi_kernel<kBF16, 0>, grid, dim3(kThreads), 0, st, x, y, pos, T, Hi, Di, ax, inv_freq,
                      mu, copy_tail);
    return launch(rope_multi_kernel<kBF16, 1>, grid, dim3(kThreads), 0, st, x, y, pos, T, Hi, Di, ax, inv_freq, mu,
                  copy_tail);
}

cudaError_t launch_rope_cos_sin(float* cos_sin, int64_t len, int64_t r, const float* inv_freq, cudaStream_t st) {
    const int64_t half = r / 2;
    const int64_t n = len * half;
    if (n == 0) return cudaSuccess;
    return launch(rope_cos_sin_table, dim3((unsigned)((n + kThreads - 1) / kThreads)), dim3(kThreads), 0, st,
                  reinterpret_cast<float2*>(cos_sin), len, (int)half, inv_freq);
}

}  // namespace gbe
