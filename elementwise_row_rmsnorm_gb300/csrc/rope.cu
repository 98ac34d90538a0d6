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
// approximation: at positions near 2^20 the angles reach 10^6 rad).  The
// pages' loop order is token, pair, head with one angle per (token, pair);
// here a thread owns a group of pairs of one token and forms their angles
// once, in registers, for a chunk of up to four heads (so an angle is formed
// once per token for every four heads), with no shared memory and no
// barrier.
//
// Both members of a pair are loaded (all loads of a thread, in fact) before
// either is stored, and no two threads touch the same entry, so the call may
// run in place (y == x).  Out of place, entries r .. D-1 are copied; in
// place they are not touched at all.
//
// The rotation is written with explicit rounding intrinsics, in the order of
// the definition: mu * ((a * c) - (b * s)) and mu * ((a * s) + (b * c)).
#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

constexpr int kThreads = 256;
constexpr int kHeadsPerThread = 4;  // heads a thread rotates with one set of angles

__device__ __forceinline__ void rotate(float a, float b, float c, float s, float mu, float& a2, float& b2) {
    a2 = __fmul_rn(mu, __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)));
    b2 = __fmul_rn(mu, __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c)));
}

// Aligned path.  A thread owns one group of P consecutive pairs (one 16-byte
// vector of each pair member) of one token, for a chunk of up to 4 heads:
// it issues the loads of all its heads first, forms the P angles and their
// cos / sin in registers while those loads are in flight, then rotates and
// stores every head.  Threads of one token and head chunk cover consecutive
// 16-byte vectors, so each warp-wide access is contiguous.
template <int DT, int LAYOUT>
__global__ void __launch_bounds__(kThreads)
rope_vec(const void* x, void* y, const int32_t* pos, int64_t T, int H, int D, int r, const float* inv_freq,
         float mu, int copy_tail) {
    using S = Store<DT>;
    constexpr int V = S::V;
    constexpr int P = LAYOUT == 0 ? V : V / 2;  // pairs per 16-byte item
    constexpr int64_t ES = sizeof(typename S::T);
    constexpr int HC = kHeadsPerThread;
    const int half = r >> 1;
    const int G = LAYOUT == 0 ? half / V : r / V;  // items per head
    const int NC = (H + HC - 1) / HC;              // head chunks per token
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int g = (int)(gt % G);
    const int64_t rest = gt / G;
    const int hc = (int)(rest % NC);
    const int64_t t = rest / NC;
    if (t >= T) return;
    const int h0 = hc * HC;
    const int nh = min(HC, H - h0);
    const char* px = static_cast<const char*>(x);
    char* py = static_cast<char*>(y);
    const int64_t row0 = (t * H + h0) * (int64_t)D;  // element offset of (t, h0, 0)
    const int64_t ia = (int64_t)g * V;                // first entry of the item in a head
    const int64_t hb = (int64_t)half * ES;            // byte distance to the b member (layout 0)

    Vec16 va[HC], vb[HC];
#pragma unroll
    for (int j = 0; j < HC; ++j) {
        if (j < nh) {
            const char* p = px + (row0 + (int64_t)j * D + ia) * ES;
            va[j] = ld_stream(p);
            if (LAYOUT == 0) vb[j] = ld_stream(p + hb);
        }
    }
    // the angles of this thread's pairs, once for all its heads
    float c[P], sn[P];
    const float pf = (float)pos[t];
    const int i0 = g * P;
#pragma unroll
    for (int e = 0; e < P; ++e) sincosf(__fmul_rn(pf, __ldg(inv_freq + i0 + e)), &sn[e], &c[e]);

#pragma unroll
    for (int j = 0; j < HC; ++j) {
        if (j < nh) {
            char* q = py + (row0 + (int64_t)j * D + ia) * ES;
            float fa[V];
            S::unpack(va[j], fa);
            if (LAYOUT == 0) {
                float fb[V];
                S::unpack(vb[j], fb);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    float a2, b2;
                    rotate(fa[e], fb[e], c[e], sn[e], mu, a2, b2);
                    fa[e] = a2;
                    fb[e] = b2;
                }
                st_stream(q, S::pack(fa));
                st_stream(q + hb, S::pack(fb));
            } else {
#pragma unroll
                for (int e = 0; e < P; ++e) {
                    float a2, b2;
                    rotate(fa[2 * e], fa[2 * e + 1], c[e], sn[e], mu, a2, b2);
                    fa[2 * e] = a2;
                    fa[2 * e + 1] = b2;
                }
                st_stream(q, S::pack(fa));
            }
        }
    }
    // pass-through entries, out of place only: the G threads of this token and
    // head chunk share the (D - r) / V tail vectors of each head
    if (copy_tail) {
        const int GT = (D - r) / V;
        for (int j = 0; j < nh; ++j)
            for (int k = g; k < GT; k += G) {
                const int64_t o = (row0 + (int64_t)j * D + r + (int64_t)k * V) * ES;
                st_stream(py + o, ld_stream(px + o));
            }
    }
}

// Unaligned path (or widths that do not split into 16-byte vectors): a
// thread owns one pair of one token, forms its angle once and rotates that
// pair in every head; the tail is copied entry by entry.
template <int DT, int LAYOUT>
__global__ void __launch_bounds__(kThreads)
rope_scalar(const void* x, void* y, const int32_t* pos, int64_t T, int H, int D, int r, const float* inv_freq,
            float mu, int copy_tail) {
    using S = Store<DT>;
    const int half = r >> 1;
    const int per_tok = half + (copy_tail ? D - r : 0);
    const int64_t gt = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t t = gt / per_tok;
    const int k = (int)(gt - t * per_tok);
    if (t >= T) return;
    if (k < half) {
        float c, sn;
        sincosf(__fmul_rn((float)pos[t], __ldg(inv_freq + k)), &sn, &c);
        const int ia = LAYOUT == 0 ? k : 2 * k;
        const int ib = LAYOUT == 0 ? k + half : 2 * k + 1;
        for (int h = 0; h < H; ++h) {
            const int64_t row = (t * H + h) * (int64_t)D;
            const float a = S::load1(x, row + ia), b = S::load1(x, row + ib);
            float a2, b2;
            rotate(a, b, c, sn, mu, a2, b2);
            S::store1(y, row + ia, a2);
            S::store1(y, row + ib, b2);
        }
    } else {
        const int j = r + (k - half);
        for (int h = 0; h < H; ++h) {
            const int64_t o = (t * H + h) * (int64_t)D + j;
            if (sizeof(typename S::T) == 4)
                static_cast<uint32_t*>(y)[o] = static_cast<const uint32_t*>(x)[o];
            else
                static_cast<uint16_t*>(y)[o] = static_cast<const uint16_t*>(x)[o];
        }
    }
}

template <int DT>
cudaError_t launch_dt(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D, int64_t r,
                      const float* inv_freq, float mu, int layout, bool vec, cudaStream_t st) {
    constexpr int V = Store<DT>::V;
    const int64_t half = r / 2;
    const bool copy_tail = x != y && r < D;
    vec = vec && r > 0 && D % V == 0 && (layout == 0 ? half % V == 0 : r % V == 0);
    const int Hi = (int)H, Di = (int)D, ri = (int)r, ct = copy_tail ? 1 : 0;
    if (vec) {
        const int64_t G = layout == 0 ? half / V : r / V;
        const int64_t NC = (H + kHeadsPerThread - 1) / kHeadsPerThread;
        const int64_t threads = T * NC * G;
        const int64_t grid = (threads + kThreads - 1) / kThreads;
        if (layout == 0)
            rope_vec<DT, 0><<<(unsigned)grid, kThreads, 0, st>>>(x, y, pos, T, Hi, Di, ri, inv_freq, mu, ct);
        else
            rope_vec<DT, 1><<<(unsigned)grid, kThreads, 0, st>>>(x, y, pos, T, Hi, Di, ri, inv_freq, mu, ct);
    } else {
        const int64_t per_tok = half + (copy_tail ? D - r : 0);
        if (per_tok == 0) return cudaSuccess;
        const int64_t grid = (T * per_tok + kThreads - 1) / kThreads;
        if (layout == 0)
            rope_scalar<DT, 0><<<(unsigned)grid, kThreads, 0, st>>>(x, y, pos, T, Hi, Di, ri, inv_freq, mu, ct);
        else
            rope_scalar<DT, 1><<<(unsigned)grid, kThreads, 0, st>>>(x, y, pos, T, Hi, Di, ri, inv_freq, mu, ct);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D, int64_t r,
                        const float* inv_freq, float mu, int layout, int dtype, bool vec, cudaStream_t st) {
    if (dtype == kF32) return launch_dt<kF32>(x, y, pos, T, H, D, r, inv_freq, mu, layout, vec, st);
    return launch_dt<kBF16>(x, y, pos, T, H, D, r, inv_freq, mu, layout, vec, st);
}

}  // namespace gbe
