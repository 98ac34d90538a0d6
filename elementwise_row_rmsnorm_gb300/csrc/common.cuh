// common.cuh -- device helpers shared by the sm_103a kernels of this library:
// storage traits (f32 and bf16 in 16-byte vectors), cache-hinted vector
// loads and stores, and fixed-order reductions.
//
// Every arithmetic step that decides result bits is written with an explicit
// rounding intrinsic (__fmul_rn, __fadd_rn, __fmaf_rn, __fdiv_rn, __fsqrt_rn)
// so the compiler cannot contract or reorder it differently between code
// paths (vector or scalar, aligned or not): a row's bits depend only on its
// own data and on the shape, never on the batch or on where it sits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace gbe {

constexpr int kF32 = 0;
constexpr int kBF16 = 1;

// ---- 16-byte vectors ---------------------------------------------------------

struct alignas(16) Vec16 {
    uint32_t w[4];
};

// Streamed read: skip L1 (each byte is read once), coherent path so it stays
// correct when the same kernel writes the location afterwards (y == x).
__device__ __forceinline__ Vec16 ld_stream(const void* p) {
    Vec16 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}

// Read-only data reused by many rows (an RMSNorm gain): keep it in L1.
__device__ __forceinline__ Vec16 ld_reuse(const void* p) {
    Vec16 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}

// Read once and written once, with evict-first priority in L2 (.cs): the
// elementwise ops' whole arrays, which nothing in the same launch reads again.
__device__ __forceinline__ Vec16 ld_once(const void* p) {
    Vec16 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}

// A hint: the 128-byte line holding p is fetched into L2 (no register holds
// it, and nothing waits for it).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void st_once(void* p, const Vec16& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]),
                 "r"(v.w[3])
                 : "memory");
}

// Output stores: written once by this launch, evict-first in L2 (.cs), so
// a large output does not push out what the next launch is about to read.
__device__ __forceinline__ void st_stream(void* p, const Vec16& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
                 "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}

// ---- programmatic dependent launch ---------------------------------------------
//
// Every kernel of this library is launched with programmatic stream
// serialization and opens with pdl_begin(): it first lets the next kernel on
// the stream be launched (that kernel's CTAs are placed on the SMs as this
// kernel's last wave drains), then waits in hardware until the kernel before
// it on the stream has completed and its writes are visible.  A chain of
// dependent ops therefore stays correct, and the launch gap between them is
// hidden.  griddepcontrol.wait is a no-op for a kernel launched without the
// attribute, and it is a hardware wait on the previous grid, not a spin loop.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) cudaGetLastError();  // clear it; the caller reports e
    return e;
}

// ---- RoPE angles ------------------------------------------------------------------

// cos and sin of a RoPE angle theta (the f32 product position * frequency).
// sincosf on an argument beyond about 10^5 takes a long exact reduction
// (positions near 2^20 give angles near 10^6 rad), which costs several times
// the rest of a RoPE launch.  So the angle is reduced by quarter turns with
// Cody and Waite's method ("Software Manual for the Elementary Functions",
// 1980): k = rint(theta * 2/pi), and r = theta - k pi/2 with pi/2 split
// into three f32 parts, P1 + P2 + P3, each the f32 nearest to what the
// parts before it leave of pi/2 (the rest, 1.1e-23, is negligible).  For
// |theta| < 2^22 the first step, fma(-k, P1, theta), is exact: theta and
// k * P1 are both multiples of 2^-23 and their difference is below 2 in
// magnitude; the other two steps round once each, so r carries an error of
// about one f32 ulp of r (about 1e-7 rad).  k may be off by one (the f32
// product theta * 2/pi rounds), which leaves |r| below 0.86 rather than
// pi/4.  On that interval sin and cos are their Taylor series to the
// r^13 and r^14 terms (the first terms left out stay below 7e-14 and
// 6e-15), evaluated by Horner's rule in r^2 with coefficients 1/n!
// rounded to f32 -- a few f32 ulps in all.  The quadrant k mod 4 maps
// (cos r, sin r) to (cos theta, sin theta).  Angles of 2^22 and beyond go
// to sincosf whole.  theta = 0 gives exactly (1, 0), so position 0 is the
// identity.  Every RoPE kernel and the cos/sin table use this one
// function, so the table-driven and the formed results agree bit for bit.
__device__ __forceinline__ void rope_sincos(float theta, float* s, float* c) {
    constexpr float kTwoOverPi = 0x1.45f306p-1f;
    constexpr float kP1 = 0x1.921fb6p+0f;
    constexpr float kP2 = -0x1.777a5cp-25f;
    constexpr float kP3 = -0x1.ee59dap-50f;
    if (fabsf(theta) < 4194304.0f) {
        const float k = rintf(__fmul_rn(theta, kTwoOverPi));
        float r = __fmaf_rn(-k, kP1, theta);
        r = __fmaf_rn(-k, kP2, r);
        r = __fmaf_rn(-k, kP3, r);
        const float r2 = __fmul_rn(r, r);
        // sin r = r + r^3 (-1/3! + r^2 (1/5! - ... + r^2 / 13!))
        float ps = 1.0f / 6227020800.0f;
        ps = __fmaf_rn(ps, r2, -1.0f / 39916800.0f);
        ps = __fmaf_rn(ps, r2, 1.0f / 362880.0f);
        ps = __fmaf_rn(ps, r2, -1.0f / 5040.0f);
        ps = __fmaf_rn(ps, r2, 1.0f / 120.0f);
        ps = __fmaf_rn(ps, r2, -1.0f / 6.0f);
        const float sr = __fmaf_rn(__fmul_rn(ps, r2), r, r);
        // cos r = 1 + r^2 (-1/2! + r^2 (1/4! - ... + r^2 / 14!))
        float pc = -1.0f / 87178291200.0f;
        pc = __fmaf_rn(pc, r2, 1.0f / 479001600.0f);
        pc = __fmaf_rn(pc, r2, -1.0f / 3628800.0f);
        pc = __fmaf_rn(pc, r2, 1.0f / 40320.0f);
        pc = __fmaf_rn(pc, r2, -1.0f / 720.0f);
        pc = __fmaf_rn(pc, r2, 1.0f / 24.0f);
        pc = __fmaf_rn(pc, r2, -0.5f);
        const float cr = __fmaf_rn(pc, r2, 1.0f);
        switch ((int)k & 3) {
            case 0: *s = sr; *c = cr; break;
            case 1: *s = cr; *c = -sr; break;
            case 2: *s = -sr; *c = -cr; break;
            default: *s = -cr; *c = sr; break;
        }
    } else {
        sincosf(theta, s, c);
    }
}

// ---- storage traits ------------------------------------------------------------

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two values rounded to bf16 (nearest, ties to even, as f32_to_bf16_bits) in
// one conversion: lo in bits 0..15, hi in bits 16..31.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2_bits(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Two f32 operations in one instruction (sm_100 and later): each lane of
// the pair is the IEEE round-to-nearest result of the scalar operation, so
// results are bit-identical to __fadd_rn / __fsub_rn / __fmul_rn (checked on
// the GPU over normals, signed zeros, subnormals, infinities and NaN).  One
// caution, also measured: a packed product that feeds a packed add or
// subtract may be fused by the assembler into one rounding despite the
// explicit .rn (a quarter of the lanes of a*c - b*s came out 1-2 ulp off),
// so packed multiplies feed only multiplies or scalar sums.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 sub2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

template <int DT>
struct Store;

template <>
struct Store<kF32> {
    using T = float;
    static constexpr int V = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static void unpack(const Vec16& v, float (&f)[V]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] = __uint_as_float(v.w[e]);
    }
    __device__ __forceinline__ static Vec16 pack(const float (&f)[V]) {
        Vec16 v;
#pragma unroll
        for (int e = 0; e < 4; ++e) v.w[e] = __float_as_uint(f[e]);
        return v;
    }
    __device__ __forceinline__ static float load1(const void* base, int64_t i) {
        return static_cast<const float*>(base)[i];
    }
    __device__ __forceinline__ static void store1(void* base, int64_t i, float f) {
        static_cast<float*>(base)[i] = f;
    }
    // storage rounding of an f32 value (identity for f32)
    __device__ __forceinline__ static float round(float f) { return f; }
};

template <>
struct Store<kBF16> {
    using T = __nv_bfloat16;
    static constexpr int V = 8;
    __device__ __forceinline__ static void unpack(const Vec16& v, float (&f)[V]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(v.w[e] << 16);
            f[2 * e + 1] = __uint_as_float(v.w[e] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static Vec16 pack(const float (&f)[V]) {
        Vec16 v;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            v.w[e] = f32x2_to_bf16x2_bits(f[2 * e], f[2 * e + 1]);
        return v;
    }
    __device__ __forceinline__ static float load1(const void* base, int64_t i) {
        return bf16_bits_to_f32(static_cast<const uint16_t*>(base)[i]);
    }
    __device__ __forceinline__ static void store1(void* base, int64_t i, float f) {
        static_cast<uint16_t*>(base)[i] = (uint16_t)f32_to_bf16_bits(f);
    }
    // one conversion: packing f with a zero low half leaves exactly the f32
    // bits of bf16(f) (the same rounding as f32_to_bf16_bits)
    __device__ __forceinline__ static float round(float f) {
        uint32_t d;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(f), "f"(0.0f));
        return __uint_as_float(d);
    }
};

// s + x * x for each of the two bf16 values of a packed word, low half
// first (element order): the mixed-precision fused multiply-add takes the
// bf16 halves as they are (widening is exact, so the result is the single
// rounding __fmaf_rn gives on the widened values -- the same bits, checked
// on the GPU over 2^25 random words and sums), with no unpacking.
__device__ __forceinline__ float bf16x2_sq_acc(uint32_t w, float s) {
    float d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "fma.rn.f32.bf16 %0, lo, lo, %2;\n\tfma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
        : "=f"(d) : "r"(w), "f"(s));
    return d;
}

// The sum of squares of a 16-byte vector's values in element order, added to s.
template <int DT>
__device__ __forceinline__ float vec_sq_acc(const Vec16& v, float s) {
    if (DT == kBF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) s = bf16x2_sq_acc(v.w[i], s);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) s = __fmaf_rn(__uint_as_float(v.w[i]), __uint_as_float(v.w[i]), s);
    }
    return s;
}

// ---- fixed-order reductions ----------------------------------------------------

// Butterfly sum over the 32 lanes.  Every lane ends with the same bits: at
// each step the two partners add the same two operands (addition commutes).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

// Sum over `nwarps` warps of one row, the warp partials added in warp order.
// `red` holds at least nwarps floats of shared memory.  All threads of the
// row's warps must call it; every one returns the same bits.
__device__ __forceinline__ float row_sum(float v, float* red, int warp, int lane, int nwarps) {
    v = warp_sum(v);
    if (nwarps == 1) return v;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = red[0];
    for (int i = 1; i < nwarps; ++i) s = __fadd_rn(s, red[i]);
    return s;
}

inline int ceil_div_i(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// SM count of the current device, cached per device.
int sm_count();

}  // namespace gbe
