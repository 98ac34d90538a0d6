// pcg64.cuh -- the seeded generator behind sample_categorical, on the device.
//
// "Operations", section 8 (Sample): sample_categorical draws "using a seeded
// RNG (Xorshift or PCG)", and the same seed with the same distribution gives
// the same draw.  The generator here is PCG64: the 128-bit linear
// congruential generator s -> M s + INC (mod 2^128) with the XSL-RR output
// (O'Neill, "PCG: A Family of Simple Fast Space-Efficient Statistically Good
// Algorithms for Random Number Generation", 2014) -- after each step, the
// xor of the state's two 64-bit halves rotated right by the state's top six
// bits.  M and INC are the generator's default 128-bit multiplier and
// increment.  A 64-bit seed is planted the way the PCG reference seeds:
// state 0, one step, plus the seed, one step.  Draw number j of the seeded
// stream is the output after j + 1 further steps, and its uniform is the
// output's top 24 bits times 2^-24 (exact in f32, in [0, 1)).
//
// Reaching draw j takes no j steps: one step is the affine map (M, INC),
// and the map of 2^b steps, (M_b, C_b) with M_{b+1} = M_b^2 and
// C_{b+1} = C_b (M_b + 1), is tabulated for every b < 128 at compile time.
// The distance j + 1 then picks one table entry per set bit, and the picked
// maps are composed (they are all powers of one map, so in any order).  A
// warp does this together: lane l takes bits l, l + 32, l + 64 and l + 96,
// and five butterfly steps of warp shuffles compose the 32 lanes' maps.
#pragma once

#include <stdint.h>

namespace gbe {
namespace pcg {

typedef unsigned long long u64;

struct U128 {
    u64 lo, hi;
};

// s -> a s + c (mod 2^128)
struct Affine {
    U128 a, c;
};

// the high 64 bits of a 64 x 64-bit product, from 32-bit pieces (usable in
// constant expressions; the device code uses the hardware instruction)
__host__ __device__ constexpr u64 mulhi_pieces(u64 a, u64 b) {
    const u64 a0 = a & 0xFFFFFFFFull, a1 = a >> 32, b0 = b & 0xFFFFFFFFull, b1 = b >> 32;
    const u64 p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
    const u64 mid = (p00 >> 32) + (p01 & 0xFFFFFFFFull) + (p10 & 0xFFFFFFFFull);
    return p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

__host__ __device__ constexpr U128 mul_const(U128 x, U128 y) {
    return U128{x.lo * y.lo, mulhi_pieces(x.lo, y.lo) + x.lo * y.hi + x.hi * y.lo};
}

__host__ __device__ constexpr U128 add128(U128 x, U128 y) {
    return U128{x.lo + y.lo, x.hi + y.hi + ((x.lo + y.lo) < x.lo ? 1ull : 0ull)};
}

__device__ __forceinline__ U128 mul128(U128 x, U128 y) {
    return U128{x.lo * y.lo, __umul64hi(x.lo, y.lo) + x.lo * y.hi + x.hi * y.lo};
}

constexpr U128 kMult{0x4385DF649FCCF645ull, 0x2360ED051FC65DA4ull};
constexpr U128 kInc{0x14057B7EF767814Full, 0x5851F42D4C957F2Dull};

struct Jumps {
    Affine e[128];
};

constexpr Jumps make_jumps() {
    Jumps t{};
    U128 a = kMult, c = kInc;
    for (int b = 0; b < 128; ++b) {
        t.e[b] = Affine{a, c};
        c = mul_const(c, add128(a, U128{1, 0}));
        a = mul_const(a, a);
    }
    return t;
}

// entry b: the map of 2^b steps
__device__ const Jumps kJumps = make_jumps();

// f then g (the maps commute here, but the composition is written in full)
__device__ __forceinline__ Affine then(const Affine& f, const Affine& g) {
    return Affine{mul128(g.a, f.a), add128(mul128(g.a, f.c), g.c)};
}

__device__ __forceinline__ U128 apply(const Affine& f, U128 s) { return add128(mul128(f.a, s), f.c); }

__device__ __forceinline__ U128 step(U128 s) { return add128(mul128(kMult, s), kInc); }

__device__ __forceinline__ U128 seeded(u64 seed) {
    U128 s = step(U128{0, 0});
    s = add128(s, U128{seed, 0});
    return step(s);
}

// the XSL-RR output of a state
__device__ __forceinline__ u64 output(U128 s) {
    const u64 x = s.hi ^ s.lo;
    const unsigned rot = (unsigned)(s.hi >> 58);
    return (x >> rot) | (x << ((64u - rot) & 63u));
}

__device__ __forceinline__ float uniform_of(u64 out) { return (float)(out >> 40) * 0x1p-24f; }

__device__ __forceinline__ Affine shfl_xor(const Affine& f, int m) {
    return Affine{U128{__shfl_xor_sync(0xFFFFFFFFu, f.a.lo, m), __shfl_xor_sync(0xFFFFFFFFu, f.a.hi, m)},
                  U128{__shfl_xor_sync(0xFFFFFFFFu, f.c.lo, m), __shfl_xor_sync(0xFFFFFFFFu, f.c.hi, m)}};
}

// The map of n steps (n < 2^128), composed by the 32 lanes of a warp; every
// lane of the warp must call it with the same n, and every lane returns it.
__device__ __forceinline__ Affine jump_warp(U128 n) {
    const int lane = threadIdx.x & 31;
    Affine f{U128{1, 0}, U128{0, 0}};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = lane + 32 * q;
        const u64 word = b < 64 ? n.lo : n.hi;
        if ((word >> (b & 63)) & 1ull) f = then(f, kJumps.e[b]);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) f = then(f, shfl_xor(f, m));
    return f;
}

// The map of n steps for n < 2^32, by one thread.
__device__ __forceinline__ Affine jump_small(uint32_t n) {
    Affine f{U128{1, 0}, U128{0, 0}};
    for (int b = 0; n != 0; ++b, n >>= 1)
        if (n & 1u) f = then(f, kJumps.e[b]);
    return f;
}

// The uniform of draw (offset + r) of the stream seeded with `seed`, by a
// whole warp (every lane gets it).
__device__ __forceinline__ float uniform_warp(u64 seed, u64 offset, u64 r) {
    const U128 n = add128(add128(U128{offset, 0}, U128{r, 0}), U128{1, 0});  // draw j is j + 1 steps on
    return uniform_of(output(apply(jump_warp(n), seeded(seed))));
}

}  // namespace pcg
}  // namespace gbe
