/*
 * oracle.c -- the plain, slow, single-threaded CPU reference of the
 * elementwise and row-wise transformer ops.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check of the package entry
 * file and the CPU-baseline leg of bench.py may load or run this code.  The
 * product (the CUDA library and its Python binding) never calls it and
 * shares no code with it: nothing here is included by, or includes, the CUDA
 * sources.
 *
 * What it follows.  The two pages define every op in f32:
 *   [Ops]  "Operations" (glia runtime spec): section 1 (Argmax, Add),
 *          section 2 (RmsNorm, LayerNorm), section 3 (Rope, Multi-axis RoPE, Cos/sin cache,
 *          TokenEmbed),
 *          section 4 (Silu), section 5 (QK-norm), section 8 (Sample),
 *          section 10 (FusedSkipNorm).  Its CPU reference computes
 *          everything in f32.
 *   [L9.6] "Elementwise kernels in C: RMSNorm, RoPE, SiLU-mul, embedding,
 *          add, argmax": section 2 (principles and the symbol table),
 *          section 2.1 to 2.4, section 3 (worked examples), section 4 (the
 *          interface), section 5 (pitfalls).
 * Each op is written as those sections define it, one operation at a time in
 * the order they state.  The file is compiled with -ffp-contract=off and
 * without fast-math, so every + - * / rounds on its own in f32, exactly as
 * written.  Where the pages leave a step open the reading taken is named in
 * the function's comment.
 *
 * Planted mistakes.  Building with -DORACLE_MUTANT=k (1..15) swaps in the
 * k-th wrong variant of the pitfalls table of [L9.6] section 5 (s01..s15);
 * k = 16 is the pitfall [Ops] section 5 warns about for QK-norm (the norm
 * taken over num_heads * head_dim instead of per head); k = 17 plants a
 * LayerNorm whose variance is not centred on the mean ([Ops] section 2);
 * k = 18 drops the rule that top-p always keeps its first entry ([Ops]
 * section 8); k = 19 rotates every slice of multi-axis RoPE at the first
 * axis's position ([Ops] section 3); k = 20 cuts min-p at p of the whole
 * mass instead of p times the largest probability, and k = 21 orders equal
 * logits by descending index ([Ops] section 8); k = 22 takes the PCG64
 * output rotation from the wrong bits of the state, k = 23 drops the
 * increment's own term from the squared step of the jump-ahead, and k = 24
 * takes an output before its step instead of after it ([Ops] section 8, the
 * seeded generator).
 * The tests build those variants on the CPU to show that their pins reject
 * each one.  A normal build (ORACLE_MUTANT undefined) contains none of them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUT(k) (ORACLE_MUTANT == (k))

enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_ID = -2, ORC_ERR_EMPTY = -3 };

int orc_mutant(void) { return ORACLE_MUTANT; }

/* ---- bf16 storage ----------------------------------------------------------
 * bf16 is the top half of an f32.  Widening is exact (bits << 16); narrowing
 * rounds to nearest, ties to even, and keeps NaN a (quiet) NaN.            */

void orc_bf16_widen(const uint16_t *in, float *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)in[i] << 16;
        memcpy(&out[i], &u, 4);
    }
}

static uint16_t orc_round_one(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

void orc_bf16_round(const float *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round_one(in[i]);
}

/* ---- RMSNorm ---------------------------------------------------------------
 * [L9.6] 2.1 and [Ops] 2: y_i = x_i / sqrt(mean(x^2) + eps) * w_i over one row,
 * eps inside the root.  Per row: sum the squares in f32 in increasing i, divide
 * by d, add eps, take the root, invert, then write x_i * inv * w_i.
 * Readings: [Ops] writes (x / rms) * g while [L9.6] writes x * inv * w; the
 * latter is taken.  [L9.6] inverts with the course's own Newton rsqrt, which
 * the pages do not specify; here 1 / sqrtf, both correctly rounded.
 * y may be x: a row's sum is complete before its first write.                */
int orc_rmsnorm(const float *x, const float *w, float *y, int64_t rows, int64_t d, float eps) {
    if (rows < 0 || d <= 0) return ORC_ERR_ARG;
#if ORACLE_MUTANT == 15
    float ss = 0.0f; /* s15: one sum for the whole call instead of one per row */
#endif
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * d;
        float *yr = y + r * d;
#if ORACLE_MUTANT != 15
        float ss = 0.0f;
#endif
        for (int64_t i = 0; i < d; ++i) {
            float sq = xr[i] * xr[i];
            ss = ss + sq;
        }
        float ms = MUT(2) ? ss : ss / (float)d;      /* s02: no division by d */
        float inv;
        if (MUT(1))
            inv = 1.0f / (sqrtf(ms) + eps);            /* s01: eps outside the root */
        else
            inv = 1.0f / sqrtf(ms + eps);
        for (int64_t i = 0; i < d; ++i) {
            float t = xr[i] * inv;
            yr[i] = MUT(3) ? t : t * w[i];             /* s03: gain forgotten */
        }
    }
    return ORC_OK;
}

/* ---- LayerNorm ---------------------------------------------------------------
 * [Ops] 2 (LayerNorm): mu = mean(x), var = mean((x - mu)^2) over one row,
 * y = (x - mu) / sqrt(var + eps) * g + b.  Per row: sum x in f32 in
 * increasing i and divide by d; then sum (x_i - mu)^2 the same way and
 * divide by d; then write ((x_i - mu) * inv) * g_i + b_i with
 * inv = 1 / sqrt(var + eps).  b may be NULL (no bias; the ruDNN page makes
 * the bias optional).  Reading: the division by the root is taken as a
 * product with its correctly rounded inverse, as for RMSNorm.  y may be x.  */
int orc_layernorm(const float *x, const float *g, const float *b, float *y, int64_t rows, int64_t d,
                  float eps) {
    if (rows < 0 || d <= 0) return ORC_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * d;
        float *yr = y + r * d;
        float s = 0.0f;
        for (int64_t i = 0; i < d; ++i) s = s + xr[i];
        float mu = s / (float)d;
        float s2 = 0.0f;
        for (int64_t i = 0; i < d; ++i) {
            float c = MUT(17) ? xr[i] : xr[i] - mu; /* s17: variance not centred on the mean */
            float sq = c * c;
            s2 = s2 + sq;
        }
        float var = s2 / (float)d;
        float inv = 1.0f / sqrtf(var + eps);
        for (int64_t i = 0; i < d; ++i) {
            float t = (xr[i] - mu) * inv;
            float u = t * g[i];
            yr[i] = b ? u + b[i] : u;
        }
    }
    return ORC_OK;
}

/* ---- Add -------------------------------------------------------------------
 * [Ops] 1 (Add) and [L9.6] 2.4: y_i = a_i + b_i, usually in place (y == a).   */
int orc_add(const float *a, const float *b, float *y, int64_t n) {
    if (n < 0) return ORC_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) y[i] = a[i] + b[i];
    return ORC_OK;
}

/* ---- Fused residual add + RMSNorm -----------------------------------------
 * [Ops] 10 (FusedSkipNorm): returns RmsNorm(x + skip) and x + skip, and must
 * equal the unfused composition.  Reading: the unfused composition stores the
 * sum in the storage type before the norm reads it, so with h_bf16 != 0 the
 * sum is rounded to bf16 first and the norm runs on the rounded h.  In f32
 * the two readings coincide.  h and y are written as f32 values (the caller
 * rounds them to bf16 storage where that applies).                          */
int orc_add_rmsnorm(const float *x, const float *res, const float *w, float *y, float *h,
                    int64_t rows, int64_t d, float eps, int h_bf16) {
    if (rows < 0 || d <= 0) return ORC_ERR_ARG;
    int st = orc_add(x, res, h, rows * d);
    if (st != ORC_OK) return st;
    if (h_bf16) {
        for (int64_t i = 0; i < rows * d; ++i) {
            uint16_t b = orc_round_one(h[i]);
            orc_bf16_widen(&b, &h[i], 1);
        }
    }
    return orc_rmsnorm(h, w, y, rows, d, eps);
}

/* ---- RoPE --------------------------------------------------------------------
 * [L9.6] 2.2 and 4, [Ops] 3.  x is [T, H, D]; pair i (0 <= i < r/2) of token t
 * turns by theta = p_t * omega_i:  a' = mu (a cos - b sin),
 * b' = mu (a sin + b cos).  Layout 0 ("half") pairs entries (i, i + r/2),
 * layout 1 ("interleaved") pairs (2i, 2i + 1).  Entries r .. D-1 pass through.
 * The angle is the double product rounded to f32 (equal to the f32 product of
 * float(p_t) and omega_i below 2^24).  One angle serves every head.  Both
 * members of a pair are read before either is written, so y may be x.
 * Readings: the pages do not say how cos and sin are evaluated; here they are
 * the double cos / sin of the f32 angle, rounded to f32.  mu multiplies the
 * rotated pair from outside, as the matrix form writes it.                   */
int orc_rope(const float *x, float *y, const int32_t *pos, int64_t T, int64_t H, int64_t D,
             int64_t r, const float *inv_freq, float mu, int layout) {
    if (T < 0 || H < 0 || D <= 0 || r < 0 || r > D || (r & 1) || (layout != 0 && layout != 1))
        return ORC_ERR_ARG;
    const int64_t half = r / 2;
    int64_t npairs = half;
    if (MUT(7)) npairs = D / 2; /* s07: every entry rotates, tail included */
    int lay = layout;
    if (MUT(4)) lay = 1 - layout; /* s04: the two layouts swapped */
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < npairs; ++i) {
            int64_t fi = i < half ? i : half - 1; /* s07 keeps its reads inside inv_freq */
            float theta = (float)((double)pos[t] * (double)inv_freq[fi]);
            if (MUT(5)) theta = -theta; /* s05: turned the other way */
            float c = (float)cos((double)theta);
            float s = (float)sin((double)theta);
            float m = MUT(8) ? 1.0f : mu; /* s08: attention scaling ignored */
            int64_t span = MUT(7) ? D / 2 : half;
            for (int64_t h = 0; h < H; ++h) {
                const float *xv = x + (t * H + h) * D;
                float *yv = y + (t * H + h) * D;
                int64_t ia = lay == 0 ? i : 2 * i;
                int64_t ib = lay == 0 ? i + span : 2 * i + 1;
                float a = xv[ia];
                float b = xv[ib];
                float ac = a * c, bs = b * s;
                float a2 = m * (ac - bs);
                float as, bc;
                if (MUT(6))
                    as = a2 * s; /* s06: b' built from the new a' */
                else
                    as = a * s;
                bc = b * c;
                float b2 = m * (as + bc);
                yv[ia] = a2;
                yv[ib] = b2;
            }
        }
        if (y != x && !MUT(7)) {
            for (int64_t h = 0; h < H; ++h)
                for (int64_t j = r; j < D; ++j) y[(t * H + h) * D + j] = x[(t * H + h) * D + j];
        }
    }
    return ORC_OK;
}

/* ---- Multi-axis RoPE -----------------------------------------------------------
 * [Ops] 3 (Multi-axis RoPE): a token's position is a vector (e.g. [t, h, w]);
 * head_dim is cut into consecutive slices of dims[a] entries, one per axis
 * (each even), and slice a -- entries off_a .. off_a + dims[a] - 1 with off_a
 * the sum of the earlier dims -- gets its own RoPE at position pos[t, a]:
 * pair j < dims[a] / 2 turns by pos[t, a] * omega_a[j].  The frequencies of
 * all axes are concatenated in inv_freq (axis a's start after the earlier
 * axes' dims / 2).  Pairs within a slice follow `layout` as in orc_rope;
 * entries past the last slice pass through.  Each slice is exactly orc_rope
 * applied to that slice alone.                                              */
int orc_rope_multi(const float *x, float *y, const int32_t *pos, int64_t T, int64_t H, int64_t D,
                   int64_t A, const int64_t *dims, const float *inv_freq, float mu, int layout) {
    if (T < 0 || H < 0 || D <= 0 || A < 0 || (layout != 0 && layout != 1)) return ORC_ERR_ARG;
    int64_t total = 0;
    for (int64_t a = 0; a < A; ++a) {
        if (dims[a] < 0 || (dims[a] & 1)) return ORC_ERR_ARG;
        total += dims[a];
    }
    if (total > D) return ORC_ERR_ARG;
    if (y != x)
        for (int64_t i = 0; i < T * H * D; ++i) y[i] = x[i];
    int64_t off = 0, foff = 0;
    for (int64_t a = 0; a < A; ++a) {
        const int64_t half = dims[a] / 2;
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t j = 0; j < half; ++j) {
                /* s19: every slice at the first axis's position */
                float theta = (float)((double)pos[t * A + (MUT(19) ? 0 : a)] * (double)inv_freq[foff + j]);
                float c = (float)cos((double)theta);
                float s = (float)sin((double)theta);
                for (int64_t h = 0; h < H; ++h) {
                    float *v = y + (t * H + h) * D + off;
                    int64_t ia = layout == 0 ? j : 2 * j;
                    int64_t ib = layout == 0 ? j + half : 2 * j + 1;
                    float av = v[ia], bv = v[ib];
                    float a2 = mu * (av * c - bv * s);
                    float b2 = mu * (av * s + bv * c);
                    v[ia] = a2;
                    v[ib] = b2;
                }
            }
        }
        off += dims[a];
        foff += half;
    }
    return ORC_OK;
}

/* ---- Cos/sin table -----------------------------------------------------------
 * [Ops] 3 (Cos/sin cache): cos[pos, i] and sin[pos, i] precomputed for every
 * position below max_seq.  Entry p * (r/2) + i holds (cos, sin) of the same
 * f32 angle orc_rope forms, evaluated the same way, so a table-driven
 * rotation equals the formed one.                                           */
int orc_rope_cos_sin(float *cos_sin, int64_t len, int64_t r, const float *inv_freq) {
    if (len < 0 || r < 0 || (r & 1)) return ORC_ERR_ARG;
    const int64_t half = r / 2;
    for (int64_t p = 0; p < len; ++p)
        for (int64_t i = 0; i < half; ++i) {
            float theta = (float)((double)p * (double)inv_freq[i]);
            cos_sin[2 * (p * half + i)] = (float)cos((double)theta);
            cos_sin[2 * (p * half + i) + 1] = (float)sin((double)theta);
        }
    return ORC_OK;
}

#if ORACLE_MUTANT == 16
/* s16 only: one RMSNorm over all H * D entries of a token, the [D] gain tiled per head. */
static int orc_rmsnorm_gain_tiled(const float *x, const float *g, float *y, int64_t T, int64_t H,
                                  int64_t D, float eps) {
    for (int64_t t = 0; t < T; ++t) {
        const float *xt = x + t * H * D;
        float ss = 0.0f;
        for (int64_t i = 0; i < H * D; ++i) ss = ss + xt[i] * xt[i];
        float inv = 1.0f / sqrtf(ss / (float)(H * D) + eps);
        for (int64_t i = 0; i < H * D; ++i) y[t * H * D + i] = (xt[i] * inv) * g[i % D];
    }
    return ORC_OK;
}
#else
#define orc_rmsnorm_gain_tiled(x, g, y, T, H, D, eps) ORC_ERR_ARG
#endif

/* ---- QK-norm, then RoPE -------------------------------------------------------
 * [Ops] 5 (QK-norm): before RoPE, q and k are RMS-normalised per head -- the
 * mean of squares runs over head_dim only, each head with the gain g[D] --
 * and then rotated by [Ops] 3 / [L9.6] 2.2.  The composition is written out:
 * orc_rmsnorm over the T*H rows of D entries, the result stored in the
 * storage type (rounded to bf16 when n_bf16 != 0, as the unfused composition
 * stores it), then orc_rope on the stored values.  x is [T, H, D]
 * contiguous; y may be x.                                                    */
int orc_qk_norm_rope(const float *x, const float *g, float *y, const int32_t *pos, int64_t T,
                     int64_t H, int64_t D, float eps, int64_t r, const float *inv_freq, float mu,
                     int layout, int n_bf16) {
    if (T < 0 || H < 0 || D <= 0) return ORC_ERR_ARG;
    int st;
    if (MUT(16)) /* s16: the norm taken over the whole token (H * D), not per head */
        st = orc_rmsnorm_gain_tiled(x, g, y, T, H, D, eps);
    else
        st = orc_rmsnorm(x, g, y, T * H, D, eps);
    if (st != ORC_OK) return st;
    if (n_bf16) {
        for (int64_t i = 0; i < T * H * D; ++i) {
            uint16_t b = orc_round_one(y[i]);
            orc_bf16_widen(&b, &y[i], 1);
        }
    }
    return orc_rope(y, y, pos, T, H, D, r, inv_freq, mu, layout);
}

/* ---- SiLU-mul ----------------------------------------------------------------
 * [L9.6] 2.3 and [Ops] 4 (Silu): y = g / (1 + e^-g) * u, silu first, then the
 * product with u.  Written this way it saturates: for g -> -inf, e^-g
 * overflows to +inf and the quotient is -0; for g -> +inf the quotient is g.
 * Reading: libm expf replaces the course's own saturating exp (both overflow
 * to +inf above about 88.7).                                                  */
int orc_silu_mul(const float *g, const float *u, float *y, int64_t n) {
    if (n < 0) return ORC_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        float e, silu;
        if (MUT(10))
            e = expf(g[i]); /* s10: e^g instead of e^-g */
        else
            e = expf(-g[i]);
        float den = 1.0f + e;
        if (MUT(9))
            silu = 1.0f / den; /* s09: the sigmoid alone */
        else
            silu = g[i] / den;
        y[i] = silu * u[i];
    }
    return ORC_OK;
}

/* ---- Embedding ---------------------------------------------------------------
 * [L9.6] 2.4 and [Ops] 3 (TokenEmbed): out row t is row ids[t] of the [V, d]
 * table, which starts at element ids[t] * d.  The pages leave the id check to
 * the caller; the oracle reports an id outside [0, V) as an error.           */
int orc_embedding(const float *table, const int32_t *ids, float *out, int64_t n, int64_t d,
                  int64_t V) {
    if (n < 0 || d <= 0 || V < 0) return ORC_ERR_ARG;
    for (int64_t t = 0; t < n; ++t) {
        int64_t id = ids[t];
        if (id < 0 || id >= V) return ORC_ERR_ID;
        int64_t start = MUT(11) ? id : id * d; /* s11: offset ids[t], not ids[t] * d */
        for (int64_t j = 0; j < d; ++j) out[t * d + j] = table[start + j];
    }
    return ORC_OK;
}

/* ---- Greedy argmax -------------------------------------------------------------
 * [L9.6] 2.4 and 4, [Ops] 1 (Argmax) and 8 (greedy sampling): scan forward,
 * skip NaN, keep an entry only if it is strictly greater than the best so
 * far, so equal values go to the lowest index; -1 when the row holds no
 * number.  -0 and +0 compare equal and so tie.  +inf is a number; a row of
 * -inf gives 0.  n == 0 also gives -1 here; orc_argmax_rows rejects it.      */
int32_t orc_argmax(const float *x, int64_t n) {
    int32_t best = -1;
    float bv = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = x[i];
        if (!MUT(13) && v != v) continue;                 /* s13: no NaN check */
        if (best < 0 || (MUT(12) ? v >= bv : v > bv)) {   /* s12: >= instead of > */
            best = (int32_t)i;
            bv = v;
        }
    }
    if (MUT(14) && best < 0) return 0; /* s14: 0 for an empty or all-NaN row */
    return best;
}

/* ---- Sampling ------------------------------------------------------------------
 * [Ops] 8 (Sample): Greedy is argmax; Temperature(t) draws from
 * softmax(logits / t); TopK(k, t) from the softmax of the k largest logits
 * (in descending order); TopP(p, t) from the sorted softmax cut to the
 * prefix whose running sum stays <= p (the first entry always kept),
 * renormalised; MinP(p, t) from the softmax cut to entries >= p * its
 * maximum, renormalised.  Readings: sample_categorical is the inverse CDF
 * -- with one uniform u in [0, 1) per row, supplied by the caller, the first
 * entry (in the distribution's order) whose running sum exceeds u times the
 * sum of all its entries; if rounding leaves none, the last entry with
 * positive weight.  NaN logits take no part (as in argmax); equal logits sort
 * by ascending index; a row with no number gives -1.  Every step is f32 in
 * the order written: z = x / t, m = max z, e = expf(z - m), sums in the
 * distribution's order, probs = e / sum.                                     */

enum { ORC_GREEDY = 0, ORC_TEMPERATURE = 1, ORC_TOP_K = 2, ORC_TOP_P = 3, ORC_MIN_P = 4 };

/* inverse CDF over q[0 .. L) with uniform u */
static int64_t orc_categorical(const float *q, int64_t L, float u) {
    float c = 0.0f;
    int64_t last = -1;
    for (int64_t j = 0; j < L; ++j) c = c + q[j];
    float target = u * c;
    c = 0.0f;
    for (int64_t j = 0; j < L; ++j) {
        c = c + q[j];
        if (q[j] > 0.0f) {
            last = j;
            if (c > target) return j;
        }
    }
    return last;
}

static const float *orc_sort_base;
static int orc_desc_cmp(const void *pa, const void *pb) {
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    float va = orc_sort_base[a], vb = orc_sort_base[b];
    if (va > vb) return -1;
    if (va < vb) return 1;
    if (MUT(21)) return a > b ? -1 : (a < b ? 1 : 0); /* s21: equal logits by descending index */
    return a < b ? -1 : (a > b ? 1 : 0);
}

/* one row; idx and buf are scratch of n entries each */
static int32_t orc_sample_one(const float *x, int64_t n, int method, float t, int64_t k, float p, float u,
                              int64_t *idx, float *buf) {
    if (method == ORC_GREEDY) return orc_argmax(x, n);
    int64_t nv = 0;
    for (int64_t i = 0; i < n; ++i)
        if (x[i] == x[i]) idx[nv++] = i;
    if (nv == 0) return -1;
    if (method == ORC_TOP_K || method == ORC_TOP_P) {
        orc_sort_base = x;
        qsort(idx, (size_t)nv, sizeof(int64_t), orc_desc_cmp);
    }
    int64_t L = nv;
    if (method == ORC_TOP_K && k < L) L = k;
    /* softmax over the (ordered) candidates */
    float m = -INFINITY;
    for (int64_t j = 0; j < L; ++j) {
        float z = x[idx[j]] / t;
        buf[j] = z;
        if (z > m) m = z;
    }
    float S = 0.0f;
    for (int64_t j = 0; j < L; ++j) {
        buf[j] = expf(buf[j] - m);
        S = S + buf[j];
    }
    for (int64_t j = 0; j < L; ++j) buf[j] = buf[j] / S;
    if (method == ORC_TOP_P) {
        float c = 0.0f;
        int64_t keep = 0;
        for (int64_t j = 0; j < L; ++j) {
            c = c + buf[j];
            if (c <= p) keep = j + 1;
            else break;
        }
        if (keep < 1 && !MUT(18)) keep = 1; /* s18: the first entry not forced into the nucleus */
        for (int64_t j = keep; j < L; ++j) buf[j] = 0.0f;
    } else if (method == ORC_MIN_P) {
        float mx = 0.0f;
        for (int64_t j = 0; j < L; ++j)
            if (buf[j] > mx) mx = buf[j];
        float thr = MUT(20) ? p : p * mx; /* s20: the cut against the whole mass, not the maximum */
        for (int64_t j = 0; j < L; ++j)
            if (!(buf[j] >= thr)) buf[j] = 0.0f;
    }
    if (method == ORC_TOP_P || method == ORC_MIN_P) {
        float S2 = 0.0f;
        for (int64_t j = 0; j < L; ++j) S2 = S2 + buf[j];
        if (S2 > 0.0f)
            for (int64_t j = 0; j < L; ++j) buf[j] = buf[j] / S2;
    }
    int64_t j = orc_categorical(buf, L, u);
    return j < 0 ? -1 : (int32_t)idx[j];
}

int orc_sample_rows(const float *x, int32_t *out, int64_t rows, int64_t n, int method, float t, int64_t k,
                    float p, const float *u, int64_t *idx, float *buf) {
    if (rows < 0 || n <= 0 || method < 0 || method > 4) return ORC_ERR_ARG;
    if (method != ORC_GREEDY && !(t > 0.0f)) return ORC_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r)
        out[r] = orc_sample_one(x + r * n, n, method, t, k, p, u ? u[r] : 0.0f, idx, buf);
    return ORC_OK;
}

/* ---- The seeded uniforms of sample_categorical ----------------------------------
 * [Ops] 8 (Sample): sample_categorical draws "using a seeded RNG (Xorshift or
 * PCG)", and the same seed with the same distribution gives the same draw.
 * Reading: PCG64 -- the 128-bit linear congruential generator
 * state' = state * M + INC (mod 2^128) with the XSL-RR output permutation,
 * as O'Neill defines it ("PCG: A Family of Simple Fast Space-Efficient
 * Statistically Good Algorithms for Random Number Generation", 2014): after
 * each step the output is the xor of the state's two 64-bit halves, rotated
 * right by the state's top 6 bits.  M and INC are that generator's default
 * 128-bit multiplier and increment.  A 64-bit seed s is planted as the PCG
 * reference seeds: state = 0, one step, state += s, one step.  Draw number j
 * (j = 0, 1, ...) of the seeded stream is the output after j + 1 further
 * steps, and its uniform is its top 24 bits times 2^-24 (exact in f32, in
 * [0, 1)).  A batch drawn at stream position `offset` gives row r draw
 * number offset + r.  The stream is entered at draw j without stepping j
 * times by the jump-ahead of an LCG (Brown, "Random Number Generation with
 * Arbitrary Strides", 1994): the affine map s -> M s + INC is composed with
 * itself by repeated squaring, over the bits of the distance.                 */
__extension__ typedef unsigned __int128 orc_u128;

static orc_u128 orc_u128_of(uint64_t hi, uint64_t lo) { return ((orc_u128)hi << 64) | lo; }
static orc_u128 orc_pcg_mult(void) { return orc_u128_of(0x2360ED051FC65DA4ULL, 0x4385DF649FCCF645ULL); }
static orc_u128 orc_pcg_inc(void) { return orc_u128_of(0x5851F42D4C957F2DULL, 0x14057B7EF767814FULL); }

static orc_u128 orc_pcg_step(orc_u128 s, orc_u128 inc) { return s * orc_pcg_mult() + inc; }

static uint64_t orc_pcg_output(orc_u128 s) {
    uint64_t x = (uint64_t)(s >> 64) ^ (uint64_t)s;
    unsigned rot = (unsigned)(s >> 122);
    if (MUT(22)) rot = (unsigned)(s >> 58) & 63u; /* s22: rotation taken from the wrong bits */
    return (x >> rot) | (x << ((64u - rot) & 63u));
}

/* the state `delta` steps after s */
static orc_u128 orc_pcg_advance(orc_u128 s, orc_u128 inc, orc_u128 delta) {
    orc_u128 acc_m = 1, acc_c = 0;   /* the map so far: s -> acc_m s + acc_c */
    orc_u128 m = orc_pcg_mult(), c = inc; /* the step map raised to 2^bit */
    while (delta != 0) {
        if (delta & 1) {
            acc_m = acc_m * m;
            acc_c = acc_c * m + c;
        }
        c = MUT(23) ? m * c : (m + 1) * c; /* s23: the squared map's increment loses its c term */
        m = m * m;
        delta >>= 1;
    }
    return acc_m * s + acc_c;
}

static orc_u128 orc_pcg_seeded(uint64_t seed) {
    orc_u128 s = orc_pcg_step(0, orc_pcg_inc());
    s = s + seed;
    return orc_pcg_step(s, orc_pcg_inc());
}

/* For the pins: the seeded state, as (hi, lo). */
void orc_pcg64_seeded_state(uint64_t seed, uint64_t *hi_lo) {
    orc_u128 s = orc_pcg_seeded(seed);
    hi_lo[0] = (uint64_t)(s >> 64);
    hi_lo[1] = (uint64_t)s;
}

/* For the pins: `count` outputs from an arbitrary (state, inc), stepping
 * first; st[0..1] receives the final state (hi, lo). */
void orc_pcg64_raw(uint64_t s_hi, uint64_t s_lo, uint64_t inc_hi, uint64_t inc_lo, int64_t count, uint64_t *out,
                   uint64_t *st) {
    orc_u128 s = orc_u128_of(s_hi, s_lo), inc = orc_u128_of(inc_hi, inc_lo);
    for (int64_t i = 0; i < count; ++i) {
        s = MUT(24) ? s : orc_pcg_step(s, inc); /* s24: output taken before the step */
        out[i] = orc_pcg_output(s);
        if (MUT(24)) s = orc_pcg_step(s, inc);
    }
    st[0] = (uint64_t)(s >> 64);
    st[1] = (uint64_t)s;
}

/* For the pins: the state delta (= d_hi 2^64 + d_lo) steps after (s, inc). */
void orc_pcg64_advance(uint64_t s_hi, uint64_t s_lo, uint64_t inc_hi, uint64_t inc_lo, uint64_t d_hi,
                       uint64_t d_lo, uint64_t *st) {
    orc_u128 s = orc_pcg_advance(orc_u128_of(s_hi, s_lo), orc_u128_of(inc_hi, inc_lo), orc_u128_of(d_hi, d_lo));
    st[0] = (uint64_t)(s >> 64);
    st[1] = (uint64_t)s;
}

/* u[i] = the uniform of draw offset + i of the stream seeded with `seed`. */
void orc_pcg64_uniforms(uint64_t seed, uint64_t offset, int64_t n, float *u) {
    orc_u128 s = orc_pcg_advance(orc_pcg_seeded(seed), orc_pcg_inc(), offset);
    for (int64_t i = 0; i < n; ++i) {
        s = orc_pcg_step(s, orc_pcg_inc());
        u[i] = (float)(orc_pcg_output(s) >> 40) * 0x1p-24f;
    }
}

/* Sample with the seeded uniforms: row r draws with the uniform of draw
 * offset + r of the stream seeded with `seed`.  u is scratch of `rows`. */
int orc_sample_rows_seeded(const float *x, int32_t *out, int64_t rows, int64_t n, int method, float t, int64_t k,
                           float p, uint64_t seed, uint64_t offset, float *u, int64_t *idx, float *buf) {
    if (rows < 0) return ORC_ERR_ARG;
    orc_pcg64_uniforms(seed, offset, rows, u);
    return orc_sample_rows(x, out, rows, n, method, t, k, p, u, idx, buf);
}

int orc_argmax_rows(const float *x, int32_t *out, int64_t rows, int64_t n) {
    if (rows < 0 || n < 0 || n > INT32_MAX) return ORC_ERR_ARG;
    if (n == 0 && rows > 0) return ORC_ERR_EMPTY;
    for (int64_t r = 0; r < rows; ++r) out[r] = orc_argmax(x + r * n, n);
    return ORC_OK;
}
