/*
 * gbe_elementwise.h -- C ABI of the GB300 (sm_103a) elementwise and
 * row-wise transformer ops: RMSNorm, fused residual add + RMSNorm, RoPE,
 * SiLU-mul, embedding gather, residual add and greedy argmax.
 *
 * Sources of the definitions (cited per entry point below):
 *   "Operations" -- the op math spec of the glia runtime (sections 1 to 10);
 *   "Elementwise kernels in C: RMSNorm, RoPE, SiLU-mul, embedding, add,
 *   argmax" -- course module L9.6 (sections 2 to 5).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every data pointer is a DEVICE pointer (or host memory the
 * device can address, e.g. pinned and mapped) of the CUDA device that is
 * current when the call is made.  The caller allocates and owns every
 * buffer; the library never allocates, frees or synchronises.  Each pointer
 * must be aligned to its element size (4 bytes for f32, int32; 2 for bf16).
 * 16-byte aligned pointers (and row widths that keep rows 16-byte aligned)
 * take the vectorised path; others take a scalar path with the same
 * per-element arithmetic and the same results.
 *
 * Stream.  Work is enqueued on `stream` (NULL = the legacy default stream)
 * and the call returns without waiting.  Results are valid once the stream
 * has reached the call.
 *
 * Storage types.  `dtype` is GBE_F32 or GBE_BF16; all float tensors of one
 * call share it (except RoPE's inv_freq, always f32).  The math is f32 in
 * both cases; bf16 values are widened exactly and each result is rounded to
 * nearest-even once.
 *
 * Aliasing.  Only the exact aliases listed per entry point are allowed (an
 * output equal to a named input, same pointer and same extent).  Any other
 * overlap between an output and any other buffer is GBE_ERR_ALIAS.
 *
 * Errors.  Every argument is checked on the host before anything is
 * launched; a nonzero status means nothing was enqueued, except
 * GBE_ERR_CUDA, which reports a launch error from the CUDA runtime.  Memory
 * checks: a pointer that is not device-addressable memory of the current
 * device, or whose extent runs past the end of its allocation, is
 * GBE_ERR_POINTER (so a wrong shape is refused instead of reading past a
 * buffer).  Empty work (rows, n or T equal to 0) returns GBE_OK without a
 * launch, except argmax over rows of length 0, which is GBE_ERR_EMPTY.
 * Calls are thread-safe; calls that write the same buffer on different
 * streams race, as any two kernels would.
 */
#ifndef GBE_ELEMENTWISE_H
#define GBE_ELEMENTWISE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gbe_dtype { GBE_F32 = 0, GBE_BF16 = 1 } gbe_dtype;

typedef enum gbe_status {
    GBE_OK = 0,
    GBE_ERR_NULL = 1,    /* a pointer is NULL while its extent is not empty */
    GBE_ERR_SHAPE = 2,   /* a size is negative or out of range (d <= 0, D <= 0, counts past int32) */
    GBE_ERR_DTYPE = 3,   /* dtype is not GBE_F32 or GBE_BF16 */
    GBE_ERR_LAYOUT = 4,  /* RoPE layout is not 0 or 1 */
    GBE_ERR_EPS = 5,     /* eps is negative, NaN or infinite */
    GBE_ERR_ROTARY = 6,  /* RoPE width r is odd, negative or larger than D; mu not finite */
    GBE_ERR_EMPTY = 7,   /* argmax over rows of length 0 */
    GBE_ERR_ALIAS = 8,   /* an output overlaps a buffer other than its permitted exact alias */
    GBE_ERR_ALIGN = 9,   /* a pointer is not aligned to its element size */
    GBE_ERR_POINTER = 10, /* not device memory of the current device, or the extent exceeds its allocation */
    GBE_ERR_CUDA = 11,   /* the CUDA runtime reported an error at launch */
    GBE_ERR_SAMPLING = 12 /* a sampling method or parameter is out of range */
} gbe_status;

/* The stream type; the same type as cudaStream_t, so either may be passed. */
typedef struct CUstream_st *gbe_stream;

/* Static description of a status code (never NULL). */
const char *gbe_status_string(int status);

/* Version of this ABI as major * 10000 + minor * 100 + patch. */
int gbe_version(void);

/* The cudaError_t value behind the last GBE_ERR_CUDA returned on the calling
 * thread (0 when there has been none). */
int gbe_last_cuda_error(void);

/*
 * gbe_rmsnorm -- RMSNorm with eps inside the root, over each row.
 *   "Elementwise kernels in C", section 2.1; "Operations", section 2 (RmsNorm).
 *   y[r, i] = x[r, i] * (1 / sqrt(sum_j x[r, j]^2 / d + eps)) * w[i]
 * x, y : [rows, d] row-major, contiguous; w : [d].  dtype for all three.
 * eps  : finite and >= 0 (0 is allowed; a zero row then gives NaN, as the
 *        definition does; with eps > 0 a zero row gives zeros).
 * Alias: y == x allowed (a row's sum is complete before its first write).
 * Each row's output bits depend only on that row, w, d, eps and dtype: the
 * same row gives the same bits in a batch of any size and at any offset.
 */
int gbe_rmsnorm(const void *x, const void *w, void *y, int64_t rows, int64_t d, float eps, int dtype,
                gbe_stream stream);

/*
 * gbe_add_rmsnorm -- fused residual add + RMSNorm, returning both.
 *   "Operations", section 10 (FusedSkipNorm); the add is "Operations",
 *   section 1 and "Elementwise kernels in C", section 2.4.
 *   h = x + residual (rounded to dtype), y = rmsnorm(h, w, eps)
 * The norm reads the stored (rounded) h, so the result equals gbe_add
 * followed by gbe_rmsnorm bit for bit.
 * x, residual, y, h : [rows, d]; w : [d].
 * Alias: h == residual and/or y == x allowed.
 */
int gbe_add_rmsnorm(const void *x, const void *residual, const void *w, void *y, void *h, int64_t rows,
                    int64_t d, float eps, int dtype, gbe_stream stream);

/*
 * gbe_layernorm -- LayerNorm over each row.
 *   "Operations", section 2 (LayerNorm): mu = mean(x), var = mean((x - mu)^2)
 *   over the row, y = (x - mu) / sqrt(var + eps) * g + b, eps inside the root.
 * x, y : [rows, d] row-major, contiguous; g : [d]; b : [d] or NULL (no bias).
 * eps  : finite and >= 0.  Alias: y == x allowed.
 * Like gbe_rmsnorm, a row's output bits depend only on that row, g, b, d,
 * eps and dtype.
 */
int gbe_layernorm(const void *x, const void *g, const void *b, void *y, int64_t rows, int64_t d, float eps,
                  int dtype, gbe_stream stream);

/*
 * gbe_rope -- rotary position embedding.
 *   "Elementwise kernels in C", section 2.2 and 4; "Operations", section 3 (Rope).
 *   For token t and pair i < r/2: theta = float(pos[t]) * inv_freq[i],
 *   a' = mu * (a cos(theta) - b sin(theta)), b' = mu * (a sin(theta) + b cos(theta)),
 *   with (a, b) = (x[t, h, i], x[t, h, i + r/2]) for layout 0 ("half", HF
 *   Llama) or (x[t, h, 2i], x[t, h, 2i + 1]) for layout 1 ("interleaved").
 *   Entries r .. D-1 of each head pass through unchanged.
 * x, y     : [T, H, D] contiguous, dtype.  pos : int32[T], 0 <= pos < 2^24
 *            (not checked: device data).  inv_freq : f32[r/2], device.
 * r        : rotated width, even, 0 <= r <= D.  mu : attention scaling
 *            (1 unless YaRN), finite.  layout : 0 or 1.
 * Alias: y == x allowed (both members of a pair are read before either is
 * written); in place the entries r .. D-1 are not touched.
 */
int gbe_rope(const void *x, void *y, const int32_t *pos, int64_t T, int64_t H, int64_t D, int64_t r,
             const float *inv_freq, float mu, int layout, int dtype, gbe_stream stream);

/*
 * gbe_rope_qk -- RoPE of q and k in one launch, from strided slices, with an
 * optional cos/sin table.
 *   The rotation of gbe_rope ("Elementwise kernels in C", section 2.2;
 *   "Operations", section 3), applied to two operands that share positions
 *   and frequencies (one angle serves every head of q and of k).  The cos /
 *   sin table is the precomputed cos[pos, i] / sin[pos, i] of "Operations",
 *   section 3 (Cos/sin cache), here an accelerator: the results are the same
 *   bits with or without it.
 * q     : [T, Hq, D] with token stride q_stride (elements, >= Hq * D), so q
 *         may be a column slice of a fused QKV buffer; q_out has the same
 *         shape and stride (q_out == q: in place).  Hq = 0: no q.
 * k     : likewise with Hk, k_stride, k_out.
 * pos, inv_freq, r, mu, layout, dtype : as for gbe_rope.
 * cos_sin : NULL (angles are formed), or a device table of cache_len * r/2
 *         (cos, sin) f32 pairs, entry p * (r/2) + i for position p and pair
 *         i, as gbe_rope_cos_sin writes it for the same r and inv_freq; a
 *         position outside [0, cache_len) is formed instead of read.  8-byte
 *         aligned.
 * Alias: q_out == q and k_out == k allowed; q and k may interleave in one
 * buffer (their rows sharing no byte), which the checks resolve row by row.
 */
int gbe_rope_qk(const void *q, void *q_out, int64_t q_stride, int64_t Hq, const void *k, void *k_out,
                int64_t k_stride, int64_t Hk, const int32_t *pos, int64_t T, int64_t D, int64_t r,
                const float *inv_freq, const float *cos_sin, int64_t cache_len, float mu, int layout, int dtype,
                gbe_stream stream);

/* One operand of gbe_rope_pair. */
typedef struct gbe_rope_operand {
    const void *x;          /* [T, H, D], consecutive tokens `stride` elements apart */
    void *y;                /* the same shape and stride; y == x: in place */
    int64_t stride;         /* elements from one token to the next, >= H * D */
    int64_t H;              /* heads; 0: the operand is absent */
    int64_t r;              /* rotated width: even, 0 <= r <= D */
    const float *inv_freq;  /* device f32[r / 2] */
    float mu;               /* scale of the rotated pairs, finite (1 unless YaRN) */
    int layout;             /* 0: half, 1: interleaved */
} gbe_rope_operand;

/*
 * gbe_rope_pair -- RoPE of two operands in one launch, each with its own
 * rotated width, frequencies, scale and layout.
 *   The rotation of gbe_rope ("Elementwise kernels in C", sections 2.2 and
 *   4: partial rotary width r, the attention scale mu, the half and the
 *   interleaved pairing; "Operations", section 3), applied to two operands
 *   that share only the positions, T, head_dim D and dtype -- for instance
 *   a query with interleaved pairs over r = 64 and a key with half pairs
 *   over r = 128 and mu = 1.2.  Each operand's result equals gbe_rope of it
 *   alone, bit for bit; one launch pays the fixed cost of a kernel once.
 * a : HOST pointer to the first operand's description (read during the
 *     call); b : likewise, or NULL for a single operand.
 * pos : device int32[T], 0 <= pos < 2^24.  T, D, dtype, stream : as for
 *     gbe_rope.
 * Alias: an operand's y == x allowed; the operands may interleave in one
 * buffer (rows sharing no byte), as for gbe_rope_qk.
 * Errors: as for gbe_rope_qk, per operand; a == NULL is GBE_ERR_NULL.
 */
int gbe_rope_pair(const gbe_rope_operand *a, const gbe_rope_operand *b, const int32_t *pos, int64_t T, int64_t D,
                  int dtype, gbe_stream stream);

/*
 * gbe_qk_norm_rope -- QK-norm, then RoPE, of q and k in one pass.
 *   "Operations", section 5 (QK-norm): each head of q and of k is
 *   RMS-normalised over head_dim alone (not over heads x head_dim) with the
 *   gain gq[D] (q) or gk[D] (k) and eps inside the root; then both are
 *   rotated as gbe_rope defines.
 * The result equals gbe_rmsnorm over the T*H head rows, stored in dtype,
 * followed by gbe_rope_qk, bit for bit.
 * q, q_out, q_stride, Hq, k, k_out, k_stride, Hk, pos, T, D, r, inv_freq,
 * cos_sin, cache_len, mu, layout, dtype : as for gbe_rope_qk.
 * gq, gk : device gains of D entries in dtype (ignored when Hq / Hk is 0).
 * eps    : finite and >= 0.
 * D      : at most 64 16-byte chunks (256 f32 or 512 bf16), else GBE_ERR_SHAPE.
 * Alias: q_out == q and k_out == k allowed.
 */
int gbe_qk_norm_rope(const void *q, void *q_out, int64_t q_stride, int64_t Hq, const void *gq, const void *k,
                     void *k_out, int64_t k_stride, int64_t Hk, const void *gk, float eps, const int32_t *pos,
                     int64_t T, int64_t D, int64_t r, const float *inv_freq, const float *cos_sin,
                     int64_t cache_len, float mu, int layout, int dtype, gbe_stream stream);

/*
 * gbe_rope_cos_sin -- build the cos/sin table for gbe_rope_qk.
 *   "Operations", section 3 (Cos/sin cache): for every position
 *   0 <= p < cache_len and pair i < r/2, entry p * (r/2) + i is
 *   (cos(theta), sin(theta)) with theta = float(p) * inv_freq[i], formed with
 *   the same arithmetic as the RoPE kernels.
 * cos_sin : device, f32[cache_len * r/2 * 2], 8-byte aligned, written.
 * inv_freq : device f32[r/2].  r even, >= 0.  cache_len in [0, 2^31).
 */
int gbe_rope_cos_sin(float *cos_sin, int64_t cache_len, int64_t r, const float *inv_freq, gbe_stream stream);

/*
 * gbe_rope_multi -- multi-axis RoPE (video / image DiT positions).
 *   "Operations", section 3 (Multi-axis RoPE): a token's position is a
 *   vector of A axis positions; head_dim is cut into consecutive slices of
 *   dims[0], ..., dims[A-1] entries (each even, summing to at most D), and
 *   slice a gets its own RoPE at position pos[t * A + a] with its own
 *   frequencies.  Within a slice the pairing follows `layout` as in
 *   gbe_rope; entries past the last slice pass through.
 * x, y     : [T, H, D] contiguous, dtype.  pos : device int32[T * A].
 * dims     : HOST array of A int64 (read during the call), 0 <= A <= 8.
 * inv_freq : device f32, the axes' frequencies concatenated: axis a's
 *            dims[a] / 2 entries follow those of the earlier axes.
 * mu, layout : as for gbe_rope.  Alias: y == x allowed.
 */
int gbe_rope_multi(const void *x, void *y, const int32_t *pos, int64_t T, int64_t H, int64_t D, int64_t A,
                   const int64_t *dims, const float *inv_freq, float mu, int layout, int dtype, gbe_stream stream);

/*
 * gbe_silu_mul -- the elementwise core of SwiGLU.
 *   "Elementwise kernels in C", section 2.3; "Operations", section 4 (Silu, SwiGlu).
 *   y[i] = gate[i] / (1 + exp(-gate[i])) * up[i]
 * Saturates without NaN: a gate of -1e4 gives -0 (times up), +100 gives gate * up.
 * gate, up, y : n elements, flat.  Alias: y == gate or y == up allowed.
 */
int gbe_silu_mul(const void *gate, const void *up, void *y, int64_t n, int dtype, gbe_stream stream);

/*
 * gbe_add -- residual add.
 *   "Operations", section 1 (Add); "Elementwise kernels in C", section 2.4.
 *   y[i] = a[i] + b[i]
 * a, b, y : n elements, flat.  Alias: y == a or y == b allowed.
 */
int gbe_add(const void *a, const void *b, void *y, int64_t n, int dtype, gbe_stream stream);

/*
 * gbe_embedding -- embedding-row gather.
 *   "Elementwise kernels in C", section 2.4; "Operations", section 3 (TokenEmbed).
 *   out[t, :] = table[ids[t], :], the source row starting at element ids[t] * d.
 * table : [V, d]; ids : int32[n], device; out : [n, d].
 * bad_id_count : NULL, or a device int32 counter.  An id outside [0, V) is
 *   never read: its output row is written as zeros and, when the counter is
 *   given, the counter is incremented once for that row (the caller zeroes
 *   it beforehand and reads it after the stream reaches the call).  The
 *   pages leave the id check to the caller; the guard keeps a bad id from
 *   reading outside the table.
 * Alias: out must not overlap table, ids or the counter.
 */
int gbe_embedding(const void *table, const int32_t *ids, void *out, int64_t n, int64_t d, int64_t V,
                  int32_t *bad_id_count, int dtype, gbe_stream stream);

/*
 * gbe_argmax -- greedy argmax of each row.
 *   "Elementwise kernels in C", section 2.4 and 4; "Operations", section 1
 *   (Argmax) and section 8 (Sample, Greedy).
 *   out[r] = the lowest index of the largest value of row r, NaN entries
 *   skipped; -1 when the row has no number.  -0 equals +0; +inf is a
 *   number; a row of -inf gives 0.
 * x : [rows, n], dtype; out : int32[rows].  n must be >= 1 when rows > 0
 * (rows of length 0 are rejected with GBE_ERR_EMPTY) and n < 2^31.
 */
int gbe_argmax(const void *x, int32_t *out, int64_t rows, int64_t n, int dtype, gbe_stream stream);

/* Sampling methods of gbe_sample. */
typedef enum gbe_sample_method {
    GBE_SAMPLE_GREEDY = 0,
    GBE_SAMPLE_TEMPERATURE = 1,
    GBE_SAMPLE_TOP_K = 2,
    GBE_SAMPLE_TOP_P = 3,
    GBE_SAMPLE_MIN_P = 4
} gbe_sample_method;

/*
 * gbe_sample -- one draw per row of logits.
 *   "Operations", section 8 (Sample: Greedy, Temperature, TopK, TopP, MinP
 *   and the categorical draw behind them).
 *   GREEDY      : gbe_argmax (u, temperature, top_k and p unused).
 *   TEMPERATURE : draw from softmax(x / t).
 *   TOP_K       : draw from the softmax of the top_k largest logits.
 *   TOP_P       : draw from the descending softmax cut to the longest prefix
 *                 whose running sum stays <= p (the first entry always kept).
 *   MIN_P       : draw from the softmax cut to the entries >= p times its
 *                 largest entry.
 *   The draw is the inverse CDF at u[r]: the first entry, in the
 *   distribution's order (index order for TEMPERATURE and MIN_P, descending
 *   logit with equal logits by ascending index for TOP_K and TOP_P), whose
 *   running sum exceeds u[r] times the sum of the kept entries.
 *   Arithmetic: e = exp2f((x - max(x)) * (log2(e) / t)) in f32 (e = 1 at the
 *   maximum), held as the integer rn(e * 2^40) -- per entry for TOP_K and
 *   TOP_P, per f32 sum of 4 (f32) or 8 (bf16) consecutive entries for
 *   TEMPERATURE and MIN_P; sums and cuts are exact integer arithmetic on
 *   those weights, so the result is deterministic and independent of the
 *   batch.  It equals an exact
 *   evaluation of the definition except where u[r] falls within rounding of
 *   a boundary between two entries (or an entry sits within rounding of a
 *   cut), where either neighbour is a valid draw.
 *   NaN logits take no part; a row with no number, or whose largest x / t is
 *   not finite (+inf in the row, or an overflow of x / t), gives -1.
 * x : [rows, n] row-major, dtype; u : f32[rows], uniforms in [0, 1) (values
 * outside are clamped: u <= 0 takes the first kept entry, u >= 1 the last);
 * out : int32[rows], which overlaps nothing else.  n in [1, 2^23]; rows of
 * length 0 are GBE_ERR_EMPTY.  temperature finite and > 0, top_k >= 1
 * (larger than n keeps all), p in [0, 1]; otherwise
 * GBE_ERR_SAMPLING.  u is read only by methods other than GREEDY, and may be
 * NULL for GREEDY.
 */
int gbe_sample(const void *x, const float *u, int32_t *out, int64_t rows, int64_t n, int method,
               float temperature, int64_t top_k, float p, int dtype, gbe_stream stream);

/*
 * gbe_sample_seeded -- gbe_sample with the uniforms drawn from a seeded
 * generator on the device.
 *   "Operations", section 8 (Sample): sample_categorical draws with a seeded
 *   generator (Xorshift or PCG), and the same seed with the same
 *   distribution gives the same draw.  The generator is PCG64 (as
 *   gbe_pcg64_uniforms defines it); row r draws with the uniform of draw
 *   number offset + r of the stream seeded with `seed`, then exactly as
 *   gbe_sample draws at that uniform.  A caller that samples batch after
 *   batch from one stream advances offset by the rows of each call.  The
 *   [sampling] configuration's "seed = 0 means non-deterministic" is the
 *   caller's to honour (by picking a fresh seed); here 0 is a seed like any
 *   other.
 * x, out, rows, n, method, temperature, top_k, p, dtype, stream, and the
 * errors : as for gbe_sample (no u).
 */
int gbe_sample_seeded(const void *x, int32_t *out, int64_t rows, int64_t n, int method, float temperature,
                      int64_t top_k, float p, uint64_t seed, uint64_t offset, int dtype, gbe_stream stream);

/*
 * gbe_pcg64_uniforms -- the uniforms of gbe_sample_seeded, written out.
 *   "Operations", section 8 (Sample, the seeded RNG of sample_categorical):
 *   PCG64 -- the 128-bit linear congruential generator
 *   s' = s * M + INC (mod 2^128), M = 0x2360ED051FC65DA44385DF649FCCF645,
 *   INC = 0x5851F42D4C957F2D14057B7EF767814F, with the XSL-RR output taken
 *   after each step (the xor of the state's 64-bit halves rotated right by
 *   its top six bits; O'Neill 2014).  Seeding: state 0, one step, plus
 *   seed, one step.  Draw j (j = 0, 1, ...) is the output after j + 1
 *   further steps; its uniform is its top 24 bits times 2^-24, in [0, 1).
 * u : device f32[n], written with the uniforms of draws offset .. offset +
 *     n - 1 (the stream continues past 2^64).  n >= 0.
 */
int gbe_pcg64_uniforms(float *u, int64_t n, uint64_t seed, uint64_t offset, gbe_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* GBE_ELEMENTWISE_H */
