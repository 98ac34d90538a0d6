// abi.cu -- the C entry points declared in include/gbe_elementwise.h.
//
// Every argument is validated here, on the host, before anything is
// enqueued, in this order: sizes and scalars; pointer presence and
// alignment; that outputs overlap nothing but their permitted exact aliases
// (address arithmetic alone); that each non-empty buffer is memory the
// current device can address and that its extent stays inside its
// allocation (driver queries, one per distinct allocation of the call).
// Only then is the launcher of the op called.  Nothing here allocates,
// frees or waits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <mutex>

#include "gbe_elementwise.h"
#include "launch.h"

namespace {

constexpr int kVersion = 10100;  // 1.1.0

thread_local int t_last_cuda_error = 0;

int elem_size(int dtype) { return dtype == GBE_F32 ? 4 : dtype == GBE_BF16 ? 2 : 0; }

typedef CUresult (*AddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);
typedef CUresult (*PointerAttributeFn)(void*, CUpointer_attribute, CUdeviceptr);

// A driver entry point, looked up once (the library does not link libcuda).
void* driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return p;
    cudaGetLastError();
    return nullptr;
}

AddressRangeFn address_range_fn() {
    static std::once_flag once;
    static AddressRangeFn fn = nullptr;
    std::call_once(once, [] { fn = reinterpret_cast<AddressRangeFn>(driver_fn("cuMemGetAddressRange")); });
    return fn;
}

PointerAttributeFn pointer_attribute_fn() {
    static std::once_flag once;
    static PointerAttributeFn fn = nullptr;
    std::call_once(once, [] { fn = reinterpret_cast<PointerAttributeFn>(driver_fn("cuPointerGetAttribute")); });
    return fn;
}

// One buffer of a call: where it starts and how many bytes the call touches.
struct Buf {
    const void* p;
    uint64_t bytes;
    uint64_t align;
};

// The checks that need no driver: a non-empty buffer has a pointer, aligned
// to its element size, whose extent does not wrap around the address space.
int check_form(const Buf& b) {
    if (b.bytes == 0) return GBE_OK;
    if (b.p == nullptr) return GBE_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(b.p) % b.align) return GBE_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(b.p) + b.bytes < reinterpret_cast<uintptr_t>(b.p)) return GBE_ERR_POINTER;
    return GBE_OK;
}

// The buffers of one call checked against the driver's record of their
// allocations: each must be memory of the current device (or managed
// memory, or pinned host memory mapped at the same address), and its extent
// must lie inside its allocation.  An allocation, once found, is remembered
// for the rest of the call, so buffers carved from one allocation (q and k
// slices of one QKV buffer, small tensors of one caching-allocator segment)
// take one driver query between them.  Nothing is remembered across calls:
// memory may be freed and reused between them.
class Checker {
  public:
    int begin() {
        if (cudaGetDevice(&dev_) != cudaSuccess) {
            t_last_cuda_error = (int)cudaGetLastError();
            return GBE_ERR_CUDA;
        }
        return GBE_OK;
    }

    int check(const Buf& b) {
        if (b.bytes == 0) return GBE_OK;
        const uintptr_t p = reinterpret_cast<uintptr_t>(b.p);
        for (int i = 0; i < n_; ++i)
            if (p >= seen_[i].lo && p + b.bytes <= seen_[i].hi) return GBE_OK;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, b.p) != cudaSuccess) {
            cudaGetLastError();
            return GBE_ERR_POINTER;
        }
        CUdeviceptr base = 0;
        size_t size = 0;
        bool ranged = false;
        switch (a.type) {
            case cudaMemoryTypeDevice:
                if (a.device != dev_) return GBE_ERR_POINTER;
                [[fallthrough]];
            case cudaMemoryTypeManaged:
                if (AddressRangeFn fn = address_range_fn())
                    ranged = fn(&base, &size, static_cast<CUdeviceptr>(p)) == CUDA_SUCCESS;
                break;
            case cudaMemoryTypeHost:
                // pinned host memory, usable only when mapped at the same
                // address, and only when the driver can say where its
                // allocation ends (else a short buffer could not be told apart)
                if (a.devicePointer != b.p) return GBE_ERR_POINTER;
                if (!host_range(p, &base, &size)) return GBE_ERR_POINTER;
                ranged = true;
                break;
            default:
                return GBE_ERR_POINTER;
        }
        if (ranged) {
            if (p < base || p + b.bytes > base + size) return GBE_ERR_POINTER;
            if (n_ < kSeen) seen_[n_++] = {static_cast<uintptr_t>(base), static_cast<uintptr_t>(base + size)};
        }
        return GBE_OK;
    }

  private:
    static bool host_range(uintptr_t p, CUdeviceptr* base, size_t* size) {
        PointerAttributeFn fn = pointer_attribute_fn();
        if (fn == nullptr) return false;
        CUdeviceptr start = 0;
        size_t len = 0;
        if (fn(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, static_cast<CUdeviceptr>(p)) != CUDA_SUCCESS ||
            fn(&len, CU_POINTER_ATTRIBUTE_RANGE_SIZE, static_cast<CUdeviceptr>(p)) != CUDA_SUCCESS)
            return false;
        *base = start;
        *size = len;
        return len > 0;
    }

    static constexpr int kSeen = 16;
    struct Span {
        uintptr_t lo, hi;
    };
    int dev_ = 0;
    Span seen_[kSeen];
    int n_ = 0;
};

bool overlaps(const Buf& a, const Buf& b) {
    if (a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a.p), y = reinterpret_cast<uintptr_t>(b.p);
    return x < y + b.bytes && y < x + a.bytes;
}

bool same(const Buf& a, const Buf& b) { return a.p == b.p && a.bytes == b.bytes; }

// A strided 2-D region: `rows` rows of `width` bytes, `stride` bytes apart
// (width <= stride).  Used for q and k slices of one fused QKV buffer, whose
// rows interleave without sharing a byte.
struct Rows {
    const void* p;
    int64_t rows, stride, width;
    Buf extent() const {
        return {p, rows > 0 && width > 0 ? (uint64_t)((rows - 1) * stride + width) : 0u, 1};
    }
};

bool rows_overlap(const Rows& a, const Rows& b) {
    if (!overlaps(a.extent(), b.extent())) return false;
    if (a.stride != b.stride || a.stride <= 0) return true;  // cannot tell: treat as overlapping
    const int64_t s = a.stride;
    const int64_t delta = (int64_t)(reinterpret_cast<intptr_t>(b.p) - reinterpret_cast<intptr_t>(a.p));
    // rows t of a and u = t + m of b meet iff -b.width < delta + m * s < a.width
    auto fdiv = [](int64_t n, int64_t d) { return n >= 0 ? n / d : -((-n + d - 1) / d); };
    for (int64_t m = fdiv(-b.width - delta, s); m * s < a.width - delta + s; ++m) {
        const int64_t off = delta + m * s;
        if (!(off > -b.width && off < a.width)) continue;
        if (m > -a.rows && m < b.rows) return true;  // some t in [0, a.rows) has t + m in [0, b.rows)
    }
    return false;
}

bool rows_same(const Rows& a, const Rows& b) {
    return a.p == b.p && a.rows == b.rows && a.stride == b.stride && a.width == b.width;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bytes = count * esize without overflow; false when it would overflow
bool extent(int64_t count, int64_t esize, uint64_t* out) {
    if (count < 0) return false;
    if (count > 0 && esize > INT64_MAX / count) return false;
    *out = (uint64_t)(count * esize);
    return true;
}

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a > 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

int finish(cudaError_t e) {
    if (e != cudaSuccess) {
        t_last_cuda_error = (int)e;
        return GBE_ERR_CUDA;
    }
    return GBE_OK;
}

// Validate the buffers of one call: the form of each (pointer, alignment),
// then every output (the first n_out entries) against every other buffer
// (`alias_ok(o, j)` says whether output o may be exactly buffer j), then each
// buffer against its allocation.
template <int N, typename AliasOk>
int check_all(const Buf (&bufs)[N], int n_out, AliasOk alias_ok) {
    for (int i = 0; i < N; ++i) {
        const int st = check_form(bufs[i]);
        if (st != GBE_OK) return st;
    }
    for (int o = 0; o < n_out; ++o)
        for (int j = 0; j < N; ++j) {
            if (j == o || !overlaps(bufs[o], bufs[j])) continue;
            if (!(alias_ok(o, j) && same(bufs[o], bufs[j]))) return GBE_ERR_ALIAS;
        }
    Checker c;
    int st = c.begin();
    for (int i = 0; i < N && st == GBE_OK; ++i) st = c.check(bufs[i]);
    return st;
}

cudaStream_t as_stream(gbe_stream s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* gbe_status_string(int status) {
    switch (status) {
        case GBE_OK: return "ok";
        case GBE_ERR_NULL: return "a pointer is NULL while its extent is not empty";
        case GBE_ERR_SHAPE: return "a size is negative or out of range";
        case GBE_ERR_DTYPE: return "dtype is not GBE_F32 or GBE_BF16";
        case GBE_ERR_LAYOUT: return "RoPE layout is not 0 (half) or 1 (interleaved)";
        case GBE_ERR_EPS: return "eps is negative, NaN or infinite";
        case GBE_ERR_ROTARY: return "RoPE width r is odd, negative or larger than D, or mu is not finite";
        case GBE_ERR_EMPTY: return "argmax over rows of length 0";
        case GBE_ERR_ALIAS: return "an output overlaps another buffer other than as its permitted exact alias";
        case GBE_ERR_ALIGN: return "a pointer is not aligned to its element size";
        case GBE_ERR_POINTER: return "a pointer is not memory of the current device, or its extent exceeds its allocation";
        case GBE_ERR_CUDA: return "the CUDA runtime reported an error at launch";
        case GBE_ERR_SAMPLING: return "a sampling method or parameter is out of range";
        default: return "unknown status";
    }
}

int gbe_version(void) { return kVersion; }

int gbe_last_cuda_error(void) { return t_last_cuda_error; }

int gbe_rmsnorm(const void* x, const void* w, void* y, int64_t rows, int64_t d, float eps, int dtype,
                gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (rows < 0 || d <= 0 || d > INT32_MAX || rows > INT32_MAX) return GBE_ERR_SHAPE;
    if (!std::isfinite(eps) || eps < 0.0f) return GBE_ERR_EPS;
    int64_t n;
    uint64_t bx, bw;
    if (!mul_ok(rows, d, &n) || !extent(n, es, &bx) || !extent(d, es, &bw)) return GBE_ERR_SHAPE;
    if (rows == 0) return GBE_OK;
    const Buf bufs[3] = {{y, bx, (uint64_t)es}, {x, bx, (uint64_t)es}, {w, bw, (uint64_t)es}};
    const int st = check_all(bufs, 1, [](int o, int j) { return o == 0 && j == 1; });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(x) && aligned16(y) && aligned16(w) && (d * es) % 16 == 0;
    return finish(gbe::launch_rmsnorm(x, nullptr, w, y, nullptr, rows, d, eps, dtype, vec, as_stream(stream)));
}

int gbe_layernorm(const void* x, const void* g, const void* b, void* y, int64_t rows, int64_t d, float eps,
                  int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (rows < 0 || d <= 0 || d > INT32_MAX || rows > INT32_MAX) return GBE_ERR_SHAPE;
    if (!std::isfinite(eps) || eps < 0.0f) return GBE_ERR_EPS;
    int64_t n;
    uint64_t bx, bw;
    if (!mul_ok(rows, d, &n) || !extent(n, es, &bx) || !extent(d, es, &bw)) return GBE_ERR_SHAPE;
    if (rows == 0) return GBE_OK;
    const Buf bufs[4] = {{y, bx, (uint64_t)es}, {x, bx, (uint64_t)es}, {g, bw, (uint64_t)es},
                         {b, b ? bw : 0u, (uint64_t)es}};
    const int st = check_all(bufs, 1, [](int o, int j) { return o == 0 && j == 1; });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(x) && aligned16(y) && aligned16(g) && aligned16(b) && (d * es) % 16 == 0;
    return finish(gbe::launch_layernorm(x, g, b, y, rows, d, eps, dtype, vec, as_stream(stream)));
}

int gbe_add_rmsnorm(const void* x, const void* residual, const void* w, void* y, void* h, int64_t rows,
                    int64_t d, float eps, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (rows < 0 || d <= 0 || d > INT32_MAX || rows > INT32_MAX) return GBE_ERR_SHAPE;
    if (!std::isfinite(eps) || eps < 0.0f) return GBE_ERR_EPS;
    int64_t n;
    uint64_t bx, bw;
    if (!mul_ok(rows, d, &n) || !extent(n, es, &bx) || !extent(d, es, &bw)) return GBE_ERR_SHAPE;
    if (rows == 0) return GBE_OK;
    // outputs first: 0 = y, 1 = h; then 2 = x, 3 = residual, 4 = w
    const Buf bufs[5] = {{y, bx, (uint64_t)es},
                         {h, bx, (uint64_t)es},
                         {x, bx, (uint64_t)es},
                         {residual, bx, (uint64_t)es},
                         {w, bw, (uint64_t)es}};
    const int st = check_all(bufs, 2, [](int o, int j) { return (o == 0 && j == 2) || (o == 1 && j == 3); });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(x) && aligned16(residual) && aligned16(w) && aligned16(y) && aligned16(h) &&
                     (d * es) % 16 == 0;
    return finish(gbe::launch_rmsnorm(x, residual, w, y, h, rows, d, eps, dtype, vec, as_stream(stream)));
}

// One operand of a RoPE launch, as the entry points describe it.
struct RopeSide {
    const void* x;
    void* y;
    int64_t stride, H, r;
    const float* inv_freq;
    float mu;
    int layout;
};

// Shared checks and launch of gbe_rope, gbe_rope_qk and gbe_rope_pair: two
// operands (H = 0: absent) sharing positions, T, D and dtype, each with its
// own token stride, width, frequencies, scale and layout; a cos/sin table
// only when they share the last four.
static int rope_common(const RopeSide (&sd)[2], const int32_t* pos, int64_t T, int64_t D, const float* cos_sin,
                       int64_t cache_len, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    for (const RopeSide& o : sd)
        if (o.layout != 0 && o.layout != 1) return GBE_ERR_LAYOUT;
    if (T < 0 || D <= 0 || T > INT32_MAX || D > INT32_MAX) return GBE_ERR_SHAPE;
    for (const RopeSide& o : sd) {
        int64_t hd;
        if (o.H < 0 || !mul_ok(o.H, D, &hd) || hd > INT32_MAX / 2) return GBE_ERR_SHAPE;
        if (o.H > 0 && (o.stride < hd || o.stride > INT64_MAX / (T > 0 ? T : 1) / es)) return GBE_ERR_SHAPE;
    }
    for (const RopeSide& o : sd)
        if (o.r < 0 || o.r > D || (o.r & 1) || !std::isfinite(o.mu)) return GBE_ERR_ROTARY;
    if (cos_sin != nullptr && cache_len < 0) return GBE_ERR_SHAPE;
    Rows in[2], out[2];
    bool any = false, work = false;
    for (int k = 0; k < 2; ++k) {
        const int64_t rows = sd[k].H > 0 ? T : 0;
        in[k] = {sd[k].x, rows, sd[k].stride * es, sd[k].H * D * es};
        out[k] = {sd[k].y, rows, sd[k].stride * es, sd[k].H * D * es};
        any = any || rows > 0;
        work = work || (rows > 0 && !(sd[k].x == sd[k].y && sd[k].r == 0));  // in place with r = 0: nothing
    }
    if (!any) return GBE_OK;
    uint64_t bp, bf[2], bc = 0;
    if (!extent(T, 4, &bp)) return GBE_ERR_SHAPE;
    for (int k = 0; k < 2; ++k)
        if (!extent(sd[k].H > 0 ? sd[k].r / 2 : 0, 4, &bf[k])) return GBE_ERR_SHAPE;
    if (cos_sin != nullptr) {
        int64_t nc = 0;
        if (!mul_ok(cache_len, sd[0].r / 2, &nc) || !extent(nc, 8, &bc)) return GBE_ERR_SHAPE;
    }
    // 0, 1 = outputs; 2, 3 = inputs; 4 = pos; 5, 6 = the operands' frequencies; 7 = cos/sin table
    Buf bufs[8] = {out[0].extent(), out[1].extent(), in[0].extent(), in[1].extent(), {pos, bp, 4},
                   {sd[0].inv_freq, bf[0], 4}, {sd[1].inv_freq, bf[1], 4}, {cos_sin, cos_sin ? bc : 0u, 8}};
    for (int k = 0; k < 4; ++k) bufs[k].align = (uint64_t)es;
    for (const Buf& b : bufs) {
        const int st = check_form(b);
        if (st != GBE_OK) return st;
    }
    for (int o = 0; o < 2; ++o) {
        // an output may be exactly its own input; it may share no byte with
        // the other operand (input or output) nor with the small arrays
        if (rows_overlap(out[o], in[o]) && !rows_same(out[o], in[o])) return GBE_ERR_ALIAS;
        if (rows_overlap(out[o], in[1 - o]) || rows_overlap(out[o], out[1 - o])) return GBE_ERR_ALIAS;
        for (int j = 4; j < 8; ++j)
            if (overlaps(bufs[o], bufs[j])) return GBE_ERR_ALIAS;
    }
    Checker chk;
    if (const int st = chk.begin()) return st;
    for (const Buf& b : bufs) {
        const int st = chk.check(b);
        if (st != GBE_OK) return st;
    }
    if (!work) return GBE_OK;  // every operand in place with nothing to rotate
    bool vec = true;
    for (const RopeSide& o : sd)
        vec = vec && aligned16(o.x) && aligned16(o.y) && (o.stride * es) % 16 == 0;
    gbe::RopeArgs a;
    for (int k = 0; k < 2; ++k)
        a.side[k] = {sd[k].x, sd[k].y, sd[k].stride, sd[k].H > 0 ? sd[k].H : 0, sd[k].r, sd[k].inv_freq, sd[k].mu,
                     sd[k].layout};
    a.pos = pos;
    a.T = T;
    a.D = D;
    a.cos_sin = cos_sin;
    a.cache_len = cos_sin ? cache_len : 0;
    return finish(gbe::launch_rope(a, dtype, vec, as_stream(stream)));
}

int gbe_rope(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D, int64_t r,
             const float* inv_freq, float mu, int layout, int dtype, gbe_stream stream) {
    int64_t hd = 0;
    if (H > 0 && D > 0 && !mul_ok(H, D, &hd)) return GBE_ERR_SHAPE;
    const RopeSide sd[2] = {{x, y, hd, H, r, inv_freq, mu, layout}, {nullptr, nullptr, 0, 0, r, inv_freq, mu, layout}};
    return rope_common(sd, pos, T, D, nullptr, 0, dtype, stream);
}

int gbe_rope_qk(const void* q, void* q_out, int64_t q_stride, int64_t Hq, const void* k, void* k_out,
                int64_t k_stride, int64_t Hk, const int32_t* pos, int64_t T, int64_t D, int64_t r,
                const float* inv_freq, const float* cos_sin, int64_t cache_len, float mu, int layout, int dtype,
                gbe_stream stream) {
    const RopeSide sd[2] = {{q, q_out, q_stride, Hq, r, inv_freq, mu, layout},
                            {k, k_out, k_stride, Hk, r, inv_freq, mu, layout}};
    return rope_common(sd, pos, T, D, cos_sin, cache_len, dtype, stream);
}

int gbe_rope_pair(const gbe_rope_operand* a, const gbe_rope_operand* b, const int32_t* pos, int64_t T, int64_t D,
                  int dtype, gbe_stream stream) {
    if (a == nullptr) return GBE_ERR_NULL;
    const gbe_rope_operand none = {nullptr, nullptr, 0, 0, 0, nullptr, 1.0f, 0};
    const gbe_rope_operand& o2 = b ? *b : none;
    const RopeSide sd[2] = {{a->x, a->y, a->stride, a->H, a->r, a->inv_freq, a->mu, a->layout},
                            {o2.x, o2.y, o2.stride, o2.H, o2.r, o2.inv_freq, o2.mu, o2.layout}};
    return rope_common(sd, pos, T, D, nullptr, 0, dtype, stream);
}

int gbe_qk_norm_rope(const void* q, void* q_out, int64_t q_stride, int64_t Hq, const void* gq, const void* k,
                     void* k_out, int64_t k_stride, int64_t Hk, const void* gk, float eps, const int32_t* pos,
                     int64_t T, int64_t D, int64_t r, const float* inv_freq, const float* cos_sin,
                     int64_t cache_len, float mu, int layout, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (layout != 0 && layout != 1) return GBE_ERR_LAYOUT;
    if (T < 0 || D <= 0 || T > INT32_MAX || D > 64 * (16 / es)) return GBE_ERR_SHAPE;  // head_dim <= 64 chunks
    if (!std::isfinite(eps) || eps < 0.0f) return GBE_ERR_EPS;
    const int64_t Hs[2] = {Hq, Hk}, strides[2] = {q_stride, k_stride};
    for (int j = 0; j < 2; ++j) {
        int64_t hd;
        if (Hs[j] < 0 || !mul_ok(Hs[j], D, &hd) || hd > INT32_MAX / 2) return GBE_ERR_SHAPE;
        if (Hs[j] > 0 && (strides[j] < hd || strides[j] > INT64_MAX / (T > 0 ? T : 1) / es)) return GBE_ERR_SHAPE;
    }
    if (r < 0 || r > D || (r & 1) || !std::isfinite(mu)) return GBE_ERR_ROTARY;
    if (cos_sin != nullptr && cache_len < 0) return GBE_ERR_SHAPE;
    if ((Hq == 0 && Hk == 0) || T == 0) return GBE_OK;
    const int64_t half = r / 2;
    const void* xs[2] = {q, k};
    void* ys[2] = {q_out, k_out};
    const void* gs[2] = {gq, gk};
    Rows in[2], out[2];
    for (int j = 0; j < 2; ++j) {
        const int64_t rows = Hs[j] > 0 ? T : 0;
        in[j] = {xs[j], rows, strides[j] * es, Hs[j] * D * es};
        out[j] = {ys[j], rows, strides[j] * es, Hs[j] * D * es};
    }
    uint64_t bp, bf, bg, bc = 0;
    int64_t nc = 0;
    if (!extent(T, 4, &bp) || !extent(half, 4, &bf) || !extent(D, es, &bg)) return GBE_ERR_SHAPE;
    if (cos_sin != nullptr && (!mul_ok(cache_len, half, &nc) || !extent(nc, 8, &bc))) return GBE_ERR_SHAPE;
    // 0, 1 outputs; 2, 3 inputs; 4, 5 gains; 6 pos; 7 inv_freq; 8 table
    Buf bufs[9] = {out[0].extent(), out[1].extent(), in[0].extent(), in[1].extent(),
                   {gq, Hq > 0 ? bg : 0u, (uint64_t)es}, {gk, Hk > 0 ? bg : 0u, (uint64_t)es},
                   {pos, bp, 4}, {inv_freq, half > 0 ? bf : 0u, 4}, {cos_sin, cos_sin ? bc : 0u, 8}};
    for (int j = 0; j < 4; ++j) bufs[j].align = (uint64_t)es;
    for (const Buf& b : bufs) {
        const int st = check_form(b);
        if (st != GBE_OK) return st;
    }
    for (int o = 0; o < 2; ++o) {
        if (rows_overlap(out[o], in[o]) && !rows_same(out[o], in[o])) return GBE_ERR_ALIAS;
        if (rows_overlap(out[o], in[1 - o]) || rows_overlap(out[o], out[1 - o])) return GBE_ERR_ALIAS;
        for (int j = 4; j < 9; ++j)
            if (overlaps(bufs[o], bufs[j])) return GBE_ERR_ALIAS;
    }
    Checker chk;
    if (const int st = chk.begin()) return st;
    for (const Buf& b : bufs) {
        const int st = chk.check(b);
        if (st != GBE_OK) return st;
    }
    const bool vec = aligned16(q) && aligned16(q_out) && aligned16(k) && aligned16(k_out) &&
                     (Hq == 0 || aligned16(gq)) && (Hk == 0 || aligned16(gk)) && (q_stride * es) % 16 == 0 &&
                     (k_stride * es) % 16 == 0;
    gbe::QkNormRopeArgs a;
    for (int j = 0; j < 2; ++j) a.side[j] = {xs[j], ys[j], gs[j], strides[j], Hs[j]};
    a.eps = eps;
    a.pos = pos;
    a.T = T;
    a.D = D;
    a.r = r;
    a.inv_freq = inv_freq;
    a.cos_sin = cos_sin;
    a.cache_len = cos_sin ? cache_len : 0;
    a.mu = mu;
    a.layout = layout;
    return finish(gbe::launch_qk_norm_rope(a, dtype, vec, as_stream(stream)));
}

int gbe_rope_multi(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D, int64_t A,
                   const int64_t* dims, const float* inv_freq, float mu, int layout, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (layout != 0 && layout != 1) return GBE_ERR_LAYOUT;
    if (T < 0 || H < 0 || D <= 0 || A < 0 || A > gbe::kMaxAxes || T > INT32_MAX) return GBE_ERR_SHAPE;
    if (A > 0 && dims == nullptr) return GBE_ERR_NULL;
    if (!std::isfinite(mu)) return GBE_ERR_ROTARY;
    gbe::MultiAxis ax;
    ax.A = (int)A;
    int64_t total = 0;
    ax.poff[0] = 0;
    for (int64_t a = 0; a < A; ++a) {
        if (dims[a] < 0 || (dims[a] & 1) || dims[a] > D) return GBE_ERR_ROTARY;
        ax.off[a] = (int)total;
        total += dims[a];
        ax.poff[a + 1] = ax.poff[a] + (int)(dims[a] / 2);
    }
    if (total > D) return GBE_ERR_ROTARY;
    int64_t hd, n;
    if (!mul_ok(H, D, &hd) || hd > INT32_MAX / 2 || !mul_ok(T, hd, &n)) return GBE_ERR_SHAPE;
    uint64_t bx, bp, bf;
    if (!extent(n, es, &bx) || !extent(T * A, 4, &bp) || !extent(total / 2, 4, &bf)) return GBE_ERR_SHAPE;
    if (n == 0 || (x == y && total == 0)) return GBE_OK;
    const Buf bufs[4] = {{y, bx, (uint64_t)es}, {x, bx, (uint64_t)es}, {pos, bp, 4}, {inv_freq, bf, 4}};
    const int st = check_all(bufs, 1, [](int o, int j) { return o == 0 && j == 1; });
    if (st != GBE_OK) return st;
    return finish(gbe::launch_rope_multi(x, y, pos, T, H, D, ax, inv_freq, mu, layout, dtype, as_stream(stream)));
}

int gbe_rope_cos_sin(float* cos_sin, int64_t cache_len, int64_t r, const float* inv_freq, gbe_stream stream) {
    if (cache_len < 0 || cache_len > INT32_MAX || r < 0 || (r & 1) || r > INT32_MAX) {
        return cache_len < 0 ? GBE_ERR_SHAPE : GBE_ERR_ROTARY;
    }
    const int64_t half = r / 2;
    int64_t n;
    uint64_t bc, bf;
    if (!mul_ok(cache_len, half, &n) || !extent(n, 8, &bc) || !extent(half, 4, &bf)) return GBE_ERR_SHAPE;
    if (n == 0) return GBE_OK;
    const Buf bufs[2] = {{cos_sin, bc, 8}, {inv_freq, bf, 4}};
    const int st = check_all(bufs, 1, [](int, int) { return false; });
    if (st != GBE_OK) return st;
    return finish(gbe::launch_rope_cos_sin(cos_sin, cache_len, r, inv_freq, as_stream(stream)));
}

static int pointwise(const void* a, const void* b, void* y, int64_t n, int dtype, gbe_stream stream, bool silu) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    uint64_t bn;
    if (n < 0 || !extent(n, es, &bn)) return GBE_ERR_SHAPE;
    if (n == 0) return GBE_OK;
    const Buf bufs[3] = {{y, bn, (uint64_t)es}, {a, bn, (uint64_t)es}, {b, bn, (uint64_t)es}};
    const int st = check_all(bufs, 1, [](int o, int j) { return o == 0 && (j == 1 || j == 2); });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(a) && aligned16(b) && aligned16(y);
    return finish(silu ? gbe::launch_silu_mul(a, b, y, n, dtype, vec, as_stream(stream))
                       : gbe::launch_add(a, b, y, n, dtype, vec, as_stream(stream)));
}

int gbe_silu_mul(const void* gate, const void* up, void* y, int64_t n, int dtype, gbe_stream stream) {
    return pointwise(gate, up, y, n, dtype, stream, true);
}

int gbe_add(const void* a, const void* b, void* y, int64_t n, int dtype, gbe_stream stream) {
    return pointwise(a, b, y, n, dtype, stream, false);
}

int gbe_embedding(const void* table, const int32_t* ids, void* out, int64_t n, int64_t d, int64_t V,
                  int32_t* bad_id_count, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (n < 0 || d <= 0 || V < 0 || n > INT32_MAX || d > INT32_MAX) return GBE_ERR_SHAPE;
    int64_t no, nt;
    uint64_t bo, bt, bi;
    if (!mul_ok(n, d, &no) || !mul_ok(V, d, &nt) || !extent(no, es, &bo) || !extent(nt, es, &bt) ||
        !extent(n, 4, &bi))
        return GBE_ERR_SHAPE;
    if (n == 0) return GBE_OK;
    // outputs first: 0 = out, 1 = counter; then 2 = table, 3 = ids
    const Buf bufs[4] = {{out, bo, (uint64_t)es},
                         {bad_id_count, bad_id_count ? 4u : 0u, 4},
                         {table, bt, (uint64_t)es},
                         {ids, bi, 4}};
    const int st = check_all(bufs, 2, [](int, int) { return false; });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(table) && aligned16(out) && (d * es) % 16 == 0;
    return finish(
        gbe::launch_embedding(table, ids, out, n, d, V, bad_id_count, dtype, vec, as_stream(stream)));
}

int gbe_argmax(const void* x, int32_t* out, int64_t rows, int64_t n, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (rows < 0 || n < 0 || n > INT32_MAX || rows > (1LL << 28)) return GBE_ERR_SHAPE;
    if (rows == 0) return GBE_OK;
    if (n == 0) return GBE_ERR_EMPTY;
    int64_t nx;
    uint64_t bx, bo;
    if (!mul_ok(rows, n, &nx) || !extent(nx, es, &bx) || !extent(rows, 4, &bo)) return GBE_ERR_SHAPE;
    const Buf bufs[2] = {{out, bo, 4}, {x, bx, (uint64_t)es}};
    const int st = check_all(bufs, 1, [](int, int) { return false; });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(x) && (n * es) % 16 == 0;
    return finish(gbe::launch_argmax(x, out, rows, n, dtype, vec, as_stream(stream)));
}

// Shared checks and launch of gbe_sample (the caller's uniforms d.u) and
// gbe_sample_seeded (seeded: d.u is NULL and the seeded stream is drawn).
static int sample_common(const void* x, gbe::Draws d, bool seeded, int32_t* out, int64_t rows, int64_t n,
                         int method, float temperature, int64_t top_k, float p, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (method < GBE_SAMPLE_GREEDY || method > GBE_SAMPLE_MIN_P) return GBE_ERR_SAMPLING;
    const bool greedy = method == GBE_SAMPLE_GREEDY;
    if (!greedy && !(temperature > 0.0f && std::isfinite(temperature))) return GBE_ERR_SAMPLING;
    if (method == GBE_SAMPLE_TOP_K && top_k < 1) return GBE_ERR_SAMPLING;
    if ((method == GBE_SAMPLE_TOP_P || method == GBE_SAMPLE_MIN_P) && !(p >= 0.0f && p <= 1.0f))
        return GBE_ERR_SAMPLING;
    if (rows < 0 || n < 0 || n > (1LL << 23) || rows > (1LL << 28)) return GBE_ERR_SHAPE;
    if (rows == 0) return GBE_OK;
    if (n == 0) return GBE_ERR_EMPTY;
    int64_t nx;
    uint64_t bx, bo, bu;
    if (!mul_ok(rows, n, &nx) || !extent(nx, es, &bx) || !extent(rows, 4, &bo) || !extent(rows, 4, &bu))
        return GBE_ERR_SHAPE;
    if (greedy || seeded) bu = 0;  // u is not read
    const Buf bufs[3] = {{out, bo, 4}, {x, bx, (uint64_t)es}, {d.u, bu, 4}};
    const int st = check_all(bufs, 1, [](int, int) { return false; });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(x) && (n * es) % 16 == 0;
    return finish(gbe::launch_sample(x, out, rows, n, method, temperature, top_k, p, d, dtype, vec,
                                     as_stream(stream)));
}

int gbe_sample(const void* x, const float* u, int32_t* out, int64_t rows, int64_t n, int method,
               float temperature, int64_t top_k, float p, int dtype, gbe_stream stream) {
    const gbe::Draws d{u, 0ull, 0ull};
    return sample_common(x, d, false, out, rows, n, method, temperature, top_k, p, dtype, stream);
}

int gbe_sample_seeded(const void* x, int32_t* out, int64_t rows, int64_t n, int method, float temperature,
                      int64_t top_k, float p, uint64_t seed, uint64_t offset, int dtype, gbe_stream stream) {
    const gbe::Draws d{nullptr, (unsigned long long)seed, (unsigned long long)offset};
    return sample_common(x, d, true, out, rows, n, method, temperature, top_k, p, dtype, stream);
}

int gbe_pcg64_uniforms(float* u, int64_t n, uint64_t seed, uint64_t offset, gbe_stream stream) {
    uint64_t bu;
    if (n < 0 || !extent(n, 4, &bu)) return GBE_ERR_SHAPE;
    if (n == 0) return GBE_OK;
    const Buf bufs[1] = {{u, bu, 4}};
    const int st = check_all(bufs, 1, [](int, int) { return false; });
    if (st != GBE_OK) return st;
    return finish(gbe::launch_pcg64_uniforms(u, n, (unsigned long long)seed, (unsigned long long)offset,
                                             as_stream(stream)));
}

}  // extern "C"
