// abi.cu -- the C entry points declared in include/gbe_elementwise.h.
//
// Every argument is validated here, on the host, before anything is
// enqueued: sizes and scalars, pointer alignment, that each non-empty buffer
// is memory the current device can address and that its extent stays inside
// its allocation, and that outputs overlap nothing but their permitted exact
// aliases.  Only then is the launcher of the op called.  Nothing here
// allocates, frees or waits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <mutex>

#include "gbe_elementwise.h"
#include "launch.h"

namespace {

constexpr int kVersion = 10000;  // 1.0.0

thread_local int t_last_cuda_error = 0;

int elem_size(int dtype) { return dtype == GBE_F32 ? 4 : dtype == GBE_BF16 ? 2 : 0; }

typedef CUresult (*AddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);

AddressRangeFn address_range_fn() {
    static std::once_flag once;
    static AddressRangeFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AddressRangeFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// One buffer of a call: where it starts and how many bytes the call touches.
struct Buf {
    const void* p;
    uint64_t bytes;
    uint64_t align;
};

int check_buf(const Buf& b, int dev) {
    if (b.bytes == 0) return GBE_OK;
    if (b.p == nullptr) return GBE_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(b.p) % b.align) return GBE_ERR_ALIGN;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, b.p) != cudaSuccess) {
        cudaGetLastError();
        return GBE_ERR_POINTER;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice:
            if (a.device != dev) return GBE_ERR_POINTER;
            break;
        case cudaMemoryTypeManaged:
            break;
        case cudaMemoryTypeHost:  // pinned host memory, usable only when mapped at the same address
            if (a.devicePointer != b.p) return GBE_ERR_POINTER;
            break;
        default:
            return GBE_ERR_POINTER;
    }
    if (a.type != cudaMemoryTypeHost) {
        if (AddressRangeFn fn = address_range_fn()) {
            CUdeviceptr base = 0;
            size_t size = 0;
            const CUdeviceptr p = reinterpret_cast<CUdeviceptr>(b.p);
            if (fn(&base, &size, p) == CUDA_SUCCESS) {
                if (p + b.bytes > base + size || p + b.bytes < p) return GBE_ERR_POINTER;
            }
        }
    }
    return GBE_OK;
}

bool overlaps(const Buf& a, const Buf& b) {
    if (a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a.p), y = reinterpret_cast<uintptr_t>(b.p);
    return x < y + b.bytes && y < x + a.bytes;
}

bool same(const Buf& a, const Buf& b) { return a.p == b.p && a.bytes == b.bytes; }

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

// Validate the buffers of one call: each one alone, then every output (the
// first n_out entries) against every other buffer; `alias_ok(o, j)` says
// whether output o may be exactly buffer j.
template <int N, typename AliasOk>
int check_all(const Buf (&bufs)[N], int n_out, AliasOk alias_ok) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        t_last_cuda_error = (int)cudaGetLastError();
        return GBE_ERR_CUDA;
    }
    for (int i = 0; i < N; ++i) {
        const int st = check_buf(bufs[i], dev);
        if (st != GBE_OK) return st;
    }
    for (int o = 0; o < n_out; ++o)
        for (int j = 0; j < N; ++j) {
            if (j == o || !overlaps(bufs[o], bufs[j])) continue;
            if (!(alias_ok(o, j) && same(bufs[o], bufs[j]))) return GBE_ERR_ALIAS;
        }
    return GBE_OK;
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

int gbe_rope(const void* x, void* y, const int32_t* pos, int64_t T, int64_t H, int64_t D, int64_t r,
             const float* inv_freq, float mu, int layout, int dtype, gbe_stream stream) {
    const int es = elem_size(dtype);
    if (!es) return GBE_ERR_DTYPE;
    if (layout != 0 && layout != 1) return GBE_ERR_LAYOUT;
    if (T < 0 || H < 0 || D <= 0 || T > INT32_MAX) return GBE_ERR_SHAPE;
    int64_t hd, n;
    if (!mul_ok(H, D, &hd) || hd > INT32_MAX / 2 || !mul_ok(T, hd, &n)) return GBE_ERR_SHAPE;
    if (r < 0 || r > D || (r & 1) || !std::isfinite(mu)) return GBE_ERR_ROTARY;
    uint64_t bx, bp, bf;
    if (!extent(n, es, &bx) || !extent(T, 4, &bp) || !extent(r / 2, 4, &bf)) return GBE_ERR_SHAPE;
    if (n == 0) return GBE_OK;
    if (x == y && r == 0) {  // in place with nothing to rotate: still validate the buffer
        const Buf b[1] = {{y, bx, (uint64_t)es}};
        return check_all(b, 0, [](int, int) { return false; });
    }
    const Buf bufs[4] = {{y, bx, (uint64_t)es}, {x, bx, (uint64_t)es}, {pos, bp, 4}, {inv_freq, bf, 4}};
    const int st = check_all(bufs, 1, [](int o, int j) { return o == 0 && j == 1; });
    if (st != GBE_OK) return st;
    const bool vec = aligned16(x) && aligned16(y);
    return finish(gbe::launch_rope(x, y, pos, T, H, D, r, inv_freq, mu, layout, dtype, vec, as_stream(stream)));
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

}  // extern "C"
