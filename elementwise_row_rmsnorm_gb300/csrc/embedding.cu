// embedding.cu -- embedding-row gather on sm_103a.
//
// Definition ("Elementwise kernels in C", section 2.4; "Operations",
// section 3, TokenEmbed): output row t is row ids[t] of the [V, d] table,
// whose first element sits at ids[t] * d.  The pages leave the id check to
// the caller; on a shared GPU an id outside [0, V) must never turn into an
// out-of-range read, so such a row is not read: it is written as zeros and,
// when the caller passes a counter, the counter is incremented once per bad
// row.  Valid rows are copied bit for bit.
//
// Map: one row per TPR threads (several one-warp rows per CTA when d is
// small); a row is cut into 16-byte chunks, chunk c goes to thread c mod TPR
// as its (c div TPR)-th slot (at most 8 slots), and all slot loads are
// issued before the stores.
#include "common.cuh"
#include "launch.h"

namespace gbe {

namespace {

template <int ES, int K, bool VEC, int MAXT>
__global__ void __launch_bounds__(MAXT)
embedding_rows(const void* table, const int32_t* ids, void* out, int64_t n, int64_t d, int64_t V, int32_t* bad,
               int tpr) {
    constexpr int VE = 16 / ES;  // elements per 16-byte chunk
    pdl_begin();
    const int rpc = blockDim.x / tpr;
    const int sub = threadIdx.x / tpr;
    const int t = threadIdx.x - sub * tpr;
    const int64_t row = (int64_t)blockIdx.x * rpc + sub;
    if (row >= n) return;
    const int64_t id = ids[row];
    const int64_t nbytes = d * ES;
    char* dst = static_cast<char*>(out) + row * nbytes;
    if (id < 0 || id >= V) {
        for (int64_t b = t; b < nbytes; b += tpr) dst[b] = 0;
        if (t == 0 && bad != nullptr) atomicAdd(bad, 1);
        return;
    }
    const char* src = static_cast<const char*>(table) + id * nbytes;
    if (VEC) {
        const int64_t nchunks = d / VE;
        if (K > 0) {
            Vec16 r[K > 0 ? K : 1];
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t c = (int64_t)k * tpr + t;
                if (c < nchunks) r[k] = ld_stream(src + c * 16);
            }
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t c = (int64_t)k * tpr + t;
                if (c < nchunks) st_stream(dst + c * 16, r[k]);
            }
        } else {  // very wide rows: stream chunk by chunk
            for (int64_t c = t; c < nchunks; c += tpr) st_stream(dst + c * 16, ld_stream(src + c * 16));
        }
    } else {
        if (ES == 4) {
            const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src);
            uint32_t* d4 = reinterpret_cast<uint32_t*>(dst);
            for (int64_t i = t; i < d; i += tpr) d4[i] = s4[i];
        } else {
            const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src);
            uint16_t* d2 = reinterpret_cast<uint16_t*>(dst);
            for (int64_t i = t; i < d; i += tpr) d2[i] = s2[i];
        }
    }
}

template <int ES>
cudaError_t launch_es(const void* table, const int32_t* ids, void* out, int64_t n, int64_t d, int64_t V,
                      int32_t* bad, bool vec, cudaStream_t st) {
    constexpr int VE = 16 / ES;
    const int64_t nchunks = (d + VE - 1) / VE;
    // enough threads per row that each owns at most 8 chunks (all 8 loads in flight)
    int64_t tpr = ((nchunks + 7) / 8 + 31) / 32 * 32;
    if (tpr < 32) tpr = 32;
    const bool wide = tpr > 1024;
    if (wide) tpr = 1024;
    const int64_t slots = (nchunks + tpr - 1) / tpr;
    const int rpc = tpr == 32 ? 4 : 1;
    const int64_t grid = (n + rpc - 1) / rpc;
    const dim3 block((unsigned)(tpr * rpc));
    const int ti = (int)tpr;
    const dim3 g((unsigned)grid);
    if (!vec) return launch(embedding_rows<ES, 0, false, 1024>, g, block, 0, st, table, ids, out, n, d, V, bad, ti);
    if (wide) return launch(embedding_rows<ES, 0, true, 1024>, g, block, 0, st, table, ids, out, n, d, V, bad, ti);
#define GBE_EMB_CASE(KK, MT)                                                                                 \
    if (slots <= KK)                                                                                         \
        return launch(embedding_rows<ES, KK, true, MT>, g, block, 0, st, table, ids, out, n, d, V, bad, ti);
    if (tpr * rpc <= 256) {
        GBE_EMB_CASE(1, 256)
        GBE_EMB_CASE(2, 256)
        GBE_EMB_CASE(4, 256)
        GBE_EMB_CASE(8, 256)
    } else {
        GBE_EMB_CASE(8, 1024)
    }
#undef GBE_EMB_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_embedding(const void* table, const int32_t* ids, void* out, int64_t n, int64_t d, int64_t V,
                             int32_t* bad_id_count, int dtype, bool vec, cudaStream_t st) {
    if (dtype == kF32) return launch_es<4>(table, ids, out, n, d, V, bad_id_count, vec, st);
    return launch_es<2>(table, ids, out, n, d, V, bad_id_count, vec, st);
}

}  // namespace gbe
