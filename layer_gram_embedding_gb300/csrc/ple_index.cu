// The per-token (request, offset) index kernel and the floored-remainder
// self-test kernel.
//
// The index is the (req[t], local[t]) pair through which the row-id kernel
// addresses the carried context (FreeToken PR #338, "perf(ple): fuse the
// n-gram row-id hash into one Triton kernel", section "What", second
// observation; section "Why it is safe": a decode is one token per request
// at offset 0).  One thread per token; a prefill token finds its request by
// binary search over cu_seqlens (the last r with cu_seqlens[r] <= t, which
// skips empty requests).  Writes are coalesced int32 stores.
#include <stdint.h>

#include "ple_divmod.cuh"
#include "ple_internal.h"

namespace ple {
namespace {

constexpr int kIndexThreads = 256;

__global__ void __launch_bounds__(kIndexThreads)
token_index_decode_kernel(int64_t T, int32_t* __restrict__ req, int32_t* __restrict__ local) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += stride) {
        req[t] = (int32_t)t;
        local[t] = 0;
    }
}

__global__ void __launch_bounds__(kIndexThreads)
token_index_prefill_kernel(const int32_t* __restrict__ cu, int32_t B, int64_t T,
                           int32_t* __restrict__ req, int32_t* __restrict__ local) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += stride) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = lo + ((hi - lo + 1) >> 1);
            if ((int64_t)__ldg(cu + mid) <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        req[t] = lo;
        local[t] = (int32_t)(t - (int64_t)__ldg(cu + lo));
    }
}

__global__ void __launch_bounds__(kIndexThreads)
selftest_floor_mod_kernel(const int64_t* __restrict__ x, const int64_t* __restrict__ v, int64_t n,
                          int64_t* __restrict__ out_fast, int64_t* __restrict__ out_ref) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t xi = x[i], vi = v[i];
        // the library's routine, exactly as the row-id kernel runs it
        const HeadConst c = make_head_const(vi, 0);
        const Magnitude m = magnitude(xi);
        out_fast[i] = (c.kind == kHeadFast) ? row_fast_positive(m, c.m_lo, c.m_hi, c.v_lo, 0)
                                            : row_general(m, c);
        // CUDA's truncating % with the floored sign fix
        int64_t r = 0;
        if (vi != 0 && vi != -1) {
            r = xi % vi;
            if (r != 0 && ((r < 0) != (vi < 0))) r += vi;
        }
        out_ref[i] = r;
    }
}

unsigned grid_for(int64_t n, const DeviceFacts& dev) {
    int64_t blocks = (n + kIndexThreads - 1) / kIndexThreads;
    const int64_t cap = 8 * (int64_t)dev.sm_count;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (unsigned)blocks;
}

}  // namespace

cudaError_t launch_token_index(const int32_t* cu, int32_t B, int64_t T, int32_t is_decode,
                               int32_t* req, int32_t* local, const DeviceFacts& dev,
                               cudaStream_t stream) {
    const unsigned g = grid_for(T, dev);
    if (is_decode)
        token_index_decode_kernel<<<g, kIndexThreads, 0, stream>>>(T, req, local);
    else
        token_index_prefill_kernel<<<g, kIndexThreads, 0, stream>>>(cu, B, T, req, local);
    return cudaGetLastError();
}

cudaError_t launch_selftest_floor_mod(const int64_t* x, const int64_t* v, int64_t n,
                                      int64_t* out_fast, int64_t* out_ref, const DeviceFacts& dev,
                                      cudaStream_t stream) {
    selftest_floor_mod_kernel<<<grid_for(n, dev), kIndexThreads, 0, stream>>>(x, v, n, out_fast,
                                                                              out_ref);
    return cudaGetLastError();
}

}  // namespace ple
