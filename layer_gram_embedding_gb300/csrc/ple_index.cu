// The per-token (request, offset) index kernel, the head-constant
// preparation kernel and the floored-remainder self-test kernel.
//
// The index is the (req[t], local[t]) pair through which the row-id kernel
// addresses the carried context (FreeToken PR #338, "perf(ple): fuse the
// n-gram row-id hash into one Triton kernel", section "What", second
// observation; section "Why it is safe": a decode is one token per request
// at offset 0).  Four consecutive tokens per thread and one 16-byte store of
// each output when the outputs are 16-byte aligned; a prefill thread finds
// its first token's request by binary search over cu_seqlens (staged in
// shared memory when it has at most 4096 entries) and walks forward for the
// other three.
#include <stdint.h>

#include "ple_divmod.cuh"
#include "ple_internal.h"

namespace ple {
namespace {

constexpr int kIndexThreads = 256;
constexpr int kTokPerThread = 4;     // one 16-byte store of req and of local
constexpr int kCuStaged = 4096;      // cu_seqlens entries kept in shared memory

template <bool kVec>
__device__ __forceinline__ void store4(int32_t* __restrict__ req, int32_t* __restrict__ local,
                                       int64_t t, int64_t T, const int (&r)[4], const int (&l)[4]) {
    if (kVec && t + 3 < T) {
        *reinterpret_cast<int4*>(req + t) = make_int4(r[0], r[1], r[2], r[3]);
        *reinterpret_cast<int4*>(local + t) = make_int4(l[0], l[1], l[2], l[3]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (t + k < T) {
                req[t + k] = r[k];
                local[t + k] = l[k];
            }
        }
    }
}

template <bool kVec>
__global__ void __launch_bounds__(kIndexThreads)
token_index_decode_kernel(int64_t T, int32_t* __restrict__ req, int32_t* __restrict__ local) {
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * kTokPerThread;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * kTokPerThread; t < T;
         t += stride) {
        const int r[4] = {(int)t, (int)t + 1, (int)t + 2, (int)t + 3};
        const int l[4] = {0, 0, 0, 0};
        store4<kVec>(req, local, t, T, r, l);
    }
}

// Request of token t: the last r in [0, B-1] with cu[r] <= t (empty requests
// own no token); the following tokens of the same thread walk forward.
template <bool kVec, bool kStaged>
__global__ void __launch_bounds__(kIndexThreads)
token_index_prefill_kernel(const int32_t* __restrict__ cu, int32_t B, int64_t T,
                           int32_t* __restrict__ req, int32_t* __restrict__ local) {
    // programmatic dependent launch, both ways: let a dependent row-id launch
    // become resident now (it waits for this grid before reading the index),
    // and wait for the previous kernel in the stream (which may still be
    // reading req / local) before touching memory
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();
    __shared__ int32_t cu_s[kStaged ? kCuStaged : 1];
    const int32_t* c = cu;
    if (kStaged) {
        for (int i = threadIdx.x; i <= B; i += blockDim.x) cu_s[i] = __ldg(cu + i);
        __syncthreads();
        c = cu_s;
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * kTokPerThread;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * kTokPerThread; t < T;
         t += stride) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = lo + ((hi - lo + 1) >> 1);
            if ((int64_t)c[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        int r[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t tk = t + k;
            while (lo < B - 1 && (int64_t)c[lo + 1] <= tk) ++lo;
            r[k] = lo;
            l[k] = (int)(tk - (int64_t)c[lo]);
        }
        store4<kVec>(req, local, t, T, r, l);
    }
}

// One rank's inputs of a batch split by token range (ple_shard_inputs): its
// cu_seqlens, rebased to its first token, and each of its requests' context
// row -- the first request's continued across the cut from the ids before
// it.  Thread j handles shard request j (and shard cu_seqlens entry j); every
// device-supplied index is clamped into its array.
template <typename IdT>
__global__ void __launch_bounds__(kIndexThreads)
shard_inputs_kernel(const IdT* __restrict__ ids, const int32_t* __restrict__ cu,
                    const IdT* __restrict__ ctx, int32_t B, int64_t T, int32_t C,
                    int64_t tok_begin, int64_t tok_end, int32_t req_begin, int32_t req_count,
                    int32_t* __restrict__ shard_cu, IdT* __restrict__ shard_ctx) {
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();
    const int64_t span = tok_end - tok_begin;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j <= req_count;
         j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = req_begin + j;  // <= B: checked on the host
        const int64_t start = __ldg(cu + r);
        shard_cu[j] = (int32_t)min(max(start - tok_begin, (int64_t)0), span);
        if (j == req_count) break;
        // tokens of request r before the cut, k: the carried row is the last
        // C ids of (context row r, those k tokens)
        const int64_t k = min(max(tok_begin - start, (int64_t)0), T);
        for (int c = 0; c < C; ++c) {
            const int64_t i = k + c;  // position in (context row, tokens)
            IdT v;
            if (i < C) {
                v = ctx[r * C + i];
            } else {
                const int64_t t = min(max(start + i - C, (int64_t)0), T - 1);
                v = ids[t];
            }
            shard_ctx[j * C + c] = v;
        }
    }
}

// First token whose (req, local) differs from the index cu_seqlens (or the
// decode rule) defines; *first_bad is lowered to it with an atomic min.
__global__ void __launch_bounds__(kIndexThreads)
validate_index_kernel(const int32_t* __restrict__ cu, int32_t B, int64_t T, int32_t is_decode,
                      const int32_t* __restrict__ req, const int32_t* __restrict__ local,
                      unsigned long long* __restrict__ first_bad) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t bad = INT64_MAX;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += stride) {
        int32_t r_exp, l_exp;
        if (is_decode) {
            r_exp = (int32_t)t;
            l_exp = 0;
        } else {
            int lo = 0, hi = B - 1;
            while (lo < hi) {
                const int mid = lo + ((hi - lo + 1) >> 1);
                if ((int64_t)__ldg(cu + mid) <= t)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            r_exp = lo;
            l_exp = (int32_t)(t - (int64_t)__ldg(cu + lo));
        }
        if (__ldg(req + t) != r_exp || __ldg(local + t) != l_exp) {
            bad = t;
            break;  // later tokens of this thread are larger
        }
    }
    if (bad != INT64_MAX) atomicMin(first_bad, (unsigned long long)bad);
}

__global__ void __launch_bounds__(kIndexThreads)
selftest_floor_mod_kernel(const int64_t* __restrict__ x, const int64_t* __restrict__ v, int64_t n,
                          int64_t* __restrict__ out_fast, int64_t* __restrict__ out_ref) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t xi = x[i], vi = v[i];
        // the library's routine, exactly as the row-id kernel runs it
        const HeadConst c = make_head_const(vi, 0);
        const OffsetBinary u = offset_binary((uint64_t)xi);
        out_fast[i] = (c.ext.z == kHeadFast) ? row_fast(u, c.fast, 0)
                                             : row_general(u, c.fast, 0, c.ext);
        // CUDA's truncating % with the floored sign fix
        int64_t r = 0;
        if (vi != 0 && vi != -1) {
            r = xi % vi;
            if (r != 0 && ((r < 0) != (vi < 0))) r += vi;
        }
        out_ref[i] = r;
    }
}

// One head per thread: the constants the row-id kernels would derive from
// (vocab, offset) at every call, stored once (three 16-byte words a head).
__global__ void __launch_bounds__(kIndexThreads)
prepare_heads_kernel(const int64_t* __restrict__ vocab, const int64_t* __restrict__ offsets,
                     int64_t n, void* __restrict__ heads) {
    cudaTriggerProgrammaticLaunchCompletion();
    cudaGridDependencySynchronize();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride)
        store_head_const(heads, k, make_head_const(vocab[k], offsets[k]));
}

unsigned grid_for(int64_t n, const DeviceFacts& dev) {
    int64_t blocks = (n + kIndexThreads - 1) / kIndexThreads;
    const int64_t cap = 8 * (int64_t)dev.sm_count;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (unsigned)blocks;
}

}  // namespace

// Launch with programmatic stream serialization (see the kernels) unless it
// is turned off; the diagnostics launch plainly.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*fn)(KArgs...), unsigned grid, cudaStream_t stream, Args... args) {
    return launch_kernel(fn, dim3(grid), dim3(kIndexThreads), 0, stream, programmatic_launch(),
                         args...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*fn)(KArgs...), unsigned grid, cudaStream_t stream, Args... args) {
    return launch_kernel(fn, dim3(grid), dim3(kIndexThreads), 0, stream, false, args...);
}

cudaError_t launch_token_index(const int32_t* cu, int32_t B, int64_t T, int32_t is_decode,
                               int32_t* req, int32_t* local, const DeviceFacts& dev,
                               cudaStream_t stream) {
    const unsigned g = grid_for((T + kTokPerThread - 1) / kTokPerThread, dev);
    const bool vec = ((uintptr_t)req % 16 == 0) && ((uintptr_t)local % 16 == 0);
    const bool staged = (int64_t)B + 1 <= kCuStaged;
    cudaError_t e;
    if (is_decode) {
        e = vec ? launch_pdl(token_index_decode_kernel<true>, g, stream, T, req, local)
                : launch_pdl(token_index_decode_kernel<false>, g, stream, T, req, local);
    } else if (vec) {
        e = staged ? launch_pdl(token_index_prefill_kernel<true, true>, g, stream, cu, B, T, req, local)
                   : launch_pdl(token_index_prefill_kernel<true, false>, g, stream, cu, B, T, req, local);
    } else {
        e = staged ? launch_pdl(token_index_prefill_kernel<false, true>, g, stream, cu, B, T, req, local)
                   : launch_pdl(token_index_prefill_kernel<false, false>, g, stream, cu, B, T, req, local);
    }
    return e;
}

cudaError_t launch_shard_inputs(const void* ids, int id_bytes, const int32_t* cu,
                                const void* ctx, int32_t B, int64_t T, int32_t C,
                                int64_t tok_begin, int64_t tok_end, int32_t req_begin,
                                int32_t req_count, int32_t* shard_cu, void* shard_ctx,
                                cudaStream_t stream) {
    const unsigned g = (unsigned)((req_count + kIndexThreads) / kIndexThreads);
    if (id_bytes == 4)
        return launch_pdl(shard_inputs_kernel<int32_t>, g, stream,
                          static_cast<const int32_t*>(ids), cu, static_cast<const int32_t*>(ctx),
                          B, T, C, tok_begin, tok_end, req_begin, req_count, shard_cu,
                          static_cast<int32_t*>(shard_ctx));
    return launch_pdl(shard_inputs_kernel<int64_t>, g, stream, static_cast<const int64_t*>(ids),
                      cu, static_cast<const int64_t*>(ctx), B, T, C, tok_begin, tok_end, req_begin,
                      req_count, shard_cu, static_cast<int64_t*>(shard_ctx));
}

cudaError_t launch_validate_index(const int32_t* cu, int32_t B, int64_t T, int32_t is_decode,
                                  const int32_t* req, const int32_t* local, int64_t* first_bad,
                                  const DeviceFacts& dev, cudaStream_t stream) {
    return launch_plain(validate_index_kernel, grid_for(T, dev), stream, cu, B, T, is_decode, req,
                        local, reinterpret_cast<unsigned long long*>(first_bad));
}

cudaError_t launch_prepare_heads(const int64_t* vocab, const int64_t* offsets, int64_t n,
                                 void* heads, const DeviceFacts& dev, cudaStream_t stream) {
    return launch_pdl(prepare_heads_kernel, grid_for(n, dev), stream, vocab, offsets, n, heads);
}

cudaError_t launch_selftest_floor_mod(const int64_t* x, const int64_t* v, int64_t n,
                                      int64_t* out_fast, int64_t* out_ref, const DeviceFacts& dev,
                                      cudaStream_t stream) {
    return launch_plain(selftest_floor_mod_kernel, grid_for(n, dev), stream, x, v, n, out_fast,
                        out_ref);
}

}  // namespace ple
