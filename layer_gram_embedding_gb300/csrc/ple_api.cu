// C ABI of the PLE n-gram row-id hash library (declared in include/ple.h).
//
// Every entry point validates its scalar arguments and pointer values on the
// host, then enqueues exactly one kernel on the caller's stream and reports
// that launch's own status; the caller's pending CUDA error state is left as
// it was.  Nothing is allocated, nothing is read back, nothing is cached
// except per-device facts (SM count, shared-memory limit) looked up once and
// the process-wide programmatic-launch switch.
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "ple.h"
#include "ple_internal.h"

namespace ple {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_facts_mu;
bool g_facts_ok[kMaxDevices];
DeviceFacts g_facts[kMaxDevices];
std::atomic<int> g_programmatic{1};
}  // namespace

bool programmatic_launch() { return g_programmatic.load(std::memory_order_relaxed) != 0; }

cudaError_t device_facts(DeviceFacts* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_facts_mu);
    if (!g_facts_ok[dev]) {
        DeviceFacts f;
        e = cudaDeviceGetAttribute(&f.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&f.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        g_facts[dev] = f;
        g_facts_ok[dev] = true;
    }
    *out = g_facts[dev];
    return cudaSuccess;
}

}  // namespace ple

namespace {

thread_local int32_t g_last_cuda_error = 0;

ple_status cuda_failure(cudaError_t e) {
    g_last_cuda_error = (int32_t)e;
    return PLE_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" ple_status ple_build_token_index(const int32_t* cu_seqlens, int32_t num_requests,
                                            int64_t num_tokens, int32_t is_decode, int32_t* req,
                                            int32_t* local, void* stream) {
    if (num_tokens < 0 || num_tokens > INT32_MAX) return PLE_ERR_SIZE;
    if (num_tokens == 0) return PLE_OK;
    if (num_requests < 1) return PLE_ERR_SIZE;
    if (is_decode && (int64_t)num_requests != num_tokens) return PLE_ERR_SIZE;
    if (!req || !local || (!is_decode && !cu_seqlens)) return PLE_ERR_NULL;
    if (!aligned(req, 4) || !aligned(local, 4) || (!is_decode && !aligned(cu_seqlens, 4)))
        return PLE_ERR_ALIGN;
    ple::DeviceFacts dev;
    cudaError_t e = ple::device_facts(&dev);
    if (e != cudaSuccess) return cuda_failure(e);
    e = ple::launch_token_index(cu_seqlens, num_requests, num_tokens, is_decode, req, local, dev,
                                static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e);
    return PLE_OK;
}

namespace {

// Checks the arguments every row-id entry point shares and fills the kernel
// parameters.  Returns PLE_OK with *empty set when there is nothing to do.
ple_status check_row_args(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                          const int32_t* req, const int32_t* local, const void* ngram_context,
                          int32_t num_requests, int32_t ctx_len,
                          const int64_t* layer_multipliers, const int64_t* vocab_sizes,
                          const int64_t* offsets, int32_t num_heads, int32_t ngram_size,
                          int32_t heads_per_ngram, int32_t num_layers, int64_t boundary_id,
                          const int32_t* cu_seqlens, const void* heads, ple::RowIdsParams* p,
                          bool* empty) {
    *empty = false;
    // sizes first, then the page's two geometry preconditions
    if (ngram_size < 2 || ngram_size > PLE_MAX_NGRAM || heads_per_ngram < 1 || num_layers < 1 ||
        num_tokens < 0 || num_tokens > INT32_MAX)
        return PLE_ERR_SIZE;
    if (ctx_len != ngram_size - 1) return PLE_ERR_GEOMETRY_CTX;
    if ((int64_t)num_heads != (int64_t)(ngram_size - 1) * heads_per_ngram)
        return PLE_ERR_GEOMETRY_HEADS;
    if (num_heads > PLE_MAX_HEADS) return PLE_ERR_SIZE;
    // the output's byte count, L * T * H int64, fits int64 (L * T < 2^62)
    if ((int64_t)num_layers * num_tokens > (INT64_MAX / 8) / num_heads) return PLE_ERR_SIZE;
    if (num_tokens == 0) {
        *empty = true;
        return PLE_OK;
    }
    if (num_requests < 1) return PLE_ERR_SIZE;
    // both index pointers NULL: the kernel finds each token's request itself,
    // by searching cu_seqlens when given, else as a decode batch (one token
    // per request at offset 0)
    const bool index_free = !req && !local;
    const int32_t mode = !index_free ? ple::kIdxArrays
                                     : (cu_seqlens ? ple::kIdxCu : ple::kIdxDecode);
    if (mode == ple::kIdxDecode && (int64_t)num_requests != num_tokens) return PLE_ERR_SIZE;
    // prepared head constants replace vocab_sizes and offsets
    if (!input_ids || (!index_free && (!req || !local)) || !ngram_context || !layer_multipliers ||
        (!heads && (!vocab_sizes || !offsets)))
        return PLE_ERR_NULL;
    if (id_dtype != PLE_I32 && id_dtype != PLE_I64) return PLE_ERR_DTYPE;
    const int id_bytes = id_dtype == PLE_I32 ? 4 : 8;
    if (!aligned(input_ids, id_bytes) || !aligned(ngram_context, id_bytes) || !aligned(req, 4) ||
        !aligned(local, 4) || !aligned(layer_multipliers, 8) || !aligned(vocab_sizes, 8) ||
        !aligned(offsets, 8) || !aligned(heads, 16) || !aligned(cu_seqlens, 4))
        return PLE_ERR_ALIGN;
    p->ids = input_ids;
    p->req = req;
    p->local = local;
    p->ctx = ngram_context;
    p->mult = layer_multipliers;
    p->vocab = vocab_sizes;
    p->offsets = offsets;
    p->out = nullptr;
    p->T = num_tokens;
    p->boundary = boundary_id;
    p->B = num_requests;
    p->N = ngram_size;
    p->hpn = heads_per_ngram;
    p->H = num_heads;
    p->L = num_layers;
    p->ids_vec_ok = aligned(input_ids, 16) ? 1 : 0;
    p->out_vec_ok = 0;
    p->index_mode = mode;
    p->out_bytes = 8;
    p->cu = cu_seqlens;
    p->next_ctx = nullptr;
    p->heads = heads;
    p->ones = 0xFFFFFFFFu;
    return PLE_OK;
}

ple_status row_ids_impl(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                        const int32_t* req, const int32_t* local, const void* ngram_context,
                        int32_t num_requests, int32_t ctx_len, const int64_t* layer_multipliers,
                        const int64_t* vocab_sizes, const int64_t* offsets, int32_t num_heads,
                        int32_t ngram_size, int32_t heads_per_ngram, int32_t num_layers,
                        int64_t boundary_id, void* out, int out_bytes, const int32_t* cu_seqlens,
                        void* next_context, const void* heads, void* stream) {
    ple::RowIdsParams p;
    bool empty = false;
    ple_status st = check_row_args(input_ids, id_dtype, num_tokens, req, local, ngram_context,
                                   num_requests, ctx_len, layer_multipliers, vocab_sizes, offsets,
                                   num_heads, ngram_size, heads_per_ngram, num_layers, boundary_id,
                                   cu_seqlens, heads, &p, &empty);
    if (st != PLE_OK) return st;
    if (out_bytes != 4 && out_bytes != 8) return PLE_ERR_DTYPE;
    if (empty) return PLE_OK;
    if (!out) return PLE_ERR_NULL;
    // the carry finds each request's last token (and empty requests) through
    // cu_seqlens, except in a decode without an index
    if (next_context && p.index_mode == ple::kIdxArrays && !cu_seqlens) return PLE_ERR_NULL;
    const int id_bytes = id_dtype == PLE_I32 ? 4 : 8;
    if (!aligned(out, out_bytes) || !aligned(next_context, id_bytes)) return PLE_ERR_ALIGN;

    ple::DeviceFacts dev;
    cudaError_t e = ple::device_facts(&dev);
    if (e != cudaSuccess) return cuda_failure(e);
    p.out = out;
    p.out_vec_ok = aligned(out, 16) ? 1 : 0;
    p.out_bytes = out_bytes;
    p.next_ctx = next_context;
    const ple::RowIdsLaunch cfg = ple::plan_row_ids(p, dev);
    if (cfg.grid.y > 65535u) return PLE_ERR_SIZE;
    e = ple::launch_row_ids(p, id_bytes, cfg, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e);
    return PLE_OK;
}

}  // namespace

extern "C" ple_status ple_row_ids(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                                  const int32_t* req, const int32_t* local,
                                  const void* ngram_context, int32_t num_requests,
                                  int32_t ctx_len, const int64_t* layer_multipliers,
                                  const int64_t* vocab_sizes, const int64_t* offsets,
                                  int32_t num_heads, int32_t ngram_size, int32_t heads_per_ngram,
                                  int32_t num_layers, int64_t boundary_id, int64_t* out,
                                  void* stream) {
    return row_ids_impl(input_ids, id_dtype, num_tokens, req, local, ngram_context, num_requests,
                        ctx_len, layer_multipliers, vocab_sizes, offsets, num_heads, ngram_size,
                        heads_per_ngram, num_layers, boundary_id, out, 8, nullptr, nullptr,
                        nullptr, stream);
}

extern "C" ple_status ple_row_ids_i32(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                                      const int32_t* req, const int32_t* local,
                                      const void* ngram_context, int32_t num_requests,
                                      int32_t ctx_len, const int64_t* layer_multipliers,
                                      const int64_t* vocab_sizes, const int64_t* offsets,
                                      int32_t num_heads, int32_t ngram_size,
                                      int32_t heads_per_ngram, int32_t num_layers,
                                      int64_t boundary_id, int32_t* out, void* stream) {
    return row_ids_impl(input_ids, id_dtype, num_tokens, req, local, ngram_context, num_requests,
                        ctx_len, layer_multipliers, vocab_sizes, offsets, num_heads, ngram_size,
                        heads_per_ngram, num_layers, boundary_id, out, 4, nullptr, nullptr,
                        nullptr, stream);
}

extern "C" ple_status ple_row_ids_ex(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                                     const int32_t* req, const int32_t* local,
                                     const void* ngram_context, int32_t num_requests,
                                     int32_t ctx_len, const int64_t* layer_multipliers,
                                     const int64_t* vocab_sizes, const int64_t* offsets,
                                     int32_t num_heads, int32_t ngram_size,
                                     int32_t heads_per_ngram, int32_t num_layers,
                                     int64_t boundary_id, void* out, int32_t out_dtype,
                                     const int32_t* cu_seqlens, void* next_context,
                                     const void* heads, void* stream) {
    const int out_bytes = out_dtype == PLE_I32 ? 4 : out_dtype == PLE_I64 ? 8 : 0;
    return row_ids_impl(input_ids, id_dtype, num_tokens, req, local, ngram_context, num_requests,
                        ctx_len, layer_multipliers, vocab_sizes, offsets, num_heads, ngram_size,
                        heads_per_ngram, num_layers, boundary_id, out, out_bytes, cu_seqlens,
                        next_context, heads, stream);
}

extern "C" ple_status ple_prepare_heads(const int64_t* vocab_sizes, const int64_t* offsets,
                                        int32_t num_layers, int32_t num_heads, void* heads,
                                        void* stream) {
    if (num_layers < 1 || num_heads < 1 || num_heads > PLE_MAX_HEADS) return PLE_ERR_SIZE;
    if (!vocab_sizes || !offsets || !heads) return PLE_ERR_NULL;
    if (!aligned(vocab_sizes, 8) || !aligned(offsets, 8) || !aligned(heads, 16))
        return PLE_ERR_ALIGN;
    ple::DeviceFacts dev;
    cudaError_t e = ple::device_facts(&dev);
    if (e != cudaSuccess) return cuda_failure(e);
    e = ple::launch_prepare_heads(vocab_sizes, offsets, (int64_t)num_layers * num_heads, heads,
                                  dev, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e);
    return PLE_OK;
}

extern "C" ple_status ple_row_embed(const void* input_ids, int32_t id_dtype, int64_t num_tokens,
                                    const int32_t* req, const int32_t* local,
                                    const void* ngram_context, int32_t num_requests,
                                    int32_t ctx_len, const int64_t* layer_multipliers,
                                    const int64_t* vocab_sizes, const int64_t* offsets,
                                    int32_t num_heads, int32_t ngram_size,
                                    int32_t heads_per_ngram, int32_t num_layers,
                                    int64_t boundary_id, const void* table, int64_t table_rows,
                                    int32_t dim, float* out, const int32_t* cu_seqlens,
                                    const void* heads, void* stream) {
    ple::RowIdsParams p;
    bool empty = false;
    ple_status st = check_row_args(input_ids, id_dtype, num_tokens, req, local, ngram_context,
                                   num_requests, ctx_len, layer_multipliers, vocab_sizes, offsets,
                                   num_heads, ngram_size, heads_per_ngram, num_layers, boundary_id,
                                   cu_seqlens, heads, &p, &empty);
    if (st != PLE_OK) return st;
    if (dim < 8 || dim % 8 != 0 || dim > PLE_MAX_EMBED_DIM || table_rows < 0) return PLE_ERR_SIZE;
    // the table's byte size must fit in 64 bits
    if (table_rows > INT64_MAX / ((int64_t)num_layers * dim * 2)) return PLE_ERR_SIZE;
    // the output's byte count, L * T * dim float, fits int64
    if ((int64_t)num_layers * num_tokens > (INT64_MAX / 4) / dim) return PLE_ERR_SIZE;
    if (empty) return PLE_OK;
    if (!out || (table_rows > 0 && !table)) return PLE_ERR_NULL;
    if (!aligned(table, 16) || !aligned(out, 16)) return PLE_ERR_ALIGN;

    ple::DeviceFacts dev;
    cudaError_t e = ple::device_facts(&dev);
    if (e != cudaSuccess) return cuda_failure(e);
    ple::EmbedArgs ea;
    ea.table = static_cast<const uint16_t*>(table);
    ea.rows = table_rows;
    ea.dim = dim;
    ea.out = out;
    const ple::RowIdsLaunch cfg = ple::plan_row_ids(p, dev, /*runtime_layout=*/true);
    if (cfg.grid.y > 65535u) return PLE_ERR_SIZE;
    e = ple::launch_row_embed(p, ea, id_dtype == PLE_I32 ? 4 : 8, cfg,
                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e);
    return PLE_OK;
}

extern "C" ple_status ple_shard_plan(const int32_t* cu_seqlens, int32_t num_requests,
                                     int64_t num_tokens, int32_t world_size, int32_t rank,
                                     int64_t* token_begin, int64_t* token_end,
                                     int32_t* request_begin, int32_t* request_count) {
    if (!token_begin || !token_end || !request_begin || !request_count) return PLE_ERR_NULL;
    if (num_tokens < 0 || num_tokens > INT32_MAX || num_requests < 1 || world_size < 1 ||
        rank < 0 || rank >= world_size)
        return PLE_ERR_SIZE;
    const int64_t T = num_tokens;
    const int64_t a = T * rank / world_size;
    const int64_t b = T * (rank + 1) / world_size;
    if (!cu_seqlens) {
        // a decode batch: token t is request t
        if ((int64_t)num_requests != T) return PLE_ERR_SIZE;
        *token_begin = a;
        *token_end = b;
        *request_begin = (int32_t)a;
        *request_count = (int32_t)(b - a);
        return PLE_OK;
    }
    // host data: check it is a prefix sum of T
    if (cu_seqlens[0] != 0 || (int64_t)cu_seqlens[num_requests] != T) return PLE_ERR_SIZE;
    for (int32_t r = 0; r < num_requests; ++r)
        if (cu_seqlens[r + 1] < cu_seqlens[r]) return PLE_ERR_SIZE;
    *token_begin = a;
    *token_end = b;
    if (a == b) {
        *request_begin = 0;
        *request_count = 0;
        return PLE_OK;
    }
    // the owner of token t: the last r with cu_seqlens[r] <= t
    auto owner = [&](int64_t t) {
        int32_t lo = 0, hi = num_requests - 1;
        while (lo < hi) {
            const int32_t mid = lo + (hi - lo + 1) / 2;
            if ((int64_t)cu_seqlens[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    };
    const int32_t r0 = owner(a);
    const int32_t r1 = owner(b - 1);
    *request_begin = r0;
    *request_count = r1 - r0 + 1;
    return PLE_OK;
}

extern "C" ple_status ple_shard_inputs(const void* input_ids, int32_t id_dtype,
                                       const int32_t* cu_seqlens, const void* ngram_context,
                                       int32_t num_requests, int64_t num_tokens, int32_t ctx_len,
                                       int64_t token_begin, int64_t token_end,
                                       int32_t request_begin, int32_t request_count,
                                       int32_t* shard_cu_seqlens, void* shard_context,
                                       void* stream) {
    if (num_requests < 1 || num_tokens < 1 || num_tokens > INT32_MAX || ctx_len < 1 ||
        ctx_len >= PLE_MAX_NGRAM || token_begin < 0 || token_end <= token_begin ||
        token_end > num_tokens || request_begin < 0 || request_count < 1 ||
        (int64_t)request_begin + request_count > num_requests)
        return PLE_ERR_SIZE;
    if (!input_ids || !cu_seqlens || !ngram_context || !shard_cu_seqlens || !shard_context)
        return PLE_ERR_NULL;
    if (id_dtype != PLE_I32 && id_dtype != PLE_I64) return PLE_ERR_DTYPE;
    const int id_bytes = id_dtype == PLE_I32 ? 4 : 8;
    if (!aligned(input_ids, id_bytes) || !aligned(ngram_context, id_bytes) ||
        !aligned(shard_context, id_bytes) || !aligned(cu_seqlens, 4) ||
        !aligned(shard_cu_seqlens, 4))
        return PLE_ERR_ALIGN;
    cudaError_t e = ple::launch_shard_inputs(
        input_ids, id_bytes, cu_seqlens, ngram_context, num_requests, num_tokens, ctx_len,
        token_begin, token_end, request_begin, request_count, shard_cu_seqlens, shard_context,
        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e);
    return PLE_OK;
}

extern "C" ple_status ple_validate_index(const int32_t* cu_seqlens, int32_t num_requests,
                                         int64_t num_tokens, int32_t is_decode,
                                         const int32_t* req, const int32_t* local,
                                         int64_t* first_bad, void* stream) {
    if (num_tokens < 0 || num_tokens > INT32_MAX) return PLE_ERR_SIZE;
    if (num_tokens == 0) return PLE_OK;
    if (num_requests < 1) return PLE_ERR_SIZE;
    if (is_decode && (int64_t)num_requests != num_tokens) return PLE_ERR_SIZE;
    if (!req || !local || !first_bad || (!is_decode && !cu_seqlens)) return PLE_ERR_NULL;
    if (!aligned(req, 4) || !aligned(local, 4) || !aligned(first_bad, 8) ||
        (!is_decode && !aligned(cu_seqlens, 4)))
        return PLE_ERR_ALIGN;
    ple::DeviceFacts dev;
    cudaError_t e = ple::device_facts(&dev);
    if (e != cudaSuccess) return cuda_failure(e);
    e = ple::launch_validate_index(cu_seqlens, num_requests, num_tokens, is_decode, req, local,
                                   first_bad, dev, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e);
    return PLE_OK;
}

extern "C" ple_status ple_selftest_floor_mod(const int64_t* x, const int64_t* v, int64_t n,
                                             int64_t* out_fast, int64_t* out_ref, void* stream) {
    if (n < 0) return PLE_ERR_SIZE;
    if (n == 0) return PLE_OK;
    if (!x || !v || !out_fast || !out_ref) return PLE_ERR_NULL;
    if (!aligned(x, 8) || !aligned(v, 8) || !aligned(out_fast, 8) || !aligned(out_ref, 8))
        return PLE_ERR_ALIGN;
    ple::DeviceFacts dev;
    cudaError_t e = ple::device_facts(&dev);
    if (e != cudaSuccess) return cuda_failure(e);
    e = ple::launch_selftest_floor_mod(x, v, n, out_fast, out_ref, dev,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_failure(e);
    return PLE_OK;
}

extern "C" const char* ple_status_string(int32_t status) {
    switch (status) {
        case PLE_OK: return "ok";
        case PLE_ERR_NULL: return "a required pointer is NULL";
        case PLE_ERR_SIZE: return "a size or count is out of the supported range";
        case PLE_ERR_GEOMETRY_CTX: return "ngram_context must hold ngram_size - 1 ids per request";
        case PLE_ERR_GEOMETRY_HEADS:
            return "num_heads must equal (ngram_size - 1) * heads_per_ngram";
        case PLE_ERR_DTYPE: return "id dtype must be PLE_I32 or PLE_I64";
        case PLE_ERR_ALIGN: return "a pointer is not aligned to its element size";
        case PLE_ERR_CUDA: return "a CUDA call failed";
        default: return "unknown status";
    }
}

extern "C" int32_t ple_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int64_t ple_small_batch_max_rows(void) { return ple::kSmallMaxRows; }

extern "C" int32_t ple_set_programmatic_launch(int32_t enabled) {
    return ple::g_programmatic.exchange(enabled ? 1 : 0) != 0 ? 1 : 0;
}
